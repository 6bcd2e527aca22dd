// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "fa.h"

namespace fa {

// A kernel's one-time set-up (its shared-memory limit) is per device: `done`
// holds one bit per device on which it has run. Racing first calls both run
// the set-up, which is idempotent.
inline bool setup_needed(const std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return true;
  return ((done.load(std::memory_order_acquire) >> dev) & 1u) == 0;
}
inline void setup_done(std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64)
    done.fetch_or(uint64_t{1} << dev, std::memory_order_release);
}

// Encode a 4-D TMA map over a bf16 tensor stored BNSD or BSND, with
// dimensions ordered (D, S, N, B) so that one box is `box_s` rows of
// `box_d` elements of one (batch, head). Returns false on failure.
bool encode_bf16_map(CUtensorMap* map, const void* base, int layout, int64_t B, int64_t N,
                     int64_t S, int64_t D, int box_d, int box_s, CUtensorMapSwizzle swizzle);

int device_sm_count();  // of the current device; 0 on failure

// Query heads one decode stage-1 CTA handles: the largest of 8/4/2/1 that
// divides the GQA group size g (at most 4 for D = 128, to stay in registers).
inline int decode_heads_per_cta(int64_t g, int64_t D) {
  if (D == 64 && g % 8 == 0) return 8;
  return (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1;
}

// Prefill tiling: query rows of one work item (two 128-row tiles; one for
// D = 256, whose O accumulator takes 256 TMEM columns) and keys per KV tile
// (64 for D = 256, so that five K/V tiles and the Q tile fit shared memory).
inline int prefill_item_rows(int64_t D) { return D == 256 ? 128 : 256; }
inline int prefill_kv_tile(int64_t D) { return D == 256 ? 64 : 128; }

// Decode stage height in rows, and the batch count up to which the length
// prefix sums travel as launch parameters (larger batches use the workspace).
constexpr int kDecodeStageRows = 112;
constexpr int kDecodeParamBatches = 1024;
// Forced split counts merge the pieces of a unit in groups of this many
// slots, then the groups.
constexpr int kDecodeMergeGroup = 32;
// Smallest share of the work space one decode CTA is given.
constexpr int kDecodeMinRowsPerCta = 224;
// Cost of a piece end (the warps' park and combine, a partial stage, the
// partial write) in K/V rows of D = 128 (scaled by 128 / D), charged when the
// shares are cut by cost instead of by rows: when there are more units than
// SMs, so that a share holds several unit starts, and (the second figure)
// when there are fewer but a CTA carries four or more query heads.
constexpr int kDecodePieceCostRows128 = 192;
constexpr int kDecodePieceCostRows128Heads = 384;

// Error codes written to the device status word (first one wins).
enum DeviceError : uint32_t {
  kDevOk = 0,
  kDevTimeoutQ = 0x101,
  kDevTimeoutKvFull = 0x102,
  kDevTimeoutKvEmpty = 0x103,
  kDevTimeoutSFull = 0x104,
  kDevTimeoutPReady = 0x105,
  kDevTimeoutOFinal = 0x106,
  kDevTimeoutDrain = 0x107,
  kDevTimeoutTurn = 0x108,
  kDevTimeoutDecodeFull = 0x201,
  kDevTimeoutDecodeEmpty = 0x202,
  kDevPendingOverflow = 0x203,  // decode: more split pieces than a CTA can record
  kDevTimeoutProbe = 0x301,
  // debug builds (FA_DEBUG): device-side index checks that failed
  kDevCheckFirst = 0x401,
  kDevCheckDecodePiece = 0x401,    // a planned piece outside its unit or batch
  kDevCheckDecodeSlot = 0x402,     // a partial result slot past max_slots
  kDevCheckDecodeRow = 0x403,      // an output row past B x Hq
  kDevCheckDecodeMerge = 0x404,    // a merge over more pieces than slots
  kDevCheckPrefillItem = 0x411,    // a work item or Q tile outside the problem
  kDevCheckPrefillKv = 0x412,      // a KV tile outside the sequence
  kDevCheckPrefillOut = 0x413,     // an output row outside the tensor
  kDevCheckLast = 0x4ff,
};

// Largest persistent prefill grid the workspace's schedule has room for.
constexpr int kMaxPrefillCtas = 1024;

struct DecodeLaunch {
  const void* q;
  const void* k;
  const void* v;
  const uint8_t* key_mask;
  long long mask_bstride, mask_hstride;  // key mask strides (elements) of batch and query head
  int B, Hq, Hkv, S_kv, D, layout;
  float scale;
  long long total;            // rows of the work space (KV heads x head groups x sum L_b)
  long long rows_per_cta;     // cost of each CTA's contiguous share (a row costs 1)
  long long piece_cost;       // cost of a unit start after the first (0: shares of rows)
  long long n_ctas;           // CTAs to launch
  bool loop_shares;           // fixed-size chunks, more than CTAs (a forced split count: split_kernel)
  int max_slots;              // piece slots per (batch, head) in the partial buffers
  const long long* prefix_host;  // [B + 1] prefix sums of the lengths
  const long long* prefix_dev;   // the same in the workspace, or null (then in params)
  float* part_o;            // [B, Hq, max_slots, D]
  float* part_lse;          // [B, Hq, max_slots] (log2 domain)
  unsigned int* counters;   // [B * units per batch] pieces (forced splits: groups) finished, zeroed before the launch
  // forced split counts: group partials [B, Hq, max_groups, D] and
  // [B, Hq, max_groups], pieces finished per group [units][max_groups] (zeroed)
  float* grp_o;
  float* grp_lse;
  unsigned int* grp_counters;
  int max_groups;
  bool has_empty;           // some sequence has length 0
  // paged K/V (block_table != null): k, v are block pools of num_blocks blocks
  // of block_size rows in `layout` (BSND: PA_BBND, BNSD: PA_BNBD), logical
  // row r of batch b lives in block block_table[b * max_blocks + r / block_size];
  // the work space then holds every length rounded up to 16 rows and
  // lens_host / lens_dev give the real ones
  const int32_t* block_table;
  int max_blocks, num_blocks, block_size;
  const int* lens_dev;      // [B] real lengths in the workspace (paged, B > kDecodeParamBatches)
  const int64_t* lens_host; // [B] real lengths (paged only)
  void* out;
  float* lse;
  uint32_t* status;
  uint64_t timeout_ns;
};
cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t stream);
// Zero `bytes` (a multiple of 4) at the start of a decode workspace, before
// launch_decode on the same stream (which may then start its set-up while
// this runs).
cudaError_t launch_clear(void* workspace, size_t bytes, cudaStream_t stream);

struct PrefillLaunch {
  const void* q;
  const void* k;
  const void* v;
  int B, Hq, Hkv, S_q, S_kv, D, layout;
  int win_left, win_right;    // key j seen by query i iff i - wl <= j <= i + wr; -1 = no limit
  float scale;
  const uint32_t* tile_bits;  // [B][ceil(S_kv/128)][4] or null
  const int32_t* sched;       // per-CTA work-item lists (offsets[grid + 1], then the lists)
  // packed sequences: [5][B] q offset, used q length, kv offset, used kv
  // length, q span (device), or null; then q/k/v/out are [T, H, D] (BSND with
  // B = 1 in the tile maps), S_q / S_kv the longest span and lse [T_q, Hq]
  const int32_t* varlen;
  long long T_q, T_kv;        // packed rows of q and k/v (packed sequences only)
  // paged K/V (block_table != null): k, v are pools of num_blocks blocks of
  // block_size rows in kv_layout (FA_LAYOUT_PA_BBND or FA_LAYOUT_PA_BNBD);
  // row r of batch b lives in block block_table[b * max_blocks + r / block_size]
  const int32_t* block_table = nullptr;
  int max_blocks = 0, num_blocks = 0, block_size = 0, kv_layout = 0;
  int grid;                   // persistent CTAs
  void* out;
  float* lse;
  uint32_t* status;
  uint64_t timeout_ns;
};
cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t stream);

// Build the per-(batch, 128-key tile) validity bit table from an optional
// key mask and optional device lengths; for packed sequences (varlen = the
// device [5][B] table) the mask is one flag per packed key and each
// sequence's keys end at its used kv length.
cudaError_t launch_tile_bits(const uint8_t* key_mask, const int* lens_dev, const int32_t* varlen,
                             int B, int S_kv, uint32_t* bits, cudaStream_t stream);

// Packed sequences: out = 0, lse = +inf for the query rows between each
// sequence's used length and its span (varlen = the device [5][B] table;
// most_rows = the largest such gap).
cudaError_t launch_truncated_rows(const int32_t* varlen, int B, int most_rows, int Hq, int D,
                                  void* out, float* lse, cudaStream_t stream);

cudaError_t launch_wait_probe(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream);

// fa_decode on a library-owned scratch array of scratch_bytes whose device
// address `scratch` returns: every argument is checked (host only) before it
// is called, and the array need only hold this call's plan (not the size
// query's bound); used by fa_decode_noalloc. Same checks and errors otherwise.
fa_status decode_on_scratch(const void* q, const void* k, const void* v,
                            const uint8_t* key_mask, const int64_t* lens, int64_t B,
                            int64_t S_kv_max, int64_t num_heads, int64_t num_kv_heads, int64_t D,
                            float scale, int layout, int num_splits, void* out, float* lse,
                            fa_status (*scratch)(void**), size_t scratch_bytes, void* stream);

// Diagnostics: events recorded around the main kernel (thread-local, may be
// null) and a process-wide count of kernel launches.
void main_kernel_begin(cudaStream_t stream);
void main_kernel_end(cudaStream_t stream);
void count_launches(int n);

// Default bounded-wait limit of the kernels (nanoseconds).
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// Lower bound of the limit of a drain wait (a kernel that gave up waits for
// its own copies and MMAs in flight before it releases shared memory and
// TMEM): those always complete, so the drain keeps a long limit even when the
// bounded-wait limit is set short.
constexpr uint64_t kDrainFloorNs = 100000000ull;
// The bounded-wait limit of the calls made from this thread
// (fa_set_wait_timeout_ns; kDefaultTimeoutNs unless set).
uint64_t wait_timeout_ns();

}  // namespace fa
