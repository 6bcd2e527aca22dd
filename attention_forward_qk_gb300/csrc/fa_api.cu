// C ABI of the attention forward library: argument validation, workspace
// layout, the decode split plan, TMA descriptor encoding and launches.
//
// The two-stage shape of the interface (size query, then a call that takes
// a caller-owned workspace and a stream) follows aclnnIncreFlashAttention
// guide §三 and §五; the checks mirror its §四 / §六 constraints
// (numHeads a multiple of numKeyValueHeads, 0 meaning "same as numHeads",
// lengths per batch) and the FlashAttn guide's layout and mask rules.
// Every argument error is returned before any CUDA call is made.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kAlign = 256;
constexpr int kChunkQuant = 64;  // forced-split chunk sizes are multiples of this
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
// K/V bytes of one prefill schedule section (see build_prefill_schedule): a
// quarter of the 126 MB L2, so that the K/V of two sections (the one ending
// and the one starting on other CTAs) and the Q tiles and outputs streaming
// through fit together
constexpr int64_t kPrefillL2Budget = int64_t(32) << 20;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t chunk_for_splits(int64_t S_kv_max, int num_splits) {
  int64_t c = ceil_div(S_kv_max, num_splits);
  c = ceil_div(c, kChunkQuant) * kChunkQuant;
  return std::max<int64_t>(c, kChunkQuant);
}

struct DecodeWs {
  size_t prefix, real_lens, counters, grp_counters, part_lse, part_o, grp_lse, grp_o, total;
  size_t clear;  // bytes from the start that are cleared before the launch
};

// [status word, unit counters, group counters | pad][length prefix sums,
// large batches only][real lengths, paged][partial lse][partial o][group lse]
// [group o]: the counters follow the status word so that one clear before the
// launch covers them all. groups: merge groups per unit (forced split counts,
// else 0).
DecodeWs decode_ws(int64_t B, int64_t Hq, int64_t D, int64_t max_slots, int64_t groups = 0) {
  DecodeWs w;
  w.counters = sizeof(uint32_t);  // per (batch, KV head, head group): pieces (or groups) finished
  w.grp_counters = w.counters + sizeof(uint32_t) * B * Hq;  // [units][groups]: pieces finished
  w.clear = w.grp_counters + sizeof(uint32_t) * B * Hq * groups;
  size_t off = align_up(w.clear);
  w.prefix = off;
  off += align_up(sizeof(int64_t) * (B + 1));
  w.real_lens = off;  // paged cache only
  off += align_up(sizeof(int32_t) * B);
  w.part_lse = off;
  off += align_up(sizeof(float) * B * Hq * max_slots);
  w.part_o = off;
  off += align_up(sizeof(float) * B * Hq * max_slots * D);
  w.grp_lse = off;
  off += align_up(sizeof(float) * B * Hq * groups);
  w.grp_o = off;
  off += align_up(sizeof(float) * B * Hq * groups * D);
  w.total = off;
  return w;
}

// Merge groups of a unit cut into `slots` pieces by a forced split count.
int64_t merge_groups(int64_t slots, int num_splits) {
  return num_splits > 0 && slots > 1 ? ceil_div(slots, kDecodeMergeGroup) : 0;
}

// Upper bound of the pieces one sequence is cut into, for the size query.
int64_t max_slots_bound(int64_t S_kv_max, int num_splits) {
  const int64_t S = std::max<int64_t>(S_kv_max, 1);
  const int64_t rc = num_splits > 0 ? chunk_for_splits(S, num_splits)
                                    : static_cast<int64_t>(kDecodeMinRowsPerCta);
  return ceil_div(S, rc) + 1;
}

struct PrefillWs {
  size_t sched, varlen, lens, bits, total;
};

// Work items of a prefill launch: 256 query rows (128 for D = 256) of one
// (batch, query head).
int64_t prefill_items(int64_t B, int64_t S_q, int64_t num_heads, int64_t D) {
  return B * num_heads * ceil_div(S_q, prefill_item_rows(D));
}

// [status, item counter | pad][schedule: offsets of kMaxPrefillCtas + 1 CTAs,
// then the item lists][packed-sequence table][lengths][per-tile key validity]
PrefillWs prefill_ws(int64_t B, int64_t S_q, int64_t S_kv, int64_t num_heads, int64_t D) {
  PrefillWs w;
  size_t off = kAlign;  // status word
  w.sched = off;
  off += align_up(sizeof(int32_t) * (kMaxPrefillCtas + 1 + prefill_items(B, S_q, num_heads, D)));
  w.varlen = off;  // packed sequences only: [5][B] offsets, used lengths, q spans
  off += align_up(sizeof(int32_t) * 5 * B);
  w.lens = off;
  off += align_up(sizeof(int32_t) * B);
  w.bits = off;
  off += align_up(sizeof(uint32_t) * 4 * B * ceil_div(std::max<int64_t>(S_kv, 1), 128));
  w.total = off;
  return w;
}


// Static schedule of the persistent prefill CTAs, in L2-sized sections (the
// FlashAttn guide §4, SectionStreamK: batch x head units are gathered into a
// section until their K/V reach an L2 budget, so that a section's K/V is not
// pushed out of L2 while its items run; each section is spread over all
// cores, and the sections follow one another). Items are numbered as the
// kernel decodes them: (batch, KV head) units one after another, inside a
// unit its query pairs heaviest (last) first, query heads innermost. A
// section is a run of consecutive units whose K/V bytes together stay within
// l2_budget (at least one unit); inside a section the items go, longest
// first, to the CTA with the least work so far (a greedy longest-processing-
// time schedule). The cost of an item is its KV tiles under the causal or
// window limits plus a constant for its start-up.
// Layout: offsets[grid + 1] into the lists, then the item lists (int32).
// lq, lkv: per-sequence lengths of packed sequences (else null); items past a
// sequence's query rows do not exist and are not scheduled. IR: query rows
// per item, BN: keys per KV tile (prefill_item_rows, prefill_kv_tile).
void build_prefill_schedule(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t S_kv,
                            int64_t D, int64_t win_left, int64_t win_right, int grid, int64_t IR,
                            int64_t BN, int64_t l2_budget, std::vector<int32_t>& sched,
                            const int32_t* lq = nullptr, const int32_t* lkv = nullptr) {
  const int64_t g = Hq / Hkv;
  const int64_t nq = ceil_div(S_q, IR);
  const int64_t n_tiles = ceil_div(std::max<int64_t>(S_kv, 1), BN);
  const int64_t per_unit = nq * g;
  const int64_t units = B * Hkv;
  const int64_t n_items = units * per_unit;
  // -1: the item does not exist
  auto cost = [&](int64_t w) -> int64_t {
    const int64_t qp = nq - 1 - (w % per_unit) / g;
    const int64_t b = (w / per_unit) / Hkv;
    const int64_t sq = lq ? lq[b] : S_q;
    const int64_t nt = lkv ? ceil_div(static_cast<int64_t>(lkv[b]), BN) : n_tiles;
    if (qp * IR >= sq) return -1;
    int64_t lo_u = nt, hi_u = 0;
    for (int64_t t = 0; t < IR / 128; ++t) {
      const int64_t r0 = qp * IR + t * 128;
      if (t == 1 && r0 >= sq) break;
      int64_t lo = 0, hi = nt;
      if (win_left >= 0) lo = std::max<int64_t>(0, r0 - win_left) / BN;
      if (win_right >= 0) hi = std::min(hi, (r0 + 127 + win_right) / BN + 1);
      lo_u = std::min(lo_u, lo);
      hi_u = std::max(hi_u, hi);
    }
    // KV tiles (of 128 keys' worth of work) plus a constant for the start-up
    return std::max<int64_t>(0, hi_u - lo_u) * BN / 128 + 3;
  };
  std::vector<std::vector<int32_t>> lists(grid);
  // min-heap of (load, cta)
  std::vector<std::pair<int64_t, int>> heap;
  heap.reserve(grid);
  for (int c = 0; c < grid; ++c) heap.emplace_back(0, c);
  auto cmp = [](const std::pair<int64_t, int>& x, const std::pair<int64_t, int>& y) {
    return x > y;
  };
  // K and V bytes of a (batch, KV head) unit
  auto unit_bytes = [&](int64_t u) -> int64_t {
    const int64_t L = lkv ? static_cast<int64_t>(lkv[u / Hkv]) : S_kv;
    return 2 * 2 * D * L;
  };
  std::vector<std::pair<int64_t, int64_t>> grp;
  for (int64_t u0 = 0, u1 = 0; u0 < units; u0 = u1) {
    // the section: units u0 .. u1-1, as many as the budget holds (at least one)
    int64_t bytes = unit_bytes(u0);
    for (u1 = u0 + 1; u1 < units && bytes + unit_bytes(u1) <= l2_budget; ++u1)
      bytes += unit_bytes(u1);
    const int64_t w0 = u0 * per_unit;
    const int64_t w1 = u1 * per_unit;
    grp.clear();
    for (int64_t w = w0; w < w1; ++w) {
      const int64_t c = cost(w);
      if (c >= 0) grp.emplace_back(-c, w);
    }
    std::stable_sort(grp.begin(), grp.end(),
                     [](const std::pair<int64_t, int64_t>& x, const std::pair<int64_t, int64_t>& y) {
                       return x.first < y.first;
                     });
    for (const auto& it : grp) {
      std::pop_heap(heap.begin(), heap.end(), cmp);
      auto& top = heap.back();
      lists[top.second].push_back(static_cast<int32_t>(it.second));
      top.first += -it.first;
      std::push_heap(heap.begin(), heap.end(), cmp);
    }
  }
  (void)n_items;
  size_t listed = 0;
  for (const auto& l : lists) listed += l.size();
  sched.assign(grid + 1 + listed, 0);
  int32_t off = 0;
  for (int c = 0; c < grid; ++c) {
    sched[c] = off;
    std::copy(lists[c].begin(), lists[c].end(), sched.begin() + grid + 1 + off);
    off += static_cast<int32_t>(lists[c].size());
  }
  sched[grid] = off;
}

// ------------------------------------------------------------ driver entry
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool encode_bf16_map(CUtensorMap* map, const void* base, int layout, int64_t B, int64_t N,
                     int64_t S, int64_t D, int box_d, int box_s, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  // dimensions (D, S, N, B), innermost first; strides in bytes for dims 1..3
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3];
  if (layout == FA_LAYOUT_BNSD) {
    strides[0] = static_cast<cuuint64_t>(D * 2);
    strides[1] = static_cast<cuuint64_t>(S * D * 2);
    strides[2] = static_cast<cuuint64_t>(N * S * D * 2);
  } else {
    strides[0] = static_cast<cuuint64_t>(N * D * 2);
    strides[1] = static_cast<cuuint64_t>(D * 2);
    strides[2] = static_cast<cuuint64_t>(S * N * D * 2);
  }
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_d), static_cast<cuuint32_t>(box_s), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
thread_local cudaEvent_t tl_before = nullptr;
thread_local cudaEvent_t tl_after = nullptr;
thread_local uint64_t tl_timeout_ns = 0;  // 0: kDefaultTimeoutNs
std::atomic<uint64_t> g_launches{0};
}  // namespace

uint64_t wait_timeout_ns() { return tl_timeout_ns != 0 ? tl_timeout_ns : kDefaultTimeoutNs; }

void main_kernel_begin(cudaStream_t stream) {
  if (tl_before != nullptr && tl_after != nullptr) cudaEventRecord(tl_before, stream);
}
void main_kernel_end(cudaStream_t stream) {
  if (tl_before != nullptr && tl_after != nullptr) cudaEventRecord(tl_after, stream);
}
void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

// SM count per device ordinal, looked up once per device (a fixed table:
// no heap allocation on any call)
int device_sm_count() {
  constexpr int kMaxCachedDevices = 64;
  static std::atomic<int> cache[kMaxCachedDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxCachedDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < kMaxCachedDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace fa

using namespace fa;

extern "C" {

int fa_abi_version(void) { return FA_ABI_VERSION; }

const char* fa_status_string(int s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_NULLPTR: return "FA_ERR_NULLPTR: a required pointer is NULL";
    case FA_ERR_PARAM_INVALID: return "FA_ERR_PARAM_INVALID: argument outside the contract";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim must be 64, 128 or 256";
    case FA_ERR_WORKSPACE_TOO_SMALL: return "FA_ERR_WORKSPACE_TOO_SMALL";
    case FA_ERR_RUNTIME: return "FA_ERR_RUNTIME: a CUDA call failed";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a kernel wait expired";
    case FA_ERR_DEVICE_CHECK: return "FA_ERR_DEVICE_CHECK: a device-side index check failed (debug build)";
    default: return "unknown fa_status";
  }
}

size_t fa_forward_workspace_size(int64_t B, int64_t S_q, int64_t S_kv, int64_t num_heads,
                                 int64_t num_kv_heads, int64_t D) {
  if (B < 0 || S_q < 0 || S_kv < 0 || num_heads < 0 || num_kv_heads < 0 || D < 0) return 0;
  (void)num_kv_heads;
  return prefill_ws(B, S_q, S_kv, num_heads, D).total;
}

namespace {
fa_status decode_plan_impl(int64_t B, int64_t S_kv_max, int64_t num_heads, int64_t num_kv_heads,
                           int64_t D, const int64_t* lens, int num_sms, int num_splits,
                           int64_t rc_align, int64_t* chunk_rows, int64_t* num_chunks,
                           int64_t* max_chunks, int64_t* piece_cost);
}  // namespace

fa_status fa_decode_plan(int64_t B, int64_t S_kv_max, int64_t num_heads, int64_t num_kv_heads,
                         int64_t D, const int64_t* lens, int num_sms, int num_splits,
                         int64_t* chunk_rows, int64_t* num_chunks, int64_t* max_chunks) {
  int64_t pc = 0;
  return decode_plan_impl(B, S_kv_max, num_heads, num_kv_heads, D, lens, num_sms, num_splits, 1,
                          chunk_rows, num_chunks, max_chunks, &pc);
}

namespace {
// rc_align: the per-CTA share is rounded up to a multiple of it (16 rows for
// a paged cache, whose work space is laid out in 16-row boxes)
fa_status decode_plan_impl(int64_t B, int64_t S_kv_max, int64_t num_heads, int64_t num_kv_heads,
                           int64_t D, const int64_t* lens, int num_sms, int num_splits,
                           int64_t rc_align, int64_t* chunk_rows, int64_t* num_chunks,
                           int64_t* max_chunks, int64_t* piece_cost) {
  if (lens == nullptr || chunk_rows == nullptr || num_chunks == nullptr || max_chunks == nullptr)
    return FA_ERR_NULLPTR;
  if (num_kv_heads == 0) num_kv_heads = num_heads;
  if (B < 0 || S_kv_max < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || num_splits < 0 || num_sms <= 0 || S_kv_max > kMaxDim)
    return FA_ERR_PARAM_INVALID;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  int64_t sum = 0;
  for (int64_t b = 0; b < B; ++b) {
    if (lens[b] < 0 || lens[b] > S_kv_max) return FA_ERR_PARAM_INVALID;
    sum += lens[b];
  }
  // work space: every (batch, KV head, head group) unit of L_b rows, end to end
  const int64_t g = num_heads / num_kv_heads;
  const int64_t KH = num_kv_heads * (g / decode_heads_per_cta(g, D));
  const int64_t total = KH * sum;
  // A share holding a unit start pays a piece end: the shares are cut by
  // cost, where a row costs 1 and every unit after the first adds pc
  // (FlashAttn guide §4: split the work into sections of equal cost), when
  // the (non-empty) units outnumber the SMs (a share then holds several unit
  // starts), and when a CTA carries four or more query heads (whose piece
  // end, with its warps' park and combine of every head, costs the most;
  // charged as more rows). Forced splits cut rows.
  int64_t units = 0, last_unit = -1;
  for (int64_t b = 0; b < B; ++b)
    if (lens[b] > 0) {
      units += KH;
      last_unit = b * KH + KH - 1;
    }
  int64_t pc = 0;
  if (num_splits == 0 && units > 1) {
    const int64_t rows128 = units > num_sms                           ? kDecodePieceCostRows128
                            : decode_heads_per_cta(g, D) >= 4 ? kDecodePieceCostRows128Heads
                                                              : 0;
    if (rows128 > 0) pc = std::max<int64_t>(rows128 * 128 / D / rc_align, 1) * rc_align;
  }
  const int64_t cost = total + pc * std::max<int64_t>(last_unit, 0);
  int64_t rc;
  if (num_splits > 0) {
    rc = chunk_for_splits(std::max<int64_t>(S_kv_max, 1), num_splits);
  } else {
    // one equal share per SM (at least a couple of stages each)
    rc = std::max<int64_t>(ceil_div(std::max<int64_t>(cost, 1), num_sms), kDecodeMinRowsPerCta);
  }
  rc = ceil_div(rc, rc_align) * rc_align;
  int64_t mx = 0, prefix = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t L = lens[b];
    if (L > 0) {
      for (int64_t kh = 0; kh < KH; ++kh) {
        const int64_t c0 = KH * prefix + kh * L + pc * (b * KH + kh);  // cost of its first row
        mx = std::max(mx, (c0 + L - 1) / rc - c0 / rc + 1);
      }
    }
    prefix += L;
  }
  *chunk_rows = rc;
  *num_chunks = total > 0 ? ceil_div(cost, rc) : 0;
  *piece_cost = pc;
  *max_chunks = mx;
  return FA_OK;
}
}  // namespace

size_t fa_decode_workspace_size(int64_t B, int64_t S_kv_max, int64_t num_heads,
                                int64_t num_kv_heads, int64_t D, int num_splits) {
  if (num_kv_heads == 0) num_kv_heads = num_heads;
  if (B < 0 || S_kv_max < 0 || num_heads < 0 || num_kv_heads < 0 || D < 0 || num_splits < 0)
    return 0;
  const int64_t slots = max_slots_bound(S_kv_max, num_splits);
  return decode_ws(B, num_heads, D, slots, merge_groups(slots, num_splits)).total;
}

// Head dims: 64, 128 and 256.
static fa_status check_common(int64_t B, int64_t S_q, int64_t S_kv, int64_t Hq, int64_t& Hkv,
                              int64_t D, float scale, int layout) {
  if (Hkv == 0) Hkv = Hq;
  if (B < 0 || S_q < 0 || S_kv < 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return FA_ERR_PARAM_INVALID;
  if (Hq % Hkv != 0) return FA_ERR_PARAM_INVALID;
  if (layout != FA_LAYOUT_BNSD && layout != FA_LAYOUT_BSND) return FA_ERR_PARAM_INVALID;
  if (!isfinite(scale)) return FA_ERR_PARAM_INVALID;
  if (B > kMaxDim || S_q > kMaxDim || S_kv > kMaxDim || Hq > 65535) return FA_ERR_PARAM_INVALID;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

namespace {

// Per host thread: the last prefill workspace header built (zeroed status
// word, schedule, packed-sequence table, lengths) and the key it was built
// for, so that a call with the same shapes and lengths builds nothing and
// allocates nothing on the host. The header goes to the device by one
// cudaMemcpyAsync from this host copy: for headers this small the driver
// carries the data in its command stream, which measured faster than a copy
// from pinned memory (tiny prefill: 11.8 us per call against 19.2 us; the
// pinned copy goes through a copy engine).
struct SchedKey {
  int64_t B, Hq, Hkv, S_q, S_kv, wl, wr, D;
  int grid;
  bool operator==(const SchedKey& o) const {
    return B == o.B && Hq == o.Hq && Hkv == o.Hkv && S_q == o.S_q && S_kv == o.S_kv &&
           wl == o.wl && wr == o.wr && D == o.D && grid == o.grid;
  }
};
struct PrefillHeader {
  bool valid = false;
  SchedKey key{};
  std::vector<int32_t> vtab, lens;            // the key's packed table and lengths
  std::vector<int32_t> vtab_next, lens_next;  // this call's, compared with the key's
  std::vector<int32_t> sched, blob;
};

PrefillHeader& prefill_header_cache() {
  thread_local PrefillHeader h;
  return h;
}

// A paged K/V cache (fa_decode_paged, fa_forward_paged); null for a
// contiguous one. kv_layout: FA_LAYOUT_PA_BBND or FA_LAYOUT_PA_BNBD (prefill;
// the decode path passes the equivalent contiguous layout itself).
struct PagedKv {
  const int32_t* block_table;
  int64_t max_blocks, num_blocks, block_size;
  int kv_layout = 0;
};

// Shared by fa_forward and fa_forward_window: the window (-1, -1) is no mask,
// (-1, 0) is causal.
// cu_q, cu_kv: HOST prefix offsets of packed sequences (else null); then
// S_q / S_kv are the longest sequences, the tensors are [T, H, D], key_mask
// (if any) is one flag per packed key [T_kv], and used_q / used_kv (HOST,
// nullable) cut each sequence to the shorter of its span and the used length.
fa_status forward_impl(const void* q, const void* k, const void* v, bool mask_ok,
                       int64_t win_left, int64_t win_right, const uint8_t* key_mask,
                       const int64_t* lens,
                       int64_t B, int64_t S_q, int64_t S_kv, int64_t num_heads,
                       int64_t num_kv_heads, int64_t D, float scale, int layout, void* out,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream,
                       const int64_t* cu_q = nullptr, const int64_t* cu_kv = nullptr,
                       const int64_t* used_q = nullptr, const int64_t* used_kv = nullptr,
                       const PagedKv* pg = nullptr) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || workspace == nullptr)
    return FA_ERR_NULLPTR;
  int64_t Hkv = num_kv_heads;
  fa_status st = check_common(B, S_q, S_kv, num_heads, Hkv, D, scale, layout);
  if (st != FA_OK) return st;
  if (!mask_ok || win_left < -1 || win_right < -1) return FA_ERR_PARAM_INVALID;
  const bool windowed = win_left >= 0 || win_right >= 0;
  if (windowed && S_q != S_kv && cu_q == nullptr) return FA_ERR_PARAM_INVALID;
  if (windowed && cu_q != nullptr)
    for (int64_t b = 0; b < B; ++b)
      if (cu_q[b + 1] - cu_q[b] != cu_kv[b + 1] - cu_kv[b]) return FA_ERR_PARAM_INVALID;
  // wider than the sequence is no limit (and keeps the tile arithmetic in int)
  if (win_left >= S_kv) win_left = -1;
  if (win_right >= S_kv) win_right = -1;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return FA_ERR_PARAM_INVALID;
  if (lens != nullptr)
    for (int64_t b = 0; b < B; ++b)
      if (lens[b] < 0 || lens[b] > S_kv) return FA_ERR_PARAM_INVALID;
  const PrefillWs ws = prefill_ws(B, S_q, S_kv, num_heads, D);
  if (workspace_bytes < ws.total) return FA_ERR_WORKSPACE_TOO_SMALL;
  if (B == 0 || S_q == 0) return FA_OK;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  const int sms = device_sm_count();
  if (sms <= 0) return FA_ERR_RUNTIME;
  const int64_t n_items = prefill_items(B, S_q, num_heads, D);
  const int64_t IR = prefill_item_rows(D), BN = prefill_kv_tile(D);
  const int grid = static_cast<int>(
      std::min<int64_t>(std::min<int64_t>(n_items, sms), kMaxPrefillCtas));
  // The workspace header (zeroed status word, the schedule, the packed-sequence
  // table, the lengths) depends on the shapes and lengths only: the last one
  // built on this host thread is kept and rebuilt only when they change.
  PrefillHeader& hc = prefill_header_cache();
  const SchedKey key{B, num_heads, Hkv, S_q, S_kv, win_left, win_right, D, grid};
  // packed sequences: [5][B] q offset, used q length, kv offset, used kv
  // length (the shorter of the span and seqused), q span; lengths as int32
  std::vector<int32_t>& vtab = hc.vtab_next;
  vtab.resize(cu_q != nullptr ? 5 * B : 0);
  bool truncated_q = false, truncated_kv = false;
  if (cu_q != nullptr) {
    for (int64_t b = 0; b < B; ++b) {
      const int64_t span_q = cu_q[b + 1] - cu_q[b];
      const int64_t span_kv = cu_kv[b + 1] - cu_kv[b];
      const int64_t uq = used_q ? std::min(span_q, used_q[b]) : span_q;
      const int64_t ukv = used_kv ? std::min(span_kv, used_kv[b]) : span_kv;
      truncated_q = truncated_q || uq < span_q;
      truncated_kv = truncated_kv || ukv < span_kv;
      vtab[b] = static_cast<int32_t>(cu_q[b]);
      vtab[B + b] = static_cast<int32_t>(uq);
      vtab[2 * B + b] = static_cast<int32_t>(cu_kv[b]);
      vtab[3 * B + b] = static_cast<int32_t>(ukv);
      vtab[4 * B + b] = static_cast<int32_t>(span_q);
    }
  }
  std::vector<int32_t>& lens32 = hc.lens_next;
  lens32.resize(lens != nullptr ? B : 0);
  for (int64_t b = 0; b < static_cast<int64_t>(lens32.size()); ++b)
    lens32[b] = static_cast<int32_t>(lens[b]);
  if (!hc.valid || !(hc.key == key) || hc.vtab != vtab || hc.lens != lens32) {
    build_prefill_schedule(B, num_heads, Hkv, S_q, S_kv, D, win_left, win_right, grid, IR, BN,
                           kPrefillL2Budget, hc.sched, cu_q ? vtab.data() + B : nullptr,
                           cu_q ? vtab.data() + 3 * B : nullptr);
    hc.blob.assign(ws.lens / 4 + lens32.size(), 0);
    std::copy(hc.sched.begin(), hc.sched.end(), hc.blob.begin() + ws.sched / 4);
    std::copy(vtab.begin(), vtab.end(), hc.blob.begin() + ws.varlen / 4);
    std::copy(lens32.begin(), lens32.end(), hc.blob.begin() + ws.lens / 4);
    hc.key = key;
    hc.vtab.swap(vtab);
    hc.lens.swap(lens32);
    hc.valid = true;
  }
  const std::vector<int32_t>& vt = hc.vtab;  // the table of this call
  if (cudaMemcpyAsync(wsb, hc.blob.data(), hc.blob.size() * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FA_ERR_RUNTIME;
  const uint32_t* bits = nullptr;
  const int32_t* vtab_dev =
      cu_q != nullptr ? reinterpret_cast<const int32_t*>(wsb + ws.varlen) : nullptr;
  // the validity table also zeroes the V rows of excluded keys: needed for a
  // key mask, for lengths, for packed keys cut by seqused_kv (the rows past a
  // used length may hold anything), and for a paged cache whose last KV tile
  // runs past S_kv (its rows there are pool rows, not the zeros a load past
  // the end of a contiguous tensor returns)
  const bool paged_ragged = pg != nullptr && S_kv % BN != 0;
  if ((key_mask != nullptr || lens != nullptr || truncated_kv || paged_ragged) && S_kv > 0) {
    uint32_t* bits_dev = reinterpret_cast<uint32_t*>(wsb + ws.bits);
    const int* lens_dev = lens ? reinterpret_cast<const int*>(wsb + ws.lens) : nullptr;
    // packed: the keys of sequence b start at its kv offset and end at its
    // used kv length (both in the table)
    if (launch_tile_bits(key_mask, lens_dev, vtab_dev, static_cast<int>(B),
                         static_cast<int>(S_kv), bits_dev, s) != cudaSuccess)
      return FA_ERR_RUNTIME;
    count_launches(1);
    bits = bits_dev;
  }
  if (truncated_q) {
    // query rows past a sequence's used length: out 0, lse +inf (the prefill
    // kernel writes only the used rows)
    int64_t most = 0;
    for (int64_t b = 0; b < B; ++b) most = std::max<int64_t>(most, vt[4 * B + b] - vt[B + b]);
    if (launch_truncated_rows(vtab_dev, static_cast<int>(B), static_cast<int>(most),
                              static_cast<int>(num_heads), static_cast<int>(D), out, lse,
                              s) != cudaSuccess)
      return FA_ERR_RUNTIME;
    count_launches(1);
  }
  PrefillLaunch x;
  x.q = q;
  x.k = k;
  x.v = v;
  x.B = static_cast<int>(B);
  x.Hq = static_cast<int>(num_heads);
  x.Hkv = static_cast<int>(Hkv);
  x.S_q = static_cast<int>(S_q);
  x.S_kv = static_cast<int>(S_kv);
  x.D = static_cast<int>(D);
  x.layout = layout;
  x.win_left = static_cast<int>(win_left);
  x.win_right = static_cast<int>(win_right);
  x.scale = scale;
  x.tile_bits = bits;
  x.sched = reinterpret_cast<const int32_t*>(wsb + ws.sched);
  x.grid = grid;
  x.varlen = vtab_dev;
  x.T_q = cu_q != nullptr ? cu_q[B] : 0;
  x.T_kv = cu_kv != nullptr ? cu_kv[B] : 0;
  if (pg != nullptr) {
    x.block_table = pg->block_table;
    x.max_blocks = static_cast<int>(pg->max_blocks);
    x.num_blocks = static_cast<int>(pg->num_blocks);
    x.block_size = static_cast<int>(pg->block_size);
    x.kv_layout = pg->kv_layout;
  }
  x.out = out;
  x.lse = lse;
  x.status = reinterpret_cast<uint32_t*>(wsb);
  x.timeout_ns = wait_timeout_ns();
  main_kernel_begin(s);
  const cudaError_t e = launch_prefill(x, s);
  main_kernel_end(s);
  if (e != cudaSuccess) return FA_ERR_RUNTIME;
  count_launches(1);
  return FA_OK;
}

}  // namespace

fa_status fa_forward(const void* q, const void* k, const void* v, int mask_mode,
                     const uint8_t* key_mask, const int64_t* lens, int64_t B, int64_t S_q,
                     int64_t S_kv, int64_t num_heads, int64_t num_kv_heads, int64_t D,
                     float scale, int layout, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, void* stream) {
  const bool mask_ok = mask_mode == FA_MASK_NONE || mask_mode == FA_MASK_CAUSAL;
  const bool causal = mask_mode == FA_MASK_CAUSAL;
  return forward_impl(q, k, v, mask_ok, -1, causal ? 0 : -1, key_mask, lens, B, S_q, S_kv, num_heads,
                      num_kv_heads, D, scale, layout, out, lse, workspace, workspace_bytes,
                      stream);
}

size_t fa_forward_varlen_workspace_size(int64_t B, int64_t max_seqlen_q, int64_t max_seqlen_kv,
                                        int64_t num_heads, int64_t num_kv_heads, int64_t D) {
  return fa_forward_workspace_size(B, max_seqlen_q, max_seqlen_kv, num_heads, num_kv_heads, D);
}

namespace {
// fa_forward_varlen and fa_forward_varlen_window: the offsets checked, then
// the window (-1, -1) no mask, (-1, 0) causal
fa_status forward_varlen_impl(const void* q, const void* k, const void* v,
                              const int64_t* cu_seqlens_q, const int64_t* cu_seqlens_kv,
                              const int64_t* seqused_q, const int64_t* seqused_kv,
                              const uint8_t* key_mask, bool mask_ok, int64_t win_left,
                              int64_t win_right, int64_t B, int64_t num_heads,
                              int64_t num_kv_heads, int64_t D, float scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (cu_seqlens_q == nullptr || cu_seqlens_kv == nullptr) return FA_ERR_NULLPTR;
  if (B < 0) return FA_ERR_PARAM_INVALID;
  if (cu_seqlens_q[0] != 0 || cu_seqlens_kv[0] != 0) return FA_ERR_PARAM_INVALID;
  int64_t max_q = 0, max_kv = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t lq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    const int64_t lkv = cu_seqlens_kv[b + 1] - cu_seqlens_kv[b];
    if (lq < 0 || lkv < 0) return FA_ERR_PARAM_INVALID;
    if ((seqused_q != nullptr && seqused_q[b] < 0) || (seqused_kv != nullptr && seqused_kv[b] < 0))
      return FA_ERR_PARAM_INVALID;
    max_q = std::max(max_q, lq);
    max_kv = std::max(max_kv, lkv);
  }
  if (cu_seqlens_q[B] > kMaxDim || cu_seqlens_kv[B] > kMaxDim) return FA_ERR_PARAM_INVALID;
  // packed tensors [T, H, D] are BSND with one batch
  return forward_impl(q, k, v, mask_ok, win_left, win_right, key_mask, nullptr, B, max_q, max_kv,
                      num_heads, num_kv_heads, D, scale, FA_LAYOUT_BSND, out, lse, workspace,
                      workspace_bytes, stream, cu_seqlens_q, cu_seqlens_kv, seqused_q,
                      seqused_kv);
}
}  // namespace

fa_status fa_forward_varlen(const void* q, const void* k, const void* v,
                            const int64_t* cu_seqlens_q, const int64_t* cu_seqlens_kv,
                            int mask_mode, int64_t B, int64_t num_heads, int64_t num_kv_heads,
                            int64_t D, float scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream) {
  const bool mask_ok = mask_mode == FA_MASK_NONE || mask_mode == FA_MASK_CAUSAL;
  const bool causal = mask_mode == FA_MASK_CAUSAL;
  return forward_varlen_impl(q, k, v, cu_seqlens_q, cu_seqlens_kv, nullptr, nullptr, nullptr,
                             mask_ok, -1, causal ? 0 : -1, B, num_heads, num_kv_heads, D, scale,
                             out, lse, workspace, workspace_bytes, stream);
}

fa_status fa_forward_varlen_window(const void* q, const void* k, const void* v,
                                   const int64_t* cu_seqlens_q, const int64_t* cu_seqlens_kv,
                                   int64_t win_left, int64_t win_right, int64_t B,
                                   int64_t num_heads, int64_t num_kv_heads, int64_t D, float scale,
                                   void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return forward_varlen_impl(q, k, v, cu_seqlens_q, cu_seqlens_kv, nullptr, nullptr, nullptr,
                             true, win_left, win_right, B, num_heads, num_kv_heads, D, scale,
                             out, lse, workspace, workspace_bytes, stream);
}

fa_status fa_forward_varlen_ex(const void* q, const void* k, const void* v,
                               const int64_t* cu_seqlens_q, const int64_t* cu_seqlens_kv,
                               const int64_t* seqused_q, const int64_t* seqused_kv,
                               const uint8_t* key_mask, int64_t win_left, int64_t win_right,
                               int64_t B, int64_t num_heads, int64_t num_kv_heads, int64_t D,
                               float scale, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return forward_varlen_impl(q, k, v, cu_seqlens_q, cu_seqlens_kv, seqused_q, seqused_kv,
                             key_mask, true, win_left, win_right, B, num_heads, num_kv_heads, D,
                             scale, out, lse, workspace, workspace_bytes, stream);
}

fa_status fa_forward_paged(const void* q, const void* k_cache, const void* v_cache, int kv_layout,
                           const int32_t* block_table, int64_t max_blocks_per_seq,
                           int64_t num_blocks, int64_t block_size, int mask_mode,
                           const uint8_t* key_mask, const int64_t* lens, int64_t B, int64_t S_q,
                           int64_t S_kv, int64_t num_heads, int64_t num_kv_heads, int64_t D,
                           float scale, int layout, void* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (block_table == nullptr && B > 0) return FA_ERR_NULLPTR;
  if (kv_layout != FA_LAYOUT_PA_BBND && kv_layout != FA_LAYOUT_PA_BNBD) return FA_ERR_PARAM_INVALID;
  if (block_size < 16 || block_size > 1024 || block_size % 16 != 0 || max_blocks_per_seq < 0 ||
      num_blocks < 0 || max_blocks_per_seq > kMaxDim / 1024 || num_blocks > kMaxDim)
    return FA_ERR_PARAM_INVALID;
  // the table covers every key row of a sequence
  if (S_kv > 0 && max_blocks_per_seq * block_size < S_kv) return FA_ERR_PARAM_INVALID;
  const bool mask_ok = mask_mode == FA_MASK_NONE || mask_mode == FA_MASK_CAUSAL;
  const bool causal = mask_mode == FA_MASK_CAUSAL;
  const PagedKv pg{block_table, std::max<int64_t>(max_blocks_per_seq, 1),
                   std::max<int64_t>(num_blocks, 1), block_size, kv_layout};
  return forward_impl(q, k_cache, v_cache, mask_ok, -1, causal ? 0 : -1, key_mask, lens, B, S_q,
                      S_kv, num_heads, num_kv_heads, D, scale, layout, out, lse, workspace,
                      workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr, &pg);
}

fa_status fa_forward_window(const void* q, const void* k, const void* v, int64_t win_left,
                            int64_t win_right, const uint8_t* key_mask, const int64_t* lens,
                            int64_t B, int64_t S_q, int64_t S_kv, int64_t num_heads,
                            int64_t num_kv_heads, int64_t D, float scale, int layout, void* out,
                            float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(q, k, v, true, win_left, win_right, key_mask, lens, B, S_q, S_kv, num_heads,
                      num_kv_heads, D, scale, layout, out, lse, workspace, workspace_bytes,
                      stream);
}

namespace {

// scratch: when given, the workspace is not the caller's but the one this
// function returns (the library-owned array of fa_decode_noalloc, looked up
// only after every argument check); it need only hold what this call's plan
// uses. Otherwise the workspace must hold the size query's bound, as the
// contract of fa_decode states.
// mask_layout: FA_KEY_MASK_B11S (one flag per key, shared by the heads),
// FA_KEY_MASK_BN1S or FA_KEY_MASK_1N1S (one row of flags per query head).
fa_status decode_impl(const void* q, const void* k, const void* v, const PagedKv* pg,
                      const uint8_t* key_mask, const int64_t* lens, int64_t B, int64_t S_kv_max,
                      int64_t num_heads, int64_t num_kv_heads, int64_t D, float scale, int layout,
                      int num_splits, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream,
                      fa_status (*scratch)(void**) = nullptr,
                      int mask_layout = FA_KEY_MASK_B11S) {
  const bool exact_ws = scratch != nullptr;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
      (workspace == nullptr && !exact_ws) || lens == nullptr)
    return FA_ERR_NULLPTR;
  int64_t Hkv = num_kv_heads;
  fa_status st = check_common(B, 1, S_kv_max, num_heads, Hkv, D, scale, layout);
  if (st != FA_OK) return st;
  if (num_splits < 0) return FA_ERR_PARAM_INVALID;
  if (mask_layout != FA_KEY_MASK_B11S && mask_layout != FA_KEY_MASK_BN1S &&
      mask_layout != FA_KEY_MASK_1N1S)
    return FA_ERR_PARAM_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return FA_ERR_PARAM_INVALID;
  for (int64_t b = 0; b < B; ++b)
    if (lens[b] < 0 || lens[b] > S_kv_max) return FA_ERR_PARAM_INVALID;
  if (exact_ws && B > kDecodeParamBatches) return FA_ERR_PARAM_INVALID;
  if (!exact_ws &&
      workspace_bytes < fa_decode_workspace_size(B, S_kv_max, num_heads, Hkv, D, num_splits))
    return FA_ERR_WORKSPACE_TOO_SMALL;
  if (B == 0) return FA_OK;

  // a paged cache is streamed in 16-row boxes: its work space holds every
  // length rounded up to 16 rows (the kernel masks the extra rows)
  std::vector<int64_t> lens16;
  const int64_t* wlens = lens;
  if (pg != nullptr) {
    lens16.resize(B);
    for (int64_t b = 0; b < B; ++b) lens16[b] = ceil_div(lens[b], 16) * 16;
    wlens = lens16.data();
  }
  const int sms = device_sm_count();
  if (sms <= 0) return FA_ERR_RUNTIME;
  int64_t rc = 0, n_ctas = 0, max_slots = 0, pc = 0;
  st = decode_plan_impl(B, S_kv_max, num_heads, Hkv, D, wlens, sms, num_splits,
                        pg != nullptr ? 16 : 1, &rc, &n_ctas, &max_slots, &pc);
  if (st != FA_OK) return st;
  const int64_t slots = std::max<int64_t>(max_slots, 1);
  if (slots > max_slots_bound(S_kv_max, num_splits)) return FA_ERR_RUNTIME;  // cannot happen
  // partial buffers only when some sequence is cut into several pieces
  const int64_t groups = max_slots > 1 ? merge_groups(slots, num_splits) : 0;
  const DecodeWs ws = decode_ws(B, num_heads, D, max_slots > 1 ? slots : 0, groups);
  if (workspace_bytes < ws.total) return FA_ERR_WORKSPACE_TOO_SMALL;
  if (exact_ws) {
    st = scratch(&workspace);
    if (st != FA_OK) return st;
  }

  // length prefix sums: on the stack for batches that travel in the launch
  // parameters, on the heap only for larger ones
  long long prefix_small[kDecodeParamBatches + 1];
  std::vector<long long> prefix_big;
  long long* prefix = prefix_small;
  if (B > kDecodeParamBatches) {
    prefix_big.resize(B + 1);
    prefix = prefix_big.data();
  }
  prefix[0] = 0;
  bool has_empty = false;
  for (int64_t b = 0; b < B; ++b) {
    prefix[b + 1] = prefix[b] + wlens[b];
    has_empty = has_empty || lens[b] == 0;
  }
  const int64_t g = num_heads / Hkv;
  const int64_t KH = Hkv * (g / decode_heads_per_cta(g, D));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  const bool in_params = B <= kDecodeParamBatches;
  if (!in_params && cudaMemcpyAsync(wsb + ws.prefix, prefix, (B + 1) * sizeof(long long),
                                    cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FA_ERR_RUNTIME;
  const int64_t total = KH * prefix[B];
  // the real lengths of a paged cache: in the launch parameters with the
  // prefix sums, else in the workspace
  if (pg != nullptr && !in_params) {
    std::vector<int> real(B);
    for (int64_t b = 0; b < B; ++b) real[b] = static_cast<int>(lens[b]);
    if (cudaMemcpyAsync(wsb + ws.real_lens, real.data(), B * sizeof(int), cudaMemcpyHostToDevice,
                        s) != cudaSuccess)
      return FA_ERR_RUNTIME;
  }
  // the status word, and the piece counters of the units cut into several
  // pieces, start at zero: one clear on the stream before the launch (a
  // clear inside the decode kernel could erase a timeout another CTA
  // recorded first); for the default plan a kernel of its own rather than a
  // memset, so that the decode kernel plans its first piece while it runs
  // (split_kernel plans after its wait: a memset costs it less)
  const size_t clear_bytes = (total > 0 && max_slots > 1) ? ws.clear : sizeof(uint32_t);
  if (num_splits > 0) {
    if (cudaMemsetAsync(wsb, 0, clear_bytes, s) != cudaSuccess) return FA_ERR_RUNTIME;
  } else {
    if (launch_clear(wsb, clear_bytes, s) != cudaSuccess) return FA_ERR_RUNTIME;
    count_launches(1);
  }

  DecodeLaunch x;
  x.q = q;
  x.k = k;
  x.v = v;
  x.key_mask = key_mask;
  const long long S_mask = std::max<int64_t>(S_kv_max, 1);
  x.mask_bstride = mask_layout == FA_KEY_MASK_B11S   ? S_mask
                   : mask_layout == FA_KEY_MASK_BN1S ? S_mask * num_heads
                                                     : 0;
  x.mask_hstride = mask_layout == FA_KEY_MASK_B11S ? 0 : S_mask;
  x.B = static_cast<int>(B);
  x.Hq = static_cast<int>(num_heads);
  x.Hkv = static_cast<int>(Hkv);
  x.S_kv = static_cast<int>(S_kv_max);
  x.D = static_cast<int>(D);
  x.layout = layout;
  x.scale = scale;
  x.total = total;
  x.rows_per_cta = rc;
  x.piece_cost = pc;
  // a forced split count cuts fixed-size chunks: one CTA per SM takes them in
  // turn and hands them to its consumer warps (split_kernel)
  x.loop_shares = num_splits > 0;
  x.n_ctas = x.loop_shares ? std::min<int64_t>(n_ctas, sms) : n_ctas;
  x.max_slots = static_cast<int>(slots);
  x.prefix_host = prefix;
  x.prefix_dev = in_params ? nullptr : reinterpret_cast<const long long*>(wsb + ws.prefix);
  x.part_o = reinterpret_cast<float*>(wsb + ws.part_o);
  x.part_lse = reinterpret_cast<float*>(wsb + ws.part_lse);
  x.counters = reinterpret_cast<unsigned int*>(wsb + ws.counters);
  x.grp_counters = reinterpret_cast<unsigned int*>(wsb + ws.grp_counters);
  x.grp_lse = reinterpret_cast<float*>(wsb + ws.grp_lse);
  x.grp_o = reinterpret_cast<float*>(wsb + ws.grp_o);
  x.max_groups = static_cast<int>(std::max<int64_t>(groups, 1));
  x.has_empty = has_empty;
  x.block_table = pg != nullptr ? pg->block_table : nullptr;
  x.max_blocks = pg != nullptr ? static_cast<int>(pg->max_blocks) : 0;
  x.num_blocks = pg != nullptr ? static_cast<int>(pg->num_blocks) : 0;
  x.block_size = pg != nullptr ? static_cast<int>(pg->block_size) : 0;
  x.lens_dev = pg != nullptr && !in_params ? reinterpret_cast<const int*>(wsb + ws.real_lens)
                                           : nullptr;
  x.lens_host = pg != nullptr ? lens : nullptr;
  x.out = out;
  x.lse = lse;
  x.status = reinterpret_cast<uint32_t*>(wsb);
  x.timeout_ns = wait_timeout_ns();
  return launch_decode(x, s) == cudaSuccess ? FA_OK : FA_ERR_RUNTIME;
}

}  // namespace

fa_status fa_decode(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                    const int64_t* lens, int64_t B, int64_t S_kv_max, int64_t num_heads,
                    int64_t num_kv_heads, int64_t D, float scale, int layout, int num_splits,
                    void* out, float* lse, void* workspace, size_t workspace_bytes,
                    void* stream) {
  return decode_impl(q, k, v, nullptr, key_mask, lens, B, S_kv_max, num_heads, num_kv_heads, D,
                     scale, layout, num_splits, out, lse, workspace, workspace_bytes, stream);
}

fa_status fa_decode_masked(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                           int key_mask_layout, const int64_t* lens, int64_t B, int64_t S_kv_max,
                           int64_t num_heads, int64_t num_kv_heads, int64_t D, float scale,
                           int layout, int num_splits, void* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream) {
  return decode_impl(q, k, v, nullptr, key_mask, lens, B, S_kv_max, num_heads, num_kv_heads, D,
                     scale, layout, num_splits, out, lse, workspace, workspace_bytes, stream,
                     nullptr, key_mask_layout);
}

fa_status fa_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                          int kv_layout, const int32_t* block_table, int64_t max_blocks_per_seq,
                          int64_t num_blocks, int64_t block_size, const uint8_t* key_mask,
                          const int64_t* lens, int64_t B, int64_t num_heads,
                          int64_t num_kv_heads, int64_t D, float scale, int num_splits, void* out,
                          float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (block_table == nullptr && B > 0) return FA_ERR_NULLPTR;
  if (kv_layout != FA_LAYOUT_PA_BBND && kv_layout != FA_LAYOUT_PA_BNBD) return FA_ERR_PARAM_INVALID;
  if (block_size < 16 || block_size > 1024 || block_size % 16 != 0 || max_blocks_per_seq < 0 ||
      num_blocks < 0 || max_blocks_per_seq > kMaxDim / 1024 || num_blocks > kMaxDim)
    return FA_ERR_PARAM_INVALID;
  const PagedKv pg{block_table, max_blocks_per_seq, std::max<int64_t>(num_blocks, 1), block_size};
  // blocks of PA_BBND hold rows as BSND does (a block is a batch of
  // block_size rows), those of PA_BNBD as BNSD
  const int layout = kv_layout == FA_LAYOUT_PA_BBND ? FA_LAYOUT_BSND : FA_LAYOUT_BNSD;
  return decode_impl(q, k_cache, v_cache, &pg, key_mask, lens, B, max_blocks_per_seq * block_size,
                     num_heads, num_kv_heads, D, scale, layout, num_splits, out, lse, workspace,
                     workspace_bytes, stream);
}

fa_status fa_workspace_status(void* workspace, void* stream) {
  if (workspace == nullptr) return FA_ERR_NULLPTR;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_RUNTIME;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_RUNTIME;
  if (word != 0) {
    if (cudaMemset(workspace, 0, sizeof(word)) != cudaSuccess) return FA_ERR_RUNTIME;
    if (word >= kDevCheckFirst && word <= kDevCheckLast) return FA_ERR_DEVICE_CHECK;
    // every other code but the (impossible) pending-list overflow is an expired wait
    return word == kDevPendingOverflow ? FA_ERR_RUNTIME : FA_ERR_DEVICE_TIMEOUT;
  }
  return FA_OK;
}

fa_status fa_selftest_wait_timeout(void* workspace, uint64_t timeout_ns, void* stream) {
  if (workspace == nullptr) return FA_ERR_NULLPTR;
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return FA_ERR_PARAM_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return FA_ERR_RUNTIME;
  if (launch_wait_probe(static_cast<uint32_t*>(workspace), timeout_ns, s) != cudaSuccess)
    return FA_ERR_RUNTIME;
  count_launches(1);
  return FA_OK;
}

fa_status fa_set_wait_timeout_ns(uint64_t timeout_ns) {
  if (timeout_ns > 10000000000ull) return FA_ERR_PARAM_INVALID;
  tl_timeout_ns = timeout_ns;
  return FA_OK;
}

void fa_set_main_kernel_events(void* before, void* after) {
  tl_before = static_cast<cudaEvent_t>(before);
  tl_after = static_cast<cudaEvent_t>(after);
}

uint64_t fa_kernel_launch_count(void) { return g_launches.load(); }

}  // extern "C"

namespace fa {
fa_status decode_on_scratch(const void* q, const void* k, const void* v,
                            const uint8_t* key_mask, const int64_t* lens, int64_t B,
                            int64_t S_kv_max, int64_t num_heads, int64_t num_kv_heads, int64_t D,
                            float scale, int layout, int num_splits, void* out, float* lse,
                            fa_status (*scratch)(void**), size_t scratch_bytes, void* stream) {
  return decode_impl(q, k, v, nullptr, key_mask, lens, B, S_kv_max, num_heads, num_kv_heads, D,
                     scale, layout, num_splits, out, lse, nullptr, scratch_bytes, stream,
                     scratch);
}
}  // namespace fa
