// Split-KV decode (S_q = 1) for sm_103a.
//
// Work space. Every (batch b, KV head, group of G query heads) is a unit of
// L_b key rows; the units are laid end to end in one global row space of
// T = KH * sum_b L_b rows (KH = KV heads x head groups), and CTA i takes the
// rows [i*Rc, (i+1)*Rc): every CTA gets the same amount of K/V to stream,
// and a CTA's range is cut into pieces only where it crosses a unit boundary
// (the load-balancing idea of the FlashAttn guide §4, SectionStreamK: split
// the KV axis so that all cores carry equal cost, and merge the split rows
// afterwards, FlashAttn guide §1.9).
//
// Stage 1 (decode_kernel): the producer warp streams each piece's K and V
// rows (112-row stages; a piece's last, partial stage with 16-row boxes)
// through one 168 KB shared-memory ring with TMA tensor loads, without a
// break between pieces; q arrives with a piece's first stage. Seven consumer
// warps compute q.k with 128-bit shared loads, packed f32x2 FMAs and a
// butterfly over the 8 lanes that share a row (the G query heads of a GQA
// group reuse each K/V row), keep an online softmax per head (running max m
// and sum l, exp2 domain) and accumulate p*v. This is the FlashDecoding
// tutorial's stage 1 (§3.2) with the scale and the length mask applied.
// At the end of a piece every warp parks its (m, l, o) in a double-buffered
// scratch slot; once all seven have, each combines a slice of the piece's
// normalised partial o/l and log-sum-exp (or, when the piece is the whole
// unit, of the final output).
//
// Stage 2 (in the same kernel): a unit cut into several pieces is counted in
// a per-unit counter (cleared before the launch) when a CTA finishes; the
// CTA that completes the count merges the unit's pieces for every query head
// by their log-sum-exp with the largest value factored out, in piece order:
//   M = max_c lse_c, w_c = 2^(lse_c - M), out = sum_c w_c o_c / sum_c w_c,
//   lse = M + log2(sum_c w_c)  (reported as natural log)
// which is aclnnIncreFlashAttention guide §8.3's combine() and the FlashAttn
// guide §10 formula written for normalised partials (FlashDecoding tutorial
// §3.3). No CTA waits for another: the merge is a stream-K fixup by whichever
// finishes last. A sequence of length 0 gets out = 0, lse = +inf (FlashAttn
// guide §1.7).
//
// Rows at or past a batch's length are never used by any arithmetic (they
// may land in shared memory with the rest of a box and are skipped), so
// stale cache contents, NaN included, cannot reach the output.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

// 7 consumer warps + 1 producer warp: 256 threads keeps the per-thread
// register budget at 255 (larger CTAs are capped at 168).
constexpr int kDecWarps = 7;                       // consumer warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + one producer warp
constexpr int kRingBytes = 172032;                 // K/V ring (168 KB)
constexpr int kMaxStages = 6;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D, int G>
struct DecCfg {
  // lanes per K/V row: 8 (D = 64: one 16-byte chunk each; D = 128: two),
  // 16 for D = 256 (two chunks each), so that q and o of a GQA group of up to
  // four heads fit the registers
  static constexpr int LPR = D == 256 ? 16 : 8;
  static constexpr int LOG_LPR = D == 256 ? 4 : 3;
  static constexpr int NCH = D / (8 * LPR);         // 16-byte chunks of a row per lane
  static constexpr int RPW = 32 / LPR;              // rows per warp per step (row groups)
  // rows per stage: 112, or 56 for D = 256 (three stages in the ring)
  static constexpr int R = D == 256 ? 56 : kDecodeStageRows;
  static constexpr int TAIL = D == 256 ? 8 : 16;    // rows per box of a partial stage
  static constexpr int RPWS = R / kDecWarps;        // rows per warp per stage (16 or 8)
  static constexpr int STEPS = RPWS / RPW;          // 4
  static constexpr int TILE_BYTES = R * D * 2;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int NST = kRingBytes / STAGE_BYTES;  // 3 (D = 128, 256) or 6 (D = 64)
  static constexpr int NP = 4 * NCH;                // fp32 pairs per lane per head
  static constexpr int LG = G >= 8 ? 3 : G >= 4 ? 2 : G >= 2 ? 1 : 0;  // log2(G)
  static constexpr int SHIFT = LOG_LPR - LG;        // head of lane `sub`: sub >> SHIFT
  static constexpr int QB = G * D * 2 > 1024 ? 2048 : 1024;  // q of one piece
  // one scratch buffer: m[warps][G] and l[warps][G], each padded to a
  // multiple of 4 floats so that o[warps][G][D] and the next buffer stay
  // 16-byte aligned for the float4 accesses; two buffers unless D = 256
  static constexpr int NSB = D == 256 ? 1 : 2;
  static constexpr int MG = (kDecWarps * G + 3) / 4 * 4;
  static constexpr int SCRATCH_FLOATS = 2 * MG + kDecWarps * G * D;
  static constexpr int SMEM = kRingBytes + NSB * SCRATCH_FLOATS * 4 + kMaxStages * QB + 1024;
  static_assert(SCRATCH_FLOATS % 4 == 0, "scratch alignment");
  static_assert(NST <= kMaxStages, "ring slots");
  static_assert(R % (kDecWarps * RPW) == 0 && R % TAIL == 0, "stage rows");
  static_assert(SMEM <= 232448, "shared memory");
};

// Where the length prefix sums live: launch parameters for small batches,
// else the workspace.
struct Prefix {
  const long long* global;  // [B + 1] or null
  long long local[kDecodeParamBatches + 1];
  __device__ __forceinline__ long long operator[](int i) const {
    return global != nullptr ? global[i] : local[i];
  }
};

struct DecodeArgs {
  const __nv_bfloat16* q;
  const uint8_t* key_mask;
  float* part_o;     // [B][Hq][max_slots][D]
  float* part_lse;   // [B][Hq][max_slots], log2 domain
  unsigned int* counters;  // [B * KH] pieces finished per unit (zero at launch)
  int has_empty;           // some sequence has length 0
  int piece_cost;          // cost of a unit start after the first (0: shares of rows)
  __nv_bfloat16* out;
  float* lse;
  uint32_t* status;
  uint64_t timeout_ns;
  long long total;         // rows of the work space
  long long rows_per_cta;  // Rc: cost of each CTA's share (a row costs 1)
  int B, Hq, Hkv, S_kv, max_slots, head_groups, G;
  float scale_log2;
  // paged K/V: block table [B][max_blocks] (null: contiguous cache), the
  // real lengths (the work space holds them rounded up to 16 rows)
  const int32_t* block_table;
  int max_blocks, block_size;
  const int* real_len;     // [B] in the workspace (paged, large batches only)
  // paged, batches that travel in the parameters: how far each length was
  // rounded up (the real length is the work-space length minus this)
  unsigned char pad16[kDecodeParamBatches];
  Prefix prefix;           // prefix[b] = sum of lengths of batches < b (work space)
  // key mask element (b, query head h, key j) at key_mask[b * mask_bstride +
  // h * mask_hstride + j]: (B, 1, 1, S) has mask_hstride 0, (1, N, 1, S)
  // mask_bstride 0
  long long mask_bstride, mask_hstride;
  // forced split counts (split_kernel): the pieces of a unit are merged in
  // groups of kMergeGroup slots, then the groups; group partials
  // [B][Hq][max_groups][D] (normalised) and [B][Hq][max_groups] (log2 lse),
  // piece counters per group [units][max_groups] (group counters per unit in
  // `counters`)
  float* grp_o;
  float* grp_lse;
  unsigned int* grp_counters;
  int max_groups;
  // shares cut by cost: the first row of CTA c's share at prefix.local[share_off
  // + c] (c = 0 .. gridDim.x, the last entry the end of the work space),
  // computed on the host; -1: found by the kernel
  int share_off;
};

// Largest b with KH * (prefix[b] + pc * b) <= r: with pc = 0 the batch whose
// rows hold row r (batches of length 0 own no row and are passed over), with
// pc = the piece cost the batch whose range of costs holds cost r. Small
// batches count the entries at or below r with independent loads, larger
// ones bisect.
__device__ __forceinline__ int find_batch(const Prefix& p, int B, long long KH, long long pc,
                                          long long r) {
  if (B <= 64) {
    int b = 0;
#pragma unroll 8
    for (int i = 1; i < B; ++i) b += (KH * (p[i] + pc * i) <= r) ? 1 : 0;
    return b;
  }
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (KH * (p[mid] + pc * mid) <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// n / d for non-negative n and positive d, in 32 bits when both fit.
__device__ __forceinline__ long long div_nn(long long n, long long d) {
  if (((n | d) >> 32) == 0)
    return static_cast<long long>(static_cast<uint32_t>(n) / static_cast<uint32_t>(d));
  return n / d;
}

// Per-slot header the producer writes before the slot's loads, so consumers
// need no global lookups.
struct SlotHeader {
  int piece;   // piece counter of this CTA, -1 = no more work
  int stage;   // stage index within the piece
  int nstage;  // stages of the piece
  int b, kh, row0, rows, slot, nsp;
  int vend;    // rows of the piece that hold keys (< rows only past a paged length)
};

// Merge the nsp normalised partials of one (batch, query head) row into the
// output (one warp): all lse and o loads of up to 8 pieces are in flight
// before any is used, the largest lse is factored out.
template <int D>
__device__ __forceinline__ void merge_row(const DecodeArgs& a, size_t row, int nsp, int lane) {
  constexpr int EPL = D / 32;  // output elements per lane
  if (!FA_CHECK(nsp <= a.max_slots && row < static_cast<size_t>(a.B) * a.Hq, a.status,
                kDevCheckDecodeMerge))
    return;
  const float* pl = a.part_lse + row * a.max_slots;
  const float* po = a.part_o + row * a.max_slots * D + lane * EPL;
  float M = -INFINITY, W = 0.f, acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  for (int k0 = 0; k0 < nsp; k0 += 8) {
    float lk[8], v[8][EPL];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = k0 + u < nsp;
      lk[u] = in ? __ldcg(pl + k0 + u) : -INFINITY;
      if constexpr (EPL % 4 == 0) {
#pragma unroll
        for (int e = 0; e < EPL; e += 4) {
          const float4 t =
              in ? __ldcg(reinterpret_cast<const float4*>(po + static_cast<size_t>(k0 + u) * D + e))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
          v[u][e] = t.x; v[u][e + 1] = t.y; v[u][e + 2] = t.z; v[u][e + 3] = t.w;
        }
      } else {
        const float2 t = in ? __ldcg(reinterpret_cast<const float2*>(po + static_cast<size_t>(k0 + u) * D))
                            : make_float2(0.f, 0.f);
        v[u][0] = t.x; v[u][1] = t.y;
      }
    }
    float mb = M;
#pragma unroll
    for (int u = 0; u < 8; ++u) mb = fmaxf(mb, lk[u]);
    if (mb == -INFINITY) continue;  // only empty pieces so far
    const float sc = ex2(M - mb);   // rescale what was summed under the old maximum (0 at first)
    W *= sc;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= sc;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float wk = ex2(lk[u] - mb);  // empty or absent piece: 0
      W += wk;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wk, v[u][e], acc[e]);
    }
    M = mb;
  }
  const bool invalid = (M == -INFINITY);
  const float inv = invalid ? 0.f : 1.f / W;
  __nv_bfloat16* dst = a.out + row * D + lane * EPL;
  if constexpr (EPL % 4 == 0) {
#pragma unroll
    for (int e = 0; e < EPL; e += 4)
      *reinterpret_cast<uint2*>(dst + e) = make_uint2(pack_bf16x2(acc[e] * inv, acc[e + 1] * inv),
                                                      pack_bf16x2(acc[e + 2] * inv, acc[e + 3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0 && a.lse != nullptr) a.lse[row] = invalid ? INFINITY : (M + log2f(W)) * kLn2;
}

struct Pending {
  int unit, nsp, b, kh;
};

// How the work space is cut into shares, one instantiation each so that the
// code of the common case carries nothing of the other:
//   kSharesRows  one share per CTA, equal in rows
//   kSharesCost  one share per CTA, equal in cost (piece_cost > 0)
// (a forced split count runs split_kernel instead)
constexpr int kSharesRows = 0, kSharesCost = 1;

template <int D, int G, int kShares>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_k16,
                  const __grid_constant__ CUtensorMap tm_v16,
                  const __grid_constant__ DecodeArgs a) {
  using C = DecCfg<D, G>;
  constexpr int NP = C::NP;
  constexpr int NST = C::NST;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* scratch = reinterpret_cast<float*>(smem + kRingBytes);  // NSB buffers
  unsigned char* qbuf = smem + kRingBytes + C::NSB * C::SCRATCH_FLOATS * 4;
  uint64_t* bars = reinterpret_cast<uint64_t*>(qbuf + kMaxStages * C::QB);
  // bars: full[kMaxStages], empty[kMaxStages], scratch free[2], scratch parked[2]
  SlotHeader* hdr = reinterpret_cast<SlotHeader*>(bars + 2 * kMaxStages + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(hdr + kMaxStages);
  // split pieces of this CTA (at most its first and its last): counted at the end
  int* n_pending = const_cast<int*>(abort_flag) + 1;
  Pending* pending = reinterpret_cast<Pending*>(n_pending + 3);  // [2]
  constexpr int kPendingCap = 2;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long KH = static_cast<long long>(a.Hkv) * a.head_groups;
  const int g_total = a.Hq / a.Hkv;

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kMaxStages);
  const uint32_t sfree0 = smem_u32(bars + 2 * kMaxStages);
  const uint32_t parked0 = smem_u32(bars + 2 * kMaxStages + 2);
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kDecWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sfree0 + 8 * i, kDecWarps);
      mbar_init(parked0 + 8 * i, kDecWarps);
    }
    *abort_flag = 0;
    *n_pending = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // The consumers' code comes first and the producer's after: a consumer's
  // first stage runs code no warp has run yet (from L2 or HBM when the caches
  // are cold), and this keeps that code where it is whatever the producer's
  // planning code holds (with the producer first, the cost-cut plan's extra
  // code before it made the first stage ≈2.5 µs slower).
  if (warp != kDecWarps) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // (the status word was cleared on the stream before this kernel)
    // work queued after this kernel may be scheduled as soon as SMs free up
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (a.has_empty) {
      // sequences of length 0: out = 0, lse = +inf; one thread per row
      for (int row = static_cast<int>(blockIdx.x) * kDecWarps * 32 + tid; row < a.B * a.Hq;
           row += static_cast<int>(gridDim.x) * kDecWarps * 32) {
        const int b = row / a.Hq;
        if (a.prefix[b + 1] != a.prefix[b]) continue;
        uint4* dst = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * D);
#pragma unroll
        for (int i = 0; i < D * 2 / 16; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
        if (a.lse != nullptr) a.lse[row] = INFINITY;
      }
    }
    // ================================================================ consumers
    // Lane layout: the LPR = 8 lanes of a row group share one K/V row (lane
    // `sub` owns its 16-byte chunks sub, sub+8). Every lane holds the q and o
    // of all G heads in the order j -> head j ^ x, x = sub >> SHIFT: with that
    // order the butterfly over the 8 lanes halves the heads still carried at
    // each of its first log2(G) levels, so that a lane ends with the full dot
    // product of one head, head x (the lanes sub with equal x hold the same
    // one), in log2(8) levels of G - 1 + (3 - log2 G) shuffles instead of 3G.
    // The softmax of a row group runs per lane for head x; p and the
    // rescale factor of the other heads come back by G - 1 shuffles.
    const int sub = lane % C::LPR;
    const int rg = lane / C::LPR;  // row group within a warp step
    const int x = sub >> C::SHIFT;
    float m = -INFINITY, l = 0.f;  // head x of this row group
    uint64_t o[G][NP];
    uint64_t qp[G][NP];  // q * scale * log2(e) of head j ^ x, as fp32 pairs
    int row_begin = 0, row_end = 0, piece_seq = -1;
    const uint8_t* mask_row = nullptr;

    for (int st = 0;; ++st) {
      const int slot = st % NST;
      bool got = mbar_wait_polled(full0 + 8 * slot, (st / NST) & 1, a.timeout_ns, a.status,
                           kDevTimeoutDecodeFull, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) break;
      const SlotHeader hd = hdr[slot];
      if (hd.piece < 0) break;

      if (hd.stage == 0) {
        // ---- a new piece: q landed with this stage; fresh softmax state
        ++piece_seq;
        row_begin = hd.row0;
        row_end = hd.row0 + hd.vend;  // rows past a paged length hold no key
        // the mask row of this lane's head x (the same row for every head of a
        // (B, 1, 1, S) mask)
        mask_row = nullptr;
        if (a.key_mask != nullptr) {
          const long long h0 = static_cast<long long>(hd.kh / a.head_groups) * g_total +
                               static_cast<long long>(hd.kh % a.head_groups) * G + x;
          mask_row = a.key_mask + hd.b * a.mask_bstride + h0 * a.mask_hstride;
        }
        const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(qbuf + slot * C::QB);
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int j = 0; j < G; ++j) {
#pragma unroll
          for (int k = 0; k < NP; ++k) o[j][k] = 0ull;
#pragma unroll
          for (int ch = 0; ch < C::NCH; ++ch) {
            const uint4 u = *reinterpret_cast<const uint4*>(qs + (j ^ x) * D + (sub + C::LPR * ch) * 8);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              qp[j][ch * 4 + k] = pair_f32(bf16lo_to_f32(w4[k]) * a.scale_log2,
                                           bf16hi_to_f32(w4[k]) * a.scale_log2);
          }
        }
      }

      // ---- one stage: R rows of K and V
      const __nv_bfloat16* Ks = reinterpret_cast<const __nv_bfloat16*>(smem + slot * C::STAGE_BYTES);
      const __nv_bfloat16* Vs = Ks + C::R * D;
      const int stage_row0 = row_begin + hd.stage * C::R;
      // every row of the stage holds a key: no per-row checks
      const bool dense = mask_row == nullptr && stage_row0 + C::R <= row_end;
      float s[C::STEPS];
      bool valid[C::STEPS];  // some head of the row group sees the key
#pragma unroll
      for (int i = 0; i < C::STEPS; ++i) {
        const int r = warp * C::RPWS + i * C::RPW + rg;
        const int gr = stage_row0 + r;
        bool ok = true;
        if (!dense) {
          ok = gr < row_end;
          if (ok && mask_row != nullptr) ok = mask_row[gr] == 0;  // head x
          // the V row is zeroed only when no head of the row group sees it
          const uint32_t seen = __ballot_sync(0xffffffffu, ok) >> (rg * C::LPR);
          valid[i] = (seen & ((1u << C::LPR) - 1u)) != 0u;
        } else {
          valid[i] = true;
        }
        uint64_t kp[NP];
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          const uint4 u = *reinterpret_cast<const uint4*>(Ks + r * D + (sub + C::LPR * ch) * 8);
          kp[ch * 4 + 0] = bf16x2_pair(u.x);
          kp[ch * 4 + 1] = bf16x2_pair(u.y);
          kp[ch * 4 + 2] = bf16x2_pair(u.z);
          kp[ch * 4 + 3] = bf16x2_pair(u.w);
        }
        float part[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
          // with few heads, two chains of FMAs keep the pipe busy
          uint64_t acc = ffma2(qp[j][0], kp[0], 0ull);
          if constexpr (G <= 2) {
            uint64_t acc2 = ffma2(qp[j][1], kp[1], 0ull);
#pragma unroll
            for (int k = 2; k < NP; k += 2) {
              acc = ffma2(qp[j][k], kp[k], acc);
              acc2 = ffma2(qp[j][k + 1], kp[k + 1], acc2);
            }
            acc = fadd2(acc, acc2);
          } else {
#pragma unroll
            for (int k = 1; k < NP; ++k) acc = ffma2(qp[j][k], kp[k], acc);
          }
          const float2 a2 = unpair(acc);
          part[j] = a2.x + a2.y;
        }
        // butterfly: the first log2(G) levels keep the lower half of the
        // heads still carried and receive the partner's sums of the same heads
#pragma unroll
        for (int lv = 0; lv < C::LG; ++lv) {
          const int half = G >> (lv + 1);
#pragma unroll
          for (int j = 0; j < half; ++j)
            part[j] += __shfl_xor_sync(0xffffffffu, part[j + half], (C::LPR / 2) >> lv);
        }
#pragma unroll
        for (int lv = C::LG; lv < C::LOG_LPR; ++lv)
          part[0] += __shfl_xor_sync(0xffffffffu, part[0], (C::LPR / 2) >> lv);
        s[i] = ok ? part[0] : -INFINITY;
      }
      // online softmax of head x over this warp's rows of the stage: the
      // running max is shared by the 4 row groups (so that their sums and
      // accumulators add up without rescaling at the end of the piece)
      float mx = s[0];
#pragma unroll
      for (int i = 1; i < C::STEPS; ++i) mx = fmaxf(mx, s[i]);
#pragma unroll
      for (int off = C::LPR; off < 32; off <<= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m, mx);
      const float m_use = (mn == -INFINITY) ? 0.f : mn;
      const float alpha = ex2(m - m_use);  // 0 when m was -inf
      m = mn;
      float ps = 0.f;
#pragma unroll
      for (int i = 0; i < C::STEPS; ++i) {
        s[i] = ex2(s[i] - m_use);  // -inf -> 0
        ps += s[i];
      }
      l = fmaf(l, alpha, ps);
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        // some running maximum moved: rescale the accumulators of every head
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float aj = j == 0 ? alpha : __shfl_xor_sync(0xffffffffu, alpha, j << C::SHIFT);
          const uint64_t a2 = pair_f32(aj, aj);
#pragma unroll
          for (int k = 0; k < NP; ++k) o[j][k] = fmul2(o[j][k], a2);
        }
      }
#pragma unroll
      for (int i = 0; i < C::STEPS; ++i) {
        const int r = warp * C::RPWS + i * C::RPW + rg;
        uint64_t vp[NP];
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          uint4 u = *reinterpret_cast<const uint4*>(Vs + r * D + (sub + C::LPR * ch) * 8);
          if (!dense && !valid[i]) u = make_uint4(0u, 0u, 0u, 0u);  // stale rows never enter a product
          vp[ch * 4 + 0] = bf16x2_pair(u.x);
          vp[ch * 4 + 1] = bf16x2_pair(u.y);
          vp[ch * 4 + 2] = bf16x2_pair(u.z);
          vp[ch * 4 + 3] = bf16x2_pair(u.w);
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float pj = j == 0 ? s[i] : __shfl_xor_sync(0xffffffffu, s[i], j << C::SHIFT);
          const uint64_t p2 = pair_f32(pj, pj);
#pragma unroll
          for (int k = 0; k < NP; ++k) o[j][k] = ffma2(p2, vp[k], o[j][k]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
      if (hd.stage != hd.nstage - 1) continue;

      // ================================================= end of the piece
      // 1) this warp's state: m is shared by the row groups, l and o add up.
      //    The accumulators are halved across the row groups (lanes xor LPR,
      //    then xor 2 LPR when there are four): a lane keeps one half and adds
      //    the partner's copy of it, so that it ends with 1/RPW of them,
      //    summed over the warp.
#pragma unroll
      for (int off = C::LPR; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      constexpr int F = G * NP;  // accumulator pairs of a lane, slot-major
      constexpr int FQ = F / C::RPW;  // pairs a lane keeps
      const bool b0 = (rg & 1) != 0, b1 = (rg & 2) != 0;
      uint64_t h1[F / 2];
#pragma unroll
      for (int f = 0; f < F / 2; ++f) {
        const uint64_t lo = o[f / NP][f % NP], hi = o[(f + F / 2) / NP][(f + F / 2) % NP];
        const uint64_t keep = b0 ? hi : lo, send = b0 ? lo : hi;
        const float2 sp = unpair(send);
        const float rx = __shfl_xor_sync(0xffffffffu, sp.x, C::LPR);
        const float ry = __shfl_xor_sync(0xffffffffu, sp.y, C::LPR);
        h1[f] = fadd2(keep, pair_f32(rx, ry));
      }
      uint64_t hq[FQ];
      if constexpr (C::RPW == 4) {
#pragma unroll
        for (int f = 0; f < F / 4; ++f) {
          const uint64_t keep = b1 ? h1[f + F / 4] : h1[f], send = b1 ? h1[f] : h1[f + F / 4];
          const float2 sp = unpair(send);
          const float rx = __shfl_xor_sync(0xffffffffu, sp.x, 2 * C::LPR);
          const float ry = __shfl_xor_sync(0xffffffffu, sp.y, 2 * C::LPR);
          hq[f] = fadd2(keep, pair_f32(rx, ry));
        }
      } else {
#pragma unroll
        for (int f = 0; f < FQ; ++f) hq[f] = h1[f];
      }
      // 2) park the state in scratch buffer piece_seq % NSB, once the combine
      //    of the piece that used it last has released it
      const int buf = piece_seq % C::NSB;
      const int use = piece_seq / C::NSB;
      const uint32_t use_parity = use & 1;
      if (use >= 1) {
        bool fr = mbar_wait_polled(sfree0 + 8 * buf, use_parity ^ 1, a.timeout_ns, a.status,
                            kDevTimeoutDecodeFull, abort_flag);
        fr = __all_sync(0xffffffffu, fr);
        if (!fr) break;
      }
      float* sb = scratch + buf * C::SCRATCH_FLOATS;
      float* sm_m = sb;              // [warps][G]
      float* sm_l = sb + C::MG;      // [warps][G]
      float* sm_o = sb + 2 * C::MG;  // [warps][G][D], 16-byte aligned
      if (rg == 0 && (sub & ((1 << C::SHIFT) - 1)) == 0) {  // one lane per head x
        sm_m[warp * G + x] = m;
        sm_l[warp * G + x] = l;
      }
      {
        // the lane's share: pairs base + f of the slot-major accumulators
        const int base = (b0 ? F / 2 : 0) + (b1 ? F / 4 : 0);
        if constexpr (FQ == 1) {
          const int j = base / NP, k = base % NP;
          const int d = (sub + C::LPR * (k / 4)) * 8 + 2 * (k % 4);
          *reinterpret_cast<float2*>(sm_o + (warp * G + (j ^ x)) * D + d) = unpair(hq[0]);
        } else {
#pragma unroll
          for (int f = 0; f < FQ; f += 2) {
            const int fl = base + f;
            const int j = fl / NP, k = fl % NP;  // k even: the pair and the next share a chunk
            const int d = (sub + C::LPR * (k / 4)) * 8 + 2 * (k % 4);
            const float2 v0 = unpair(hq[f]);
            const float2 v1 = unpair(hq[f + 1]);
            *reinterpret_cast<float4*>(sm_o + (warp * G + (j ^ x)) * D + d) =
                make_float4(v0.x, v0.y, v1.x, v1.y);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(parked0 + 8 * buf);
      // 3) every consumer warp combines a slice of the G x D results once all
      //    of them have parked
      bool pk = mbar_wait_polled(parked0 + 8 * buf, use_parity, a.timeout_ns, a.status,
                          kDevTimeoutDecodeFull, abort_flag);
      pk = __all_sync(0xffffffffu, pk);
      if (!pk) break;
      {
        const int kvh = hd.kh / a.head_groups;
        const int hg = hd.kh % a.head_groups;
        const size_t bh0 = static_cast<size_t>(hd.b) * a.Hq + kvh * g_total + hg * G;
        for (int t = warp * 32 + lane; t < G * D / 4; t += kDecWarps * 32) {
          const int h = (t * 4) / D, d = (t * 4) % D;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm_m[w * G + h]);
          const bool empty = (M == -INFINITY);
          float Ls = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) {
            const float fw = empty ? 0.f : ex2(sm_m[w * G + h] - M);
            Ls = fmaf(sm_l[w * G + h], fw, Ls);
            const float4 v = *reinterpret_cast<const float4*>(sm_o + (w * G + h) * D + d);
            acc.x = fmaf(v.x, fw, acc.x);
            acc.y = fmaf(v.y, fw, acc.y);
            acc.z = fmaf(v.z, fw, acc.z);
            acc.w = fmaf(v.w, fw, acc.w);
          }
          const float inv = empty ? 0.f : 1.f / Ls;
          acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          if (!FA_CHECK(bh0 + h < static_cast<size_t>(a.B) * a.Hq, a.status, kDevCheckDecodeRow) ||
              !FA_CHECK(hd.nsp == 1 || hd.slot < a.max_slots, a.status, kDevCheckDecodeSlot))
            continue;
          if (hd.nsp == 1) {
            __nv_bfloat16* dst = a.out + (bh0 + h) * D + d;
            *reinterpret_cast<uint2*>(dst) =
                make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
            if (d == 0 && a.lse != nullptr)
              a.lse[bh0 + h] = empty ? INFINITY : (M + log2f(Ls)) * kLn2;
          } else {
            *reinterpret_cast<float4*>(a.part_o + ((bh0 + h) * a.max_slots + hd.slot) * D + d) = acc;
            if (d == 0)
              a.part_lse[(bh0 + h) * a.max_slots + hd.slot] = empty ? -INFINITY : M + log2f(Ls);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(sfree0 + 8 * buf);  // this warp is done with the buffer
        if (warp == 0 && hd.nsp > 1) {
          const int i = (*n_pending)++;
          if (i < kPendingCap)
            pending[i] = Pending{static_cast<int>(hd.b * KH + hd.kh), hd.nsp, hd.b, hd.kh};
          else
            record_error(a.status, kDevPendingOverflow);  // the host plan prevents this
        }
      }
    }
  } else {
    // ================================================================ producer
    // The shares are equal in cost: a row costs 1 and, when piece_cost > 0,
    // the start of every unit after the first costs piece_cost more (the
    // piece end it brings), so that a share holding unit starts takes fewer
    // rows. Row x of unit k costs x + piece_cost * k; CTA c holds the rows of
    // cost [c Rc, (c+1) Rc).
    const long long Rc = a.rows_per_cta;
    constexpr bool kWeighted = kShares == kSharesCost;
    const long long pc = kWeighted ? a.piece_cost : 0;
    // the first row whose cost is at least T
    auto row_at_cost = [&](long long T) -> long long {
      const int b = find_batch(a.prefix, a.B, KH, pc, T);
      const long long L = a.prefix[b + 1] - a.prefix[b];
      const long long cb = KH * (a.prefix[b] + pc * b);  // cost of the batch's first row
      const long long kh = min(KH - 1, div_nn(T - cb, L + pc));  // L + pc > 0 here
      const long long off = T - cb - kh * (L + pc);
      const long long u0 = KH * a.prefix[b] + kh * L;
      return off < L ? u0 + off : u0 + L;  // in the gap before the next unit: its first row
    };
    const long long T0 = static_cast<long long>(blockIdx.x) * Rc;
    long long r = T0;
    long long r1 = min(T0 + Rc, a.total);
    long long v = blockIdx.x;  // the share being planned
    if constexpr (kWeighted) {
      if (a.share_off >= 0) {
        r = a.prefix.local[a.share_off + blockIdx.x];
        r1 = a.prefix.local[a.share_off + blockIdx.x + 1];
      } else {
        if (T0 > 0) r = row_at_cost(T0);
        r1 = blockIdx.x + 1 == gridDim.x ? a.total : min(row_at_cost(T0 + Rc), a.total);
      }
    }
    // the next piece of this CTA's range [r, r1): its unit, rows and stages
    auto plan = [&](int piece, SlotHeader& h, int& kvh, int& hg) {
      h = SlotHeader{-1, 0, 1, 0, 0, 0, 0, 0, 0, 0};
      if (r >= r1) return;
      const int b = find_batch(a.prefix, a.B, KH, 0, r);
      const long long base = KH * a.prefix[b];
      const long long L = a.prefix[b + 1] - a.prefix[b];
      const long long kh = div_nn(r - base, L);
      const long long u0 = base + kh * L;  // the unit's first row in the work space
      const long long u1 = u0 + L;
      const long long rows = min(u1, r1) - r;
      h.piece = piece;
      h.b = b;
      h.kh = static_cast<int>(kh);
      h.row0 = static_cast<int>(r - u0);
      h.rows = static_cast<int>(rows);
      const long long cu = kWeighted ? u0 + pc * (b * KH + kh) : u0;  // cost of its first row
      const long long c0 = div_nn(cu, Rc);  // the CTA holding the unit's first row
      h.slot = static_cast<int>(v - c0);
      h.nsp = static_cast<int>(div_nn(cu + L - 1, Rc) - c0 + 1);
      h.nstage = static_cast<int>((rows + C::R - 1) / C::R);
      h.vend = h.rows;
      if (a.block_table != nullptr) {
        const long long real = a.real_len != nullptr ? __ldg(a.real_len + b) : L - a.pad16[b];
        h.vend = static_cast<int>(max(0ll, min(static_cast<long long>(h.rows), real - h.row0)));
      }
      kvh = h.kh / a.head_groups;
      hg = h.kh % a.head_groups;
      r += rows;
      if (!FA_CHECK(b >= 0 && b < a.B && kh >= 0 && kh < KH && h.row0 >= 0 && rows > 0 &&
                        h.row0 + rows <= L && h.slot >= 0 && h.slot < h.nsp,
                    a.status, kDevCheckDecodePiece))
        h.piece = -1;  // stop: nothing of this piece is loaded
    };
    SlotHeader h{};
    int kvh = 0, hg = 0;
    // the first piece needs only the launch parameters (unless the prefix
    // sums or the paged lengths sit in the workspace): plan it while the
    // work before this kernel may still be running
    const bool early = a.prefix.global == nullptr && a.real_len == nullptr;
    if (lane == 0) {
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_k16);
      tma_prefetch_map(&tm_v16);
      if (early) plan(0, h, kvh, hg);
    }
    // launched with programmatic dependent launch: wait until the work that
    // precedes this kernel on the stream (which may produce q, K, V) is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (lane == 0) {
      int st = 0;  // stages issued by this CTA
      bool ok = true;
      // the first stage, when it is a full stage of a contiguous cache, is
      // issued here, next to the planning code, rather than from the loop
      // below (whose code is then fetched while the stage is in flight)
      bool first_issued = false;
      if (early && h.piece >= 0 && a.block_table == nullptr && h.rows >= C::R) {
        h.stage = 0;
        hdr[0] = h;
        mbar_expect_tx(full0, C::STAGE_BYTES + G * D * 2);
        tma_load_4d(smem_u32(smem), &tm_k, full0, 0, h.row0, kvh, h.b);
        tma_load_4d(smem_u32(smem + C::TILE_BYTES), &tm_v, full0, 0, h.row0, kvh, h.b);
        bulk_load(smem_u32(qbuf), a.q + (static_cast<size_t>(h.b) * a.Hq + kvh * g_total + hg * G) * D,
                  G * D * 2, full0);
        first_issued = true;
        st = 1;
      }
      for (int piece = 0; ok; ++piece) {
        if (piece > 0 || !early) plan(piece, h, kvh, hg);
        const bool done = h.piece < 0;
        for (int s = piece == 0 && first_issued ? 1 : 0; s < h.nstage; ++s, ++st) {
          const int slot = st % NST;
          const int use = st / NST;
          if (use > 0 && !mbar_wait_polled(empty0 + 8 * slot, (use - 1) & 1, a.timeout_ns, a.status,
                                    kDevTimeoutDecodeEmpty, abort_flag)) {
            ok = false;
            break;
          }
          h.stage = s;
          hdr[slot] = h;
          if (done) {
            mbar_arrive(full0 + 8 * slot);  // end marker: no data
            ok = false;
            ++st;
            break;
          }
          const uint32_t dst = smem_u32(smem + slot * C::STAGE_BYTES);
          const int row = h.row0 + s * C::R;
          const int rows_here = min(C::R, h.rows - s * C::R);
          const uint32_t q_bytes = s == 0 ? G * D * 2 : 0;
          if (a.block_table != nullptr) {
            // paged: 16-row boxes (pieces and lengths are multiples of 16 rows in
            // the work space, blocks are multiples of 16 rows), each from its block
            const int nb = (rows_here + C::TAIL - 1) / C::TAIL;
            mbar_expect_tx(full0 + 8 * slot, 2 * nb * C::TAIL * D * 2 + q_bytes);
            const int32_t* bt = a.block_table + static_cast<size_t>(h.b) * a.max_blocks;
            for (int t = 0; t < nb; ++t) {
              const int lr = row + t * C::TAIL;
              const int blk = __ldg(bt + lr / a.block_size);
              const int in_blk = lr % a.block_size;
              tma_load_4d(dst + t * C::TAIL * D * 2, &tm_k16, full0 + 8 * slot, 0, in_blk, kvh,
                          blk);
              tma_load_4d(dst + C::TILE_BYTES + t * C::TAIL * D * 2, &tm_v16, full0 + 8 * slot,
                          0, in_blk, kvh, blk);
            }
          } else if (rows_here == C::R) {
            mbar_expect_tx(full0 + 8 * slot, C::STAGE_BYTES + q_bytes);
            tma_load_4d(dst, &tm_k, full0 + 8 * slot, 0, row, kvh, h.b);
            tma_load_4d(dst + C::TILE_BYTES, &tm_v, full0 + 8 * slot, 0, row, kvh, h.b);
          } else {
            // partial last stage: 16-row boxes, only as many as the piece needs
            const int nb = (rows_here + C::TAIL - 1) / C::TAIL;
            mbar_expect_tx(full0 + 8 * slot, 2 * nb * C::TAIL * D * 2 + q_bytes);
            for (int t = 0; t < nb; ++t) {
              tma_load_4d(dst + t * C::TAIL * D * 2, &tm_k16, full0 + 8 * slot, 0,
                          row + t * C::TAIL, kvh, h.b);
              tma_load_4d(dst + C::TILE_BYTES + t * C::TAIL * D * 2, &tm_v16, full0 + 8 * slot,
                          0, row + t * C::TAIL, kvh, h.b);
            }
          }
          if (s == 0) {
            const __nv_bfloat16* qsrc =
                a.q + (static_cast<size_t>(h.b) * a.Hq + kvh * g_total + hg * G) * D;
            bulk_load(smem_u32(qbuf + slot * C::QB), qsrc, q_bytes, full0 + 8 * slot);
          }
        }
      }
      if (*abort_flag) {
        // let every copy this CTA started land before shared memory is released
        const uint64_t drain_ns = a.timeout_ns > kDrainFloorNs ? a.timeout_ns : kDrainFloorNs;
        for (int s = max(0, st - NST); s < st; ++s)
          mbar_wait_polled(full0 + 8 * (s % NST), (s / NST) & 1, drain_ns, a.status,
                    kDevTimeoutDrain, nullptr);
      }
    }
  }
  __syncthreads();
  // ---- count this CTA's split pieces; the CTA that finishes a unit's last
  // piece merges the unit (every partial of it is visible by then)
  const int np = min(*n_pending, 2);
  if (np == 0 || *abort_flag) return;
  volatile int* merge_mask = n_pending + 1;
  if (tid == 0) {
    // release: the partials of this CTA, written before the barrier, before
    // the count; acquire: the other pieces' partials after it (for the merge)
    const unsigned c0 = atom_add_acq_rel_gpu(a.counters + pending[0].unit, 1u);
    const unsigned c1 = np > 1 ? atom_add_acq_rel_gpu(a.counters + pending[1].unit, 1u) : 0u;
    int mm = c0 == static_cast<unsigned>(pending[0].nsp - 1) ? 1 : 0;
    if (np > 1 && c1 == static_cast<unsigned>(pending[1].nsp - 1)) mm |= 2;
    *merge_mask = mm;
  }
  __syncthreads();
  const int mm = *merge_mask;
  // the G rows of each unit to merge, one warp per row
  const int n0 = (mm & 1) ? G : 0;
  const int nrows = n0 + ((mm & 2) ? G : 0);
  for (int t = warp; t < nrows; t += kDecWarps + 1) {
    const Pending p = pending[t < n0 ? 0 : 1];
    const int h = t < n0 ? t : t - n0;
    const int kvh = p.kh / a.head_groups;
    const int hg = p.kh % a.head_groups;
    const size_t bh0 = static_cast<size_t>(p.b) * a.Hq + kvh * g_total + hg * G;
    merge_row<D>(a, bh0 + h, p.nsp, lane);
  }
}

// ---------------------------------------------------------------------------
// Forced split counts (num_splits > 0: the FlashDecoding tutorial's fixed
// number of KV chunks per sequence, §三 3.2). The work space is cut into
// chunks of Rc rows (the last one shorter); CTA c takes a contiguous run of
// ceil(chunks / gridDim.x) of them and hands them to its consumer warps in
// turn: warp w takes the run's chunks w, w + 7, w + 14, ... A run covers
// whole groups of a unit's pieces, so the CTA that completes a group is
// mostly the one that streamed it, and a slow SM delays few groups. Every stage carries one
// slice (one tail box of RPWS rows) per warp, from that warp's current chunk,
// so that each warp walks its own chunks slice by slice. A piece is a chunk's
// rows within one unit; the warp ends each of its pieces by itself: it sums
// its row groups, writes the piece's normalised partial o and log-sum-exp (or
// the output, when the piece is the whole unit) and counts the piece in the
// unit's counter; the warp that completes a unit's count merges the unit.
// No piece end waits for the other warps, so pieces of a few stages stay
// cheap.
// A group of the pieces of one unit, complete and to be merged.
struct GroupTask {
  int unit, nsp, b, kh, g;
};
// pieces of a unit merged together before the groups are
constexpr int kMergeGroup = kDecodeMergeGroup;

struct WarpSlice {
  int b, kh;   // batch and unit (KV head x head group) of the slice
  int row;     // first key row of the slice within the unit
  int rows;    // rows of the slice in the piece (0: the warp has nothing in this stage)
  int vend;    // rows of the slice that hold keys (fewer only past a paged length)
  int slot;    // the piece's partial slot within the unit
  int nsp;     // pieces of the unit
  int flags;   // kSliceFirst | kSliceLast
};
constexpr int kSliceFirst = 1, kSliceLast = 2;

template <int D, int G>
struct SplitCfg {
  using C = DecCfg<D, G>;
  static constexpr int SLICE = C::RPWS;  // rows of a warp's slice
  static_assert(SLICE == C::TAIL, "a slice is one tail box");
  // ring | q of each (slot, warp) | slices [slot][warp] | barriers, flags
  static constexpr int QW_OFF = kRingBytes;
  static constexpr int SL_OFF = QW_OFF + C::NST * kDecWarps * C::QB;
  static constexpr int BAR_OFF = SL_OFF + C::NST * kDecWarps * static_cast<int>(sizeof(WarpSlice));
  // groups of pieces whose count this CTA completed, merged after its stream
  static constexpr int DEF_OFF = BAR_OFF + 256;
  static constexpr int MAX_DEFERRED = 512;
  static constexpr int SMEM = DEF_OFF + MAX_DEFERRED * static_cast<int>(sizeof(GroupTask)) + 1024;
  static_assert(SMEM <= 232448, "shared memory");
};

// Merge partials [k0, k1) of one (batch, query head) row (normalised o of D
// floats each at o_row, log2 lse at lse_row) into a running state (M, W,
// acc), as merge_row does: all lse and o loads of up to 8 partials in flight
// before any is used, the largest lse factored out.
template <int D>
__device__ __forceinline__ void merge_range(const float* lse_row, const float* o_row, int k0,
                                            int k1, int lane, float& M, float& W,
                                            float (&acc)[D / 32]) {
  constexpr int EPL = D / 32;
  const float* pl = lse_row;
  const float* po = o_row + lane * EPL;
  for (int kb = k0; kb < k1; kb += 8) {
    float lk[8], v[8][EPL];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = kb + u < k1;
      lk[u] = in ? __ldcg(pl + kb + u) : -INFINITY;
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const float2 t = in ? __ldcg(reinterpret_cast<const float2*>(po + static_cast<size_t>(kb + u) * D + e))
                            : make_float2(0.f, 0.f);
        v[u][e] = t.x;
        v[u][e + 1] = t.y;
      }
    }
    float mb = M;
#pragma unroll
    for (int u = 0; u < 8; ++u) mb = fmaxf(mb, lk[u]);
    if (mb == -INFINITY) continue;  // only empty pieces so far
    const float sc = ex2(M - mb);
    W *= sc;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= sc;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float wk = ex2(lk[u] - mb);
      W += wk;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wk, v[u][e], acc[e]);
    }
    M = mb;
  }
}

// merge_range for at most 32 partials, in one or two rounds of loads: lane k
// loads partial k's lse while every lane loads its part of a whole batch of
// o rows; the largest lse and the weights then come by shuffles, and the
// batch is summed without a rescale chain. Same result as merge_range up to
// the order of the additions within the batch (fixed, so still deterministic).
template <int D>
__device__ __forceinline__ void merge_few(const float* lse_row, const float* o_row, int k0, int k1,
                                          int lane, float& M, float& W, float (&acc)[D / 32]) {
  constexpr int EPL = D / 32;
  constexpr int BK = 128 / EPL < 32 ? 128 / EPL : 32;  // pieces per batch of loads
  const int n = k1 - k0;  // <= 32
  const float* po = o_row + static_cast<size_t>(k0) * D + lane * EPL;
  const float lk = lane < n ? __ldcg(lse_row + k0 + lane) : -INFINITY;
  float v[BK][EPL];
#pragma unroll
  for (int u = 0; u < BK; ++u)
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
      const float2 t = u < n ? __ldcg(reinterpret_cast<const float2*>(po + static_cast<size_t>(u) * D + e))
                             : make_float2(0.f, 0.f);
      v[u][e] = t.x;
      v[u][e + 1] = t.y;
    }
  float mx = lk;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  M = mx;
  W = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  if (mx == -INFINITY) return;  // only empty pieces
  const float wk = ex2(lk - mx);  // 0 for an empty or absent piece
  float ws = wk;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
  W = ws;
#pragma unroll
  for (int u = 0; u < BK; ++u) {
    const float w = __shfl_sync(0xffffffffu, wk, u);
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
  }
#pragma unroll 1
  for (int kb = BK; kb < n; kb += BK) {  // D = 256: a second batch
#pragma unroll
    for (int u = 0; u < BK; ++u)
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const float2 t = kb + u < n
                             ? __ldcg(reinterpret_cast<const float2*>(po + static_cast<size_t>(kb + u) * D + e))
                             : make_float2(0.f, 0.f);
        v[u][e] = t.x;
        v[u][e + 1] = t.y;
      }
#pragma unroll
    for (int u = 0; u < BK; ++u) {
      const float w = __shfl_sync(0xffffffffu, wk, (kb + u) & 31);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
    }
  }
}

// Write a merged row: out = acc / W (bf16), lse = M + log2 W (natural log);
// no valid key at all: out 0, lse +inf.
template <int D>
__device__ __forceinline__ void write_merged(const DecodeArgs& a, size_t row, int lane, float M,
                                             float W, const float (&acc)[D / 32]) {
  constexpr int EPL = D / 32;
  const bool invalid = (M == -INFINITY);
  const float inv = invalid ? 0.f : 1.f / W;
  __nv_bfloat16* dst = a.out + row * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; e += 2)
    *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0 && a.lse != nullptr) a.lse[row] = invalid ? INFINITY : (M + log2f(W)) * kLn2;
}

// One warp finishes a complete group of pieces: for each of the G rows it
// merges the group's pieces in slot order into the group partial (or, when
// the unit has one group, into the output); then it counts the group, and
// the warp that completes the unit's groups merges them, in order, into the
// output. Nothing waits for another warp or CTA.
// kBatched: merge with merge_few (after the stream, when nothing else is
// live); the rare call from inside the streaming loop (a full list) uses
// merge_range, whose few registers keep the loop free of spills.
template <int D, int G, bool kBatched>
__device__ __forceinline__ void finish_group(const DecodeArgs& a, const GroupTask& t, int lane) {
  constexpr int EPL = D / 32;
  const int g_total = a.Hq / a.Hkv;
  const size_t bh0 = static_cast<size_t>(t.b) * a.Hq + (t.kh / a.head_groups) * g_total +
                     (t.kh % a.head_groups) * G;
  const int ng = (t.nsp + kMergeGroup - 1) / kMergeGroup;
  const int k0 = t.g * kMergeGroup, k1 = min(k0 + kMergeGroup, t.nsp);
#pragma unroll 1
  for (int h = 0; h < G; ++h) {
    const size_t row = bh0 + h;
    float M = -INFINITY, W = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    if constexpr (kBatched)
      merge_few<D>(a.part_lse + row * a.max_slots, a.part_o + row * a.max_slots * D, k0, k1,
                   lane, M, W, acc);
    else
      merge_range<D>(a.part_lse + row * a.max_slots, a.part_o + row * a.max_slots * D, k0, k1,
                     lane, M, W, acc);
    if (ng == 1) {
      write_merged<D>(a, row, lane, M, W, acc);
    } else {
      const bool empty = (M == -INFINITY);
      const float inv = empty ? 0.f : 1.f / W;
      float* dst = a.grp_o + (row * a.max_groups + t.g) * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; e += 2)
        *reinterpret_cast<float2*>(dst + e) = make_float2(acc[e] * inv, acc[e + 1] * inv);
      if (lane == 0) a.grp_lse[row * a.max_groups + t.g] = empty ? -INFINITY : M + log2f(W);
    }
  }
  if (ng == 1) return;
  __threadfence();  // this lane's group partials, before the count
  __syncwarp();
  unsigned c = 0;
  if (lane == 0) c = atomicAdd(a.counters + t.unit, 1u);
  c = __shfl_sync(0xffffffffu, c, 0);
  if (c != static_cast<unsigned>(ng - 1)) return;
  __threadfence();  // the other groups' partials, before they are read
#pragma unroll 1
  for (int h = 0; h < G; ++h) {
    const size_t row = bh0 + h;
    float M = -INFINITY, W = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    if (kBatched && ng <= 32)
      merge_few<D>(a.grp_lse + row * a.max_groups, a.grp_o + row * a.max_groups * D, 0, ng, lane,
                   M, W, acc);
    else
      merge_range<D>(a.grp_lse + row * a.max_groups, a.grp_o + row * a.max_groups * D, 0, ng,
                     lane, M, W, acc);
    write_merged<D>(a, row, lane, M, W, acc);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, 1)
    split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_k16,
                 const __grid_constant__ CUtensorMap tm_v16,
                 const __grid_constant__ DecodeArgs a) {
  using C = DecCfg<D, G>;
  using SC = SplitCfg<D, G>;
  constexpr int NP = C::NP;
  constexpr int NST = C::NST;
  constexpr int SLICE = SC::SLICE;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* qw = smem + SC::QW_OFF;  // [NST][warps][QB]
  WarpSlice* slices = reinterpret_cast<WarpSlice*>(smem + SC::SL_OFF);  // [NST][warps]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SC::BAR_OFF);     // full[NST], empty[NST]
  volatile int* done = reinterpret_cast<volatile int*>(bars + 2 * kMaxStages);  // [NST]: no more work
  volatile int* abort_flag = done + kMaxStages;
  int* n_deferred = const_cast<int*>(abort_flag) + 1;
  GroupTask* deferred = reinterpret_cast<GroupTask*>(smem + SC::DEF_OFF);  // [MAX_DEFERRED]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long KH = static_cast<long long>(a.Hkv) * a.head_groups;
  const int g_total = a.Hq / a.Hkv;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kMaxStages);
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kDecWarps);
    }
    *abort_flag = 0;
    *n_deferred = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDecWarps) {
    // ================================================================ producer
    // lane w < 7 plans the slices of consumer warp w; lane 0 completes the
    // stage's barrier bookkeeping
    const long long Rc = a.rows_per_cta;  // chunk rows
    const long long n_chunks = (a.total + Rc - 1) / Rc;
    // this CTA's chunks: a contiguous run, so that the groups of pieces it
    // completes (and merges) are mostly its own
    const long long per_cta = (n_chunks + gridDim.x - 1) / gridDim.x;
    const long long c_end = min(n_chunks, (static_cast<long long>(blockIdx.x) + 1) * per_cta);
    long long v = static_cast<long long>(blockIdx.x) * per_cta + lane;
    bool have = lane < kDecWarps && v < c_end;
    long long r = have ? v * Rc : 0;
    long long r_end = have ? min(r + Rc, a.total) : 0;
    long long u0 = 0, u1 = 0;  // the unit holding row r (rows of the work space)
    int ub = 0, ukh = 0;
    if (lane == 0) {
      tma_prefetch_map(&tm_k16);
      tma_prefetch_map(&tm_v16);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int st = 0;
    bool ok = true;
    for (;; ++st) {
      const int slot = st % NST;
      const int use = st / NST;
      if (use > 0) {
        ok = mbar_wait_polled(empty0 + 8 * slot, (use - 1) & 1, a.timeout_ns, a.status,
                              kDevTimeoutDecodeEmpty, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      // this warp's next slice
      if (have && r >= r_end) {
        v += kDecWarps;  // the warp's next chunk
        have = v < c_end;
        if (have) {
          r = v * Rc;
          r_end = min(r + Rc, a.total);
        }
      }
      WarpSlice ws{0, 0, 0, 0, 0, 0, 0, 0};
      uint32_t bytes = 0;
      if (have) {
        if (r < u0 || r >= u1) {
          const int b = find_batch(a.prefix, a.B, KH, 0, r);
          const long long base = KH * a.prefix[b];
          const long long L = a.prefix[b + 1] - a.prefix[b];
          const long long kh = div_nn(r - base, L);
          u0 = base + kh * L;
          u1 = u0 + L;
          ub = b;
          ukh = static_cast<int>(kh);
        }
        const long long p0 = max(u0, v * Rc), p1 = min(u1, r_end);  // this piece
        const int rows = static_cast<int>(min(static_cast<long long>(SLICE), p1 - r));
        ws.b = ub;
        ws.kh = ukh;
        ws.row = static_cast<int>(r - u0);
        ws.rows = rows;
        ws.vend = rows;
        if (a.block_table != nullptr) {
          const long long real =
              a.real_len != nullptr ? __ldg(a.real_len + ub) : (u1 - u0) - a.pad16[ub];
          ws.vend = static_cast<int>(max(0ll, min(static_cast<long long>(rows), real - ws.row)));
        }
        ws.slot = static_cast<int>(v - div_nn(u0, Rc));
        ws.nsp = static_cast<int>(div_nn(u1 - 1, Rc) - div_nn(u0, Rc) + 1);
        ws.flags = (r == p0 ? kSliceFirst : 0) | (r + rows == p1 ? kSliceLast : 0);
        bytes = 2u * SLICE * D * 2 + ((ws.flags & kSliceFirst) ? G * D * 2 : 0);
        r += rows;
      }
      uint32_t total_bytes = bytes;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        total_bytes += __shfl_xor_sync(0xffffffffu, total_bytes, off);
      const bool any = __any_sync(0xffffffffu, have);
      if (lane < kDecWarps) slices[slot * kDecWarps + lane] = ws;
      __syncwarp();  // every lane's slice is written before lane 0 publishes the stage
      if (!any) {
        if (lane == 0) {
          done[slot] = 1;
          mbar_arrive(full0 + 8 * slot);  // end marker: no data
        }
        ++st;
        break;
      }
      if (lane == 0) {
        done[slot] = 0;
        mbar_expect_tx(full0 + 8 * slot, total_bytes);
      }
      __syncwarp();
      if (have) {
        const uint32_t dst = smem_u32(smem + slot * C::STAGE_BYTES) + lane * SLICE * D * 2;
        const int kvh = ws.kh / a.head_groups;
        const int hg = ws.kh % a.head_groups;
        if (a.block_table != nullptr) {
          // a slice never straddles a block: blocks are multiples of 16 rows and
          // slices start at multiples of SLICE rows of the (16-row rounded) unit
          const int32_t* bt = a.block_table + static_cast<size_t>(ws.b) * a.max_blocks;
          const int blk = __ldg(bt + ws.row / a.block_size);
          const int in_blk = ws.row % a.block_size;
          tma_load_4d(dst, &tm_k16, full0 + 8 * slot, 0, in_blk, kvh, blk);
          tma_load_4d(dst + C::TILE_BYTES, &tm_v16, full0 + 8 * slot, 0, in_blk, kvh, blk);
        } else {
          tma_load_4d(dst, &tm_k16, full0 + 8 * slot, 0, ws.row, kvh, ws.b);
          tma_load_4d(dst + C::TILE_BYTES, &tm_v16, full0 + 8 * slot, 0, ws.row, kvh, ws.b);
        }
        if (ws.flags & kSliceFirst) {
          const __nv_bfloat16* qsrc =
              a.q + (static_cast<size_t>(ws.b) * a.Hq + kvh * g_total + hg * G) * D;
          bulk_load(smem_u32(qw + (slot * kDecWarps + lane) * C::QB), qsrc, G * D * 2,
                    full0 + 8 * slot);
        }
      }
    }
    if (*abort_flag && lane == 0) {
      // let every copy this CTA started land before shared memory is released
      const uint64_t drain_ns = a.timeout_ns > kDrainFloorNs ? a.timeout_ns : kDrainFloorNs;
      for (int s = max(0, st - NST); s < st; ++s)
        mbar_wait_polled(full0 + 8 * (s % NST), (s / NST) & 1, drain_ns, a.status,
                         kDevTimeoutDrain, nullptr);
    }
    return;
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.has_empty) {
    // sequences of length 0: out = 0, lse = +inf; one thread per row
    for (int row = static_cast<int>(blockIdx.x) * kDecWarps * 32 + tid; row < a.B * a.Hq;
         row += static_cast<int>(gridDim.x) * kDecWarps * 32) {
      const int b = row / a.Hq;
      if (a.prefix[b + 1] != a.prefix[b]) continue;
      uint4* dst = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * D);
#pragma unroll
      for (int i = 0; i < D * 2 / 16; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      if (a.lse != nullptr) a.lse[row] = INFINITY;
    }
  }
  // ================================================================ consumers
  // The lane layout of decode_kernel: LPR lanes share a K/V row, each lane
  // holds q and o of all G heads in the order j -> head j ^ x (x = sub >>
  // SHIFT) and ends the butterfly with the score of head x.
  const int sub = lane % C::LPR;
  const int rg = lane / C::LPR;
  const int x = sub >> C::SHIFT;
  float m = -INFINITY, l = 0.f;  // head x of this row group
  uint64_t o[G][NP];
  uint64_t qp[G][NP];
  const uint8_t* mask_row = nullptr;
  size_t bh0 = 0;  // the piece's first (batch, query head) row
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int k = 0; k < NP; ++k) o[j][k] = 0ull;

  for (int st = 0;; ++st) {
    const int slot = st % NST;
    bool got = mbar_wait_polled(full0 + 8 * slot, (st / NST) & 1, a.timeout_ns, a.status,
                                kDevTimeoutDecodeFull, abort_flag);
    got = __all_sync(0xffffffffu, got);
    if (!got || done[slot]) break;
    const WarpSlice ws = slices[slot * kDecWarps + warp];
    if (ws.rows > 0) {
      if (ws.flags & kSliceFirst) {
        // ---- a new piece of this warp: q landed with this stage; fresh state
        const int kvh = ws.kh / a.head_groups;
        const int hg = ws.kh % a.head_groups;
        bh0 = static_cast<size_t>(ws.b) * a.Hq + kvh * g_total + hg * G;
        mask_row = nullptr;
        if (a.key_mask != nullptr)
          mask_row = a.key_mask + ws.b * a.mask_bstride +
                     (static_cast<long long>(kvh) * g_total + hg * G + x) * a.mask_hstride;
        const __nv_bfloat16* qs =
            reinterpret_cast<const __nv_bfloat16*>(qw + (slot * kDecWarps + warp) * C::QB);
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int j = 0; j < G; ++j) {
#pragma unroll
          for (int k = 0; k < NP; ++k) o[j][k] = 0ull;
#pragma unroll
          for (int ch = 0; ch < C::NCH; ++ch) {
            const uint4 u =
                *reinterpret_cast<const uint4*>(qs + (j ^ x) * D + (sub + C::LPR * ch) * 8);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              qp[j][ch * 4 + k] = pair_f32(bf16lo_to_f32(w4[k]) * a.scale_log2,
                                           bf16hi_to_f32(w4[k]) * a.scale_log2);
          }
        }
      }
      // ---- this warp's slice: SLICE rows of K and V at rows
      // [warp * SLICE, (warp + 1) * SLICE) of the stage
      const __nv_bfloat16* Ks = reinterpret_cast<const __nv_bfloat16*>(smem + slot * C::STAGE_BYTES);
      const __nv_bfloat16* Vs = Ks + C::R * D;
      const int stage_row0 = ws.row - warp * SLICE;  // key row of stage row 0
      const int row_end = ws.row + ws.vend;
      const bool dense = mask_row == nullptr && ws.vend == SLICE;
      float s[C::STEPS];
      bool valid[C::STEPS];  // some head of the row group sees the key
#pragma unroll
      for (int i = 0; i < C::STEPS; ++i) {
        const int rr = warp * SLICE + i * C::RPW + rg;
        const int gr = stage_row0 + rr;
        bool ok = true;
        if (!dense) {
          ok = gr < row_end;
          if (ok && mask_row != nullptr) ok = mask_row[gr] == 0;
          const uint32_t seen = __ballot_sync(0xffffffffu, ok) >> (rg * C::LPR);
          valid[i] = (seen & ((1u << C::LPR) - 1u)) != 0u;
        } else {
          valid[i] = true;
        }
        uint64_t kp[NP];
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          const uint4 u = *reinterpret_cast<const uint4*>(Ks + rr * D + (sub + C::LPR * ch) * 8);
          kp[ch * 4 + 0] = bf16x2_pair(u.x);
          kp[ch * 4 + 1] = bf16x2_pair(u.y);
          kp[ch * 4 + 2] = bf16x2_pair(u.z);
          kp[ch * 4 + 3] = bf16x2_pair(u.w);
        }
        float part[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
          uint64_t ac = ffma2(qp[j][0], kp[0], 0ull);
          if constexpr (G <= 2) {
            uint64_t ac2 = ffma2(qp[j][1], kp[1], 0ull);
#pragma unroll
            for (int k = 2; k < NP; k += 2) {
              ac = ffma2(qp[j][k], kp[k], ac);
              ac2 = ffma2(qp[j][k + 1], kp[k + 1], ac2);
            }
            ac = fadd2(ac, ac2);
          } else {
#pragma unroll
            for (int k = 1; k < NP; ++k) ac = ffma2(qp[j][k], kp[k], ac);
          }
          const float2 a2 = unpair(ac);
          part[j] = a2.x + a2.y;
        }
#pragma unroll
        for (int lv = 0; lv < C::LG; ++lv) {
          const int half = G >> (lv + 1);
#pragma unroll
          for (int j = 0; j < half; ++j)
            part[j] += __shfl_xor_sync(0xffffffffu, part[j + half], (C::LPR / 2) >> lv);
        }
#pragma unroll
        for (int lv = C::LG; lv < C::LOG_LPR; ++lv)
          part[0] += __shfl_xor_sync(0xffffffffu, part[0], (C::LPR / 2) >> lv);
        s[i] = ok ? part[0] : -INFINITY;
      }
      // online softmax of head x over this slice (running max shared by the row groups)
      float mx = s[0];
#pragma unroll
      for (int i = 1; i < C::STEPS; ++i) mx = fmaxf(mx, s[i]);
#pragma unroll
      for (int off = C::LPR; off < 32; off <<= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m, mx);
      const float m_use = (mn == -INFINITY) ? 0.f : mn;
      const float alpha = ex2(m - m_use);  // 0 when m was -inf
      m = mn;
      float ps = 0.f;
#pragma unroll
      for (int i = 0; i < C::STEPS; ++i) {
        s[i] = ex2(s[i] - m_use);  // -inf -> 0
        ps += s[i];
      }
      l = fmaf(l, alpha, ps);
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float aj = j == 0 ? alpha : __shfl_xor_sync(0xffffffffu, alpha, j << C::SHIFT);
          const uint64_t a2 = pair_f32(aj, aj);
#pragma unroll
          for (int k = 0; k < NP; ++k) o[j][k] = fmul2(o[j][k], a2);
        }
      }
#pragma unroll
      for (int i = 0; i < C::STEPS; ++i) {
        const int rr = warp * SLICE + i * C::RPW + rg;
        uint64_t vp[NP];
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          uint4 u = *reinterpret_cast<const uint4*>(Vs + rr * D + (sub + C::LPR * ch) * 8);
          if (!dense && !valid[i]) u = make_uint4(0u, 0u, 0u, 0u);  // never a stale row
          vp[ch * 4 + 0] = bf16x2_pair(u.x);
          vp[ch * 4 + 1] = bf16x2_pair(u.y);
          vp[ch * 4 + 2] = bf16x2_pair(u.z);
          vp[ch * 4 + 3] = bf16x2_pair(u.w);
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float pj = j == 0 ? s[i] : __shfl_xor_sync(0xffffffffu, s[i], j << C::SHIFT);
          const uint64_t p2 = pair_f32(pj, pj);
#pragma unroll
          for (int k = 0; k < NP; ++k) o[j][k] = ffma2(p2, vp[k], o[j][k]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    if (ws.rows == 0 || !(ws.flags & kSliceLast)) continue;

    // ================================================= end of this warp's piece
    // l of head x over the row groups (m is shared); the accumulators halved
    // across the row groups so that a lane keeps 1/RPW of them, summed
#pragma unroll
    for (int off = C::LPR; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    constexpr int F = G * NP;
    constexpr int FQ = F / C::RPW;
    const bool b0 = (rg & 1) != 0, b1 = (rg & 2) != 0;
    uint64_t h1[F / 2];
#pragma unroll
    for (int f = 0; f < F / 2; ++f) {
      const uint64_t lo = o[f / NP][f % NP], hi = o[(f + F / 2) / NP][(f + F / 2) % NP];
      const uint64_t keep = b0 ? hi : lo, send = b0 ? lo : hi;
      const float2 sp = unpair(send);
      const float rx = __shfl_xor_sync(0xffffffffu, sp.x, C::LPR);
      const float ry = __shfl_xor_sync(0xffffffffu, sp.y, C::LPR);
      h1[f] = fadd2(keep, pair_f32(rx, ry));
    }
    uint64_t hq[FQ];
    if constexpr (C::RPW == 4) {
#pragma unroll
      for (int f = 0; f < F / 4; ++f) {
        const uint64_t keep = b1 ? h1[f + F / 4] : h1[f], send = b1 ? h1[f] : h1[f + F / 4];
        const float2 sp = unpair(send);
        const float rx = __shfl_xor_sync(0xffffffffu, sp.x, 2 * C::LPR);
        const float ry = __shfl_xor_sync(0xffffffffu, sp.y, 2 * C::LPR);
        hq[f] = fadd2(keep, pair_f32(rx, ry));
      }
    } else {
#pragma unroll
      for (int f = 0; f < FQ; ++f) hq[f] = h1[f];
    }
    // write the piece: o / l of every head (l of head h from a lane whose
    // head x is h) and one lse per head
    const int base = (b0 ? F / 2 : 0) + (b1 ? F / 4 : 0);
#pragma unroll
    for (int f = 0; f < FQ; ++f) {
      const int fl = base + f;
      const int j = fl / NP, k = fl % NP;
      const int h = j ^ x;
      const float lh = __shfl_sync(0xffffffffu, l, h << C::SHIFT);
      const float inv = lh > 0.f ? 1.f / lh : 0.f;
      const int d = (sub + C::LPR * (k / 4)) * 8 + 2 * (k % 4);
      const float2 v2 = unpair(hq[f]);
      if (FA_CHECK(bh0 + h < static_cast<size_t>(a.B) * a.Hq, a.status, kDevCheckDecodeRow) &&
          FA_CHECK(ws.nsp == 1 || ws.slot < a.max_slots, a.status, kDevCheckDecodeSlot)) {
        if (ws.nsp == 1)
          *reinterpret_cast<uint32_t*>(a.out + (bh0 + h) * D + d) = pack_bf16x2(v2.x * inv, v2.y * inv);
        else
          *reinterpret_cast<float2*>(a.part_o + ((bh0 + h) * a.max_slots + ws.slot) * D + d) =
              make_float2(v2.x * inv, v2.y * inv);
      }
    }
    if (rg == 0 && (sub & ((1 << C::SHIFT) - 1)) == 0) {  // one lane per head x
      const bool empty = !(l > 0.f);
      if (ws.nsp == 1) {
        if (a.lse != nullptr) a.lse[bh0 + x] = empty ? INFINITY : (m + log2f(l)) * kLn2;
      } else {
        a.part_lse[(bh0 + x) * a.max_slots + ws.slot] = empty ? -INFINITY : m + log2f(l);
      }
    }
    if (ws.nsp > 1) {
      // count the piece in its group; the CTA that completes a group merges
      // it after its stream (at once when its list is full)
      __threadfence();  // this lane's partial, before the count
      __syncwarp();
      const int unit = static_cast<int>(ws.b * KH + ws.kh);
      const int g = ws.slot / kMergeGroup;
      const int gsize = min(kMergeGroup, ws.nsp - g * kMergeGroup);
      int slot_def = -2;  // -2: the group is not complete
      if (lane == 0) {
        const unsigned c =
            atomicAdd(a.grp_counters + static_cast<size_t>(unit) * a.max_groups + g, 1u);
        if (c == static_cast<unsigned>(gsize - 1)) {
          __threadfence();  // the other pieces' partials, before they are read
          slot_def = atomicAdd(n_deferred, 1);
          if (slot_def < SC::MAX_DEFERRED)
            deferred[slot_def] = GroupTask{unit, ws.nsp, ws.b, ws.kh, g};
          else
            slot_def = -1;
        }
      }
      slot_def = __shfl_sync(0xffffffffu, slot_def, 0);
      if (slot_def == -1)
        finish_group<D, G, false>(a, GroupTask{unit, ws.nsp, ws.b, ws.kh, g}, lane);
    }
  }

  // ---- the groups this CTA completed, one warp each
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
  if (*abort_flag) return;
  const int nd = min(*n_deferred, SC::MAX_DEFERRED);
#pragma unroll 1
  for (int t = warp; t < nd; t += kDecWarps) finish_group<D, G, true>(a, deferred[t], lane);
}

// When no sequence has a key stage 1 is not launched: every row gets out = 0
// and lse = +inf here (one warp per (batch, query head)).
template <int D>
__global__ void __launch_bounds__(128) decode_empty_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int EPL = D / 32;  // output elements per lane
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row >= a.B * a.Hq) return;
  __nv_bfloat16* dst = a.out + static_cast<size_t>(row) * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = 0u;
  if (lane == 0 && a.lse != nullptr) a.lse[row] = INFINITY;
}

template <int D, int G>
cudaError_t launch_decode_dg(int grid, bool loop, const CUtensorMap* m, const DecodeArgs& da,
                             cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};  // devices with the attributes set
  if (setup_needed(configured)) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G, kSharesRows>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DecCfg<D, G>::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_kernel<D, G, kSharesCost>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, DecCfg<D, G>::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(split_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SplitCfg<D, G>::SMEM);
    if (e != cudaSuccess) return e;
    setup_done(configured);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = DecCfg<D, G>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (loop) {
    cfg.dynamicSmemBytes = SplitCfg<D, G>::SMEM;
    return cudaLaunchKernelEx(&cfg, split_kernel<D, G>, m[0], m[1], m[2], m[3], da);
  }
  if (da.piece_cost != 0)
    return cudaLaunchKernelEx(&cfg, decode_kernel<D, G, kSharesCost>, m[0], m[1], m[2], m[3], da);
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, G, kSharesRows>, m[0], m[1], m[2], m[3], da);
}

template <int D>
cudaError_t launch_decode_d(int G, int grid, bool loop, const CUtensorMap* m,
                            const DecodeArgs& da, cudaStream_t s) {
  switch (G) {
    case 8:
      if constexpr (D == 64) return launch_decode_dg<D, 8>(grid, loop, m, da, s);
      return cudaErrorInvalidValue;
    case 4: return launch_decode_dg<D, 4>(grid, loop, m, da, s);
    case 2: return launch_decode_dg<D, 2>(grid, loop, m, da, s);
    default: return launch_decode_dg<D, 1>(grid, loop, m, da, s);
  }
}

}  // namespace

// Zeroes the first n words of a decode workspace (the status word and the
// piece counters) on the stream before the decode kernel. It lets that
// kernel start at once (programmatic dependent launch), so the kernel plans
// its first piece while this runs; the kernel reads the counters and the
// status word only after its griddepcontrol.wait, which waits for this
// kernel's writes. It is launched in stream order itself, after all earlier
// work (a decode kernel before it may still use the same counters).
__global__ void __launch_bounds__(256) clear_kernel(uint32_t* __restrict__ p, int n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = static_cast<int>(blockIdx.x) * 256 + static_cast<int>(threadIdx.x); i < n;
       i += static_cast<int>(gridDim.x) * 256)
    p[i] = 0u;
}

cudaError_t launch_clear(void* workspace, size_t bytes, cudaStream_t stream) {
  const int n = static_cast<int>(bytes / sizeof(uint32_t));
  const int grid = std::max(1, std::min((n + 255) / 256, 128));
  clear_kernel<<<grid, 256, 0, stream>>>(static_cast<uint32_t*>(workspace), n);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeLaunch& x, cudaStream_t stream) {
  const int g_total = x.Hq / x.Hkv;
  const int G = decode_heads_per_cta(g_total, x.D);
  DecodeArgs da;
  da.q = static_cast<const __nv_bfloat16*>(x.q);
  da.key_mask = x.key_mask;
  da.part_o = x.part_o;
  da.part_lse = x.part_lse;
  da.out = static_cast<__nv_bfloat16*>(x.out);
  da.lse = x.lse;
  da.status = x.status;
  da.timeout_ns = x.timeout_ns;
  da.total = x.total;
  da.rows_per_cta = x.rows_per_cta;
  da.piece_cost = static_cast<int>(x.piece_cost);
  da.B = x.B;
  da.Hq = x.Hq;
  da.Hkv = x.Hkv;
  da.S_kv = std::max(x.S_kv, 1);
  da.max_slots = x.max_slots;
  da.head_groups = g_total / G;
  da.G = G;
  da.scale_log2 = x.scale * 1.4426950408889634f;
  da.prefix.global = x.prefix_dev;
  if (x.prefix_dev == nullptr)
    for (int b = 0; b <= x.B; ++b) da.prefix.local[b] = x.prefix_host[b];
  da.block_table = x.block_table;
  da.max_blocks = x.max_blocks;
  da.block_size = x.block_size;
  da.real_len = x.lens_dev;
  if (x.block_table != nullptr && x.lens_dev == nullptr)
    for (int b = 0; b < x.B; ++b)
      da.pad16[b] = static_cast<unsigned char>(x.prefix_host[b + 1] - x.prefix_host[b] -
                                               x.lens_host[b]);
  da.counters = x.counters;
  da.has_empty = x.has_empty ? 1 : 0;
  // shares cut by cost: their first rows, as the kernel's search would find
  // them (the row whose cost is the first at or above c * Rc), in the unused
  // end of the parameters' prefix array when it has room; this spares every
  // CTA two searches of the prefix sums before its first copy
  da.share_off = -1;
  const long long n_share = x.n_ctas + 1;
  const long long off = x.prefix_dev == nullptr ? x.B + 1 : 0;
  if (x.piece_cost != 0 && !x.loop_shares && x.total > 0 &&
      off + n_share <= kDecodeParamBatches + 1) {
    const long long KH = static_cast<long long>(x.Hkv) * (g_total / G);
    const long long pc = x.piece_cost;
    const long long* pre = x.prefix_host;
    auto row_at_cost = [&](long long T) -> long long {
      int b = 0;  // the last batch whose first row costs at most T
      for (int i = 1; i < x.B; ++i)
        if (KH * (pre[i] + pc * i) <= T) b = i;
      const long long L = pre[b + 1] - pre[b];
      const long long cb = KH * (pre[b] + pc * b);
      const long long kh = std::min(KH - 1, (T - cb) / (L + pc));
      const long long o = T - cb - kh * (L + pc);
      const long long u0 = KH * pre[b] + kh * L;
      return o < L ? u0 + o : u0 + L;
    };
    for (long long c = 0; c < n_share; ++c)
      da.prefix.local[off + c] = c == 0             ? 0
                                 : c == n_share - 1 ? x.total
                                                    : std::min(row_at_cost(c * x.rows_per_cta), x.total);
    da.share_off = static_cast<int>(off);
  }
  da.mask_bstride = x.mask_bstride;
  da.mask_hstride = x.mask_hstride;
  da.grp_o = x.grp_o;
  da.grp_lse = x.grp_lse;
  da.grp_counters = x.grp_counters;
  da.max_groups = x.max_groups;

  if (x.total > 0) {
    // K, V with stage-high boxes (112 rows, 56 for D = 256); K, V with the
    // boxes of a partial stage (16 rows, 8 for D = 256)
    CUtensorMap maps[4];
    const int stage_rows = x.D == 256 ? 56 : kDecodeStageRows;
    const int tail_rows = x.D == 256 ? 8 : 16;
    // a paged cache is a batch of num_blocks sequences of block_size rows
    const int nbat = x.block_table != nullptr ? x.num_blocks : x.B;
    const int S_map = x.block_table != nullptr ? x.block_size : std::max(x.S_kv, 1);
    // (the stage-high maps are not used for a paged cache, whose blocks may be shorter)
    const int box_rows = x.block_table != nullptr ? tail_rows : stage_rows;
    if (!encode_bf16_map(&maps[0], x.k, x.layout, nbat, x.Hkv, S_map, x.D, x.D, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_bf16_map(&maps[1], x.v, x.layout, nbat, x.Hkv, S_map, x.D, x.D, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_bf16_map(&maps[2], x.k, x.layout, nbat, x.Hkv, S_map, x.D, x.D, tail_rows,
                         CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_bf16_map(&maps[3], x.v, x.layout, nbat, x.Hkv, S_map, x.D, x.D, tail_rows,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    const int grid = static_cast<int>(x.n_ctas);
    main_kernel_begin(stream);
    const bool loop = x.loop_shares;
    const cudaError_t e = x.D == 256   ? launch_decode_d<256>(G, grid, loop, maps, da, stream)
                          : x.D == 128 ? launch_decode_d<128>(G, grid, loop, maps, da, stream)
                                       : launch_decode_d<64>(G, grid, loop, maps, da, stream);
    main_kernel_end(stream);
    if (e != cudaSuccess) return e;
    count_launches(1);
  }
  if (x.total > 0 || x.B == 0) return cudaSuccess;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((x.B * x.Hq + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = x.D == 256   ? cudaLaunchKernelEx(&cfg, decode_empty_kernel<256>, da)
                        : x.D == 128 ? cudaLaunchKernelEx(&cfg, decode_empty_kernel<128>, da)
                                     : cudaLaunchKernelEx(&cfg, decode_empty_kernel<64>, da);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace fa
