// Fused attention forward (prefill) for sm_103a on the 5th-generation
// tensor cores.
//
// One CTA owns 256 consecutive query rows of one (batch, head) as two
// 128-row tiles Q0, Q1 and walks the KV sequence in 128-key tiles
// (FlashAttn guide, developer guide §3: tile the Q_S x KV_S matrix; never
// store it). Per KV tile j and Q tile t:
//     S_t   = Q_t K_j^T                          (tcgen05.mma, fp32 in TMEM)
//     m'    = max(m, rowmax(scale*S_t)), P = 2^(scale*log2e*S_t - m')
//     l     = l*2^(m-m') + rowsum(P),  O_t = O_t*2^(m-m') + P V_j  (tcgen05.mma)
// and finally out = O_t / l, lse = ln2*(m + log2 l)  (aclnnIncreFlashAttention
// guide §8.1: per-tile max/exp/sum refresh, division by the sum moved to
// the end; FlashAttn guide §1.6 LSE and §1.7 invalid rows).
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  softmax of Q0 (thread i <-> query row i <-> TMEM lane i)
//   warps 4-7  softmax of Q1
//   warp 8     TMA producer: Q0/Q1 once, then K_j, V_j through a 5-slot ring
//   warp 9     TMEM allocator and MMA issue stream of Q0 (one lane)
//   warp 10    MMA issue stream of Q1 (the two streams take turns)
//   warp 11    idle (it completes the third warpgroup for setmaxnreg)
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D).
// D = 256 (FlashAttn guide §3's largest head dim): one 128-row Q tile per
// work item (O0 takes [256,512)), 64-key KV tiles, warps 4-7 and the Q1
// issue stream idle.
// P_t (bf16, two per column) overwrites the first 64 columns of S_t and is
// the A operand of O_t += P_t V_j straight from TMEM.
// The MMA warp interleaves the two tiles (S0 S1 | PV0 S0' | PV1 S1' | ...)
// so that one tile's softmax runs while the tensor core works on the other.
//
// Causal (FlashAttn guide §1.5, mode 3): KV tiles above the diagonal are
// never loaded or multiplied; only the diagonal tile and tiles that hold
// masked or out-of-range keys pay for per-element predicates. Keys excluded
// by the key mask or the actual length have their V rows zeroed in shared
// memory before the P*V product, so whatever they hold cannot leak.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <numeric>
#include <type_traits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;        // query rows per Q tile
constexpr int kBitsTile = 128;  // keys per entry of the key-validity table
constexpr int kRing = 5;        // K/V ring slots (tiles of K or V)
constexpr int kThreads = 384;   // three warpgroups
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;     // MMA issue for Q0 (warp 10 for Q1); warp 11 idle
// Register split (setmaxnreg): the launch gives 168 per thread (384 x 168 =
// 64512), shared out between the two softmax warpgroups and the load/MMA
// warpgroup (PCfg::kSoftmaxRegs, kControlRegs).
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows by > 2^8

// D = 64, 128: two Q tiles per work item and 128-key KV tiles. D = 256: one
// Q tile (its O accumulator takes 256 TMEM columns) and 64-key KV tiles, so
// that the Q tile and five K/V tiles fit in shared memory.
template <int D>
struct PCfg {
  static constexpr int QT = D == 256 ? 1 : 2;           // Q tiles per work item
  static constexpr int BN = D == 256 ? 64 : 128;        // keys per KV tile
  static constexpr int NQ4 = BN / 32;                   // 32-key groups of a KV tile
  static constexpr int kQTileBytes = kBM * D * 2;       // one Q tile
  static constexpr int kKvTileBytes = BN * D * 2;       // one K or V tile
  static constexpr int kQSub = kBM * 128;               // a Q tile's 64-column swizzle slab
  static constexpr int kKvSub = BN * 128;               // a K/V tile's 64-column slab
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = QT * kQTileBytes;
  static constexpr int kBarOff = kRingOff + kRing * kKvTileBytes;
  // barriers + alignment slack; at least 116 KB so that two CTAs never share
  // an SM (each allocates all 512 TMEM columns)
  static constexpr int kSmemBytes = (kBarOff + 256 + 1024) > 118784 ? (kBarOff + 256 + 1024) : 118784;
  static_assert(kSmemBytes <= 232448, "shared memory");
  // register split (setmaxnreg) of the softmax and load/MMA warpgroups; the
  // D = 256 issue stream keeps 16 more registers:
  // 128 x (216 + 216 + 72) = 128 x (208 + 208 + 88) = 64512
  static constexpr int kSoftmaxRegs = D == 256 ? 208 : 216;
  static constexpr int kControlRegs = D == 256 ? 88 : 72;
  static_assert(2 * kSoftmaxRegs + kControlRegs == 504, "register split");
};

struct PrefillArgs {
  __nv_bfloat16* out;
  float* lse;
  const uint32_t* tile_bits;  // [B][n_kv_tiles][4], bit set = key valid; or null
  const int32_t* sched;       // offsets[grid + 1], then each CTA's work items in order
  // packed variable-length sequences (TND): q offset, q length, kv offset, kv
  // length per sequence ([4][B]); null for the padded layouts
  const int32_t* varlen;
  uint32_t* status;
  uint64_t timeout_ns;
  int B, Hq, Hkv, S_q, S_kv;
  int win_left, win_right;    // key j is seen by query i iff i - wl <= j <= i + wr; -1 = no limit
  int n_qpairs, n_kv_tiles, n_items;  // work items per (batch, head), KV tiles, all items
  long long out_row_stride, out_head_stride, out_batch_stride;  // elements
  float scale_log2;
#ifdef FA_DEBUG
  long long T_q;  // packed query rows (index checks only)
#endif
};

// Paged K/V (prefill_kernel<D, Pages>): k and v are pools of blocks of
// block_size rows; row r of batch b lives in block
// block_table[b * max_blocks + r / block_size] at row r % block_size; a KV
// tile is loaded as boxes of box_rows rows (a divisor of block_size), each
// inside one block. A kernel parameter of its own (an empty one for a
// contiguous cache), so that the contiguous instantiations' parameters and
// code stay as they are.
struct Pages {
  const int32_t* block_table;
  int max_blocks, block_size, box_rows;
};
struct NoPages {};

// Barrier slots (8 bytes each) after the tiles.
enum : int {
  kBarQ = 0,                        // Q tiles of the current work item landed
  kBarQFree = 1,                    // both streams' S products of the item done
  kBarKvFull = 2,                   // + slot
  kBarKvEmpty = kBarKvFull + kRing,
  kBarSFull = kBarKvEmpty + kRing,  // + tile
  kBarPReady = kBarSFull + 2,       // + tile
  kBarOFinal = kBarPReady + 2,      // + tile
  kBarODrained = kBarOFinal + 2,    // + tile: the epilogue has read O_t
  kBarFix = kBarODrained + 2,
  kBarDrain = kBarFix + 1,          // + issue stream
  kNumBars = kBarDrain + 2
};

// KV tiles of BN keys; with BN = 64 a tile is half an entry of the 128-key
// validity table.
template <int BN>
struct TileSeq {
  static constexpr bool half = BN == 64;
  const uint32_t* bits;  // this batch's rows of the tile table, or null
  int begin;             // first KV tile any Q tile of the item needs
  int end;               // one past the last KV tile any Q tile of the item needs
  // validity words of KV tile j (4 for 128 keys, the first 2 used for 64)
  __device__ __forceinline__ uint4 words(int j) const {
    if constexpr (!half) return __ldg(reinterpret_cast<const uint4*>(bits) + j);
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(bits) + j);
    return make_uint4(w.x, w.y, 0u, 0u);
  }
  __device__ __forceinline__ int next(int j) const {
    for (j = max(j, begin); j < end; ++j) {
      if (bits == nullptr) return j;
      const uint4 w = words(j);
      if ((w.x | w.y | w.z | w.w) != 0u) return j;
    }
    return end;
  }
  __device__ __forceinline__ bool full(int j) const {
    if (bits == nullptr) return true;
    const uint4 w = words(j);
    return half ? (w.x & w.y) == 0xFFFFFFFFu : (w.x & w.y & w.z & w.w) == 0xFFFFFFFFu;
  }
};

// One work item: 256 consecutive query rows (two 128-row tiles; 128 rows,
// one tile, for D = 256) of one (batch, query head). Items are numbered KV-head-major: all query pairs of
// the g query heads of one (batch, KV head) are consecutive, heaviest (last)
// pairs first and heads innermost, so the items in flight at any time read
// the same K/V tiles out of L2.
template <int D>
struct WorkItem {
  int b, kvh, h, q_row0;
  int S_q, S_kv, n_kv;   // this sequence's query rows, keys and KV tiles
  int q_base, kv_base;   // its first row in the q and k/v tensors (packed layout)
  int tma_b;             // batch coordinate of its tiles (0 when packed)
  bool has_t1;
  int lo_t[2], n_t[2];  // KV tiles [lo_t, n_t) each Q tile needs
  TileSeq<PCfg<D>::BN> seq;
};

template <int D>
__device__ __forceinline__ WorkItem<D> work_item(const PrefillArgs& a, int w) {
  using C = PCfg<D>;
  constexpr int kBN = C::BN;
  WorkItem<D> it;
  const int g = a.Hq / a.Hkv;
  const int per_kv = a.n_qpairs * g;
  const int bkv = w / per_kv;
  const int rem = w % per_kv;
  const int qp = a.n_qpairs - 1 - rem / g;
  it.b = bkv / a.Hkv;
  it.kvh = bkv % a.Hkv;
  it.h = it.kvh * g + rem % g;
  it.q_row0 = qp * C::QT * kBM;
  if (a.varlen != nullptr) {
    it.q_base = __ldg(a.varlen + it.b);
    it.S_q = __ldg(a.varlen + a.B + it.b);
    it.kv_base = __ldg(a.varlen + 2 * a.B + it.b);
    it.S_kv = __ldg(a.varlen + 3 * a.B + it.b);
    it.n_kv = (it.S_kv + kBN - 1) / kBN;
    it.tma_b = 0;
  } else {
    it.q_base = 0;
    it.S_q = a.S_q;
    it.kv_base = 0;
    it.S_kv = a.S_kv;
    it.n_kv = a.n_kv_tiles;
    it.tma_b = it.b;
  }
  it.has_t1 = C::QT == 2 && it.q_row0 + kBM < it.S_q;
  for (int t = 0; t < 2; ++t) {
    // rows r0 .. r0+127 see keys r0 - wl .. r0 + 127 + wr (window, causal = (-1, 0))
    const int r0 = it.q_row0 + t * kBM;
    int lo = 0, n = it.n_kv;
    if (a.win_left >= 0) lo = max(0, r0 - a.win_left) / kBN;
    if (a.win_right >= 0) n = min(n, (r0 + kBM - 1 + a.win_right) / kBN + 1);
    if (t == 1 && !it.has_t1) n = 0;
    it.lo_t[t] = min(lo, n);
    it.n_t[t] = n;
  }
  // the validity table has one entry per 128 keys of the padded sequence
  // (no table for packed sequences)
  constexpr int kPerEntry = kBitsTile / kBN;
  it.seq.bits = a.tile_bits ? a.tile_bits + static_cast<size_t>(it.b) *
                                                ((a.n_kv_tiles + kPerEntry - 1) / kPerEntry) * 4
                            : nullptr;
  // the union of the two ranges (contiguous: the second tile's range is the
  // first one shifted by one tile)
  it.seq.begin = it.n_t[1] > it.lo_t[1] ? min(it.lo_t[0], it.lo_t[1]) : it.lo_t[0];
  it.seq.end = max(it.n_t[0], it.n_t[1]);
  return it;
}

template <int D, class PG = NoPages>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a, const PG pgs) {
  constexpr bool kPaged = std::is_same_v<PG, Pages>;
  using C = PCfg<D>;
  constexpr int kBN = C::BN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* turn = reinterpret_cast<volatile int*>(tmem_slot + 2);  // MMA issue turn
  auto bar = [&](int i) -> uint32_t { return smem_u32(bars + i); };

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- persistent schedule: this CTA's list of work items, built on the
  // host (longest first, per group of 8 (batch, KV head) units, to the least
  // loaded CTA); n_items past the end of the list
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  const int list0 = __ldg(a.sched + cta);
  const int list_n = __ldg(a.sched + cta + 1) - list0;
  auto item_of = [&](int r) -> int {
    return r < list_n ? __ldg(a.sched + G + 1 + list0 + r) : a.n_items;
  };

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kBarPReady || i == kBarPReady + 1) cnt = kBM;
      if (i == kBarODrained || i == kBarODrained + 1) cnt = kBM;
      if (i >= kBarKvEmpty && i < kBarKvEmpty + kRing) cnt = 2;  // both issue streams
      if (i == kBarQFree) cnt = 2;                                // both issue streams
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    *turn = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kControlRegs));
  if (warp == kProducerWarp) {
    // ================================================================ TMA
    // Every lane waits on the same barriers and the warp votes on the result,
    // so the warp always takes one path (also when a wait gives up).
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
    }
    // paged K/V: KV tile j of batch b, box by box (every box inside one
    // block; the rows of a box past the table's last block, which lie past
    // every key, come from that last block and are masked)
    auto load_paged_tile = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar_addr, int b,
                               int j, int kvh) {
      if constexpr (kPaged) {
        const int32_t* bt = pgs.block_table + static_cast<size_t>(b) * pgs.max_blocks;
        for (int r = 0; r < kBN; r += pgs.box_rows) {
          const int row = j * kBN + r;
          const int blk = __ldg(bt + min(row / pgs.block_size, pgs.max_blocks - 1));
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(dst + s * C::kKvSub + r * 128, map, bar_addr, s * 64,
                        row % pgs.block_size, kvh, blk);
        }
      }
    };
    int item = 0;  // ring items issued so far (K_j and V_j are one item each)
    int fixes = 0;
    int q_loads = 0;  // work items whose Q tiles were requested
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int w = item_of(r);
      if (w >= a.n_items) break;
      const WorkItem<D> wi = work_item<D>(a, w);
      const int kvh = wi.kvh;
      const auto& seq = wi.seq;
      if (!FA_CHECK(w >= 0 && wi.b < a.B && wi.h < a.Hq && wi.q_row0 < wi.S_q &&
                        wi.q_base + wi.S_q <= (a.varlen != nullptr ? a.T_q : a.S_q) &&
                        seq.end <= wi.n_kv,
                    a.status, kDevCheckPrefillItem)) {
        ok = false;
        break;
      }
      if (r > 0) {
        // the Q region is free once both streams' S products of the last item are done
        ok = mbar_wait(bar(kBarQFree), (r - 1) & 1, a.timeout_ns, a.status, kDevTimeoutQ,
                       abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      ++q_loads;
      if (lane == 0) {
        const int nq = wi.has_t1 ? 2 : 1;
        mbar_expect_tx(bar(kBarQ), nq * C::kQTileBytes);
        for (int t = 0; t < nq; ++t)
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(smem_u32(smem + C::kQOff + t * C::kQTileBytes + s * C::kQSub), &tm_q,
                        bar(kBarQ), s * 64, wi.q_base + wi.q_row0 + t * kBM, wi.h, wi.tma_b);
      }
      __syncwarp();
      for (int j = seq.next(0); ok && j < seq.end; j = seq.next(j + 1)) {
      if (!FA_CHECK(j >= 0 && j * kBN < wi.S_kv, a.status, kDevCheckPrefillKv)) {
        ok = false;
        break;
      }
      const bool fix_v = !seq.full(j);
      for (int kv = 0; kv < 2; ++kv) {
        const int slot = item % kRing;
        const int use = item / kRing;
        if (use > 0) {
          ok = mbar_wait(bar(kBarKvEmpty + slot), (use - 1) & 1, a.timeout_ns, a.status,
                         kDevTimeoutKvEmpty, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        const uint32_t dst = smem_u32(smem + C::kRingOff + slot * C::kKvTileBytes);
        const CUtensorMap* map = kv == 0 ? &tm_k : &tm_v;
        if (kv == 1 && fix_v) {
          // land V on the side barrier, zero the rows of excluded keys, publish
          if (lane == 0) {
            mbar_expect_tx(bar(kBarFix), C::kKvTileBytes);
            if constexpr (kPaged) {
              load_paged_tile(dst, map, bar(kBarFix), wi.b, j, kvh);
            } else {
              for (int s = 0; s < D / 64; ++s)
                tma_load_4d(dst + s * C::kKvSub, map, bar(kBarFix), s * 64,
                            wi.kv_base + j * kBN, kvh, wi.tma_b);
            }
          }
          ++item;
          ok = mbar_wait(bar(kBarFix), fixes & 1, a.timeout_ns, a.status, kDevTimeoutKvFull,
                         abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          ++fixes;
          if (!ok) break;
          const uint4 w = seq.words(j);
          uint4* tile = reinterpret_cast<uint4*>(smem + C::kRingOff + slot * C::kKvTileBytes);
          // kBN rows x (D/64 slabs) x 8 chunks of 16 B; a row of a slab is 128
          // contiguous bytes whatever the swizzle
          for (int idx = lane; idx < kBN * (D / 64) * 8; idx += 32) {
            const int r = idx / ((D / 64) * 8);
            const int rest = idx % ((D / 64) * 8);
            const int s = rest / 8, ch = rest % 8;
            const uint32_t word = r < 64 ? (r < 32 ? w.x : w.y) : (r < 96 ? w.z : w.w);
            if (((word >> (r & 31)) & 1u) == 0u)
              tile[(s * C::kKvSub + r * 128) / 16 + ch] = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarKvFull + slot));
        } else {
          if (lane == 0) {
            mbar_expect_tx(bar(kBarKvFull + slot), C::kKvTileBytes);
            if constexpr (kPaged) {
              load_paged_tile(dst, map, bar(kBarKvFull + slot), wi.b, j, kvh);
            } else {
              for (int s = 0; s < D / 64; ++s)
                tma_load_4d(dst + s * C::kKvSub, map, bar(kBarKvFull + slot), s * 64,
                            wi.kv_base + j * kBN, kvh, wi.tma_b);
            }
          }
          ++item;
        }
        __syncwarp();
      }
    }
    }
    if (ok) {
      // tail: wait until the MMA warps have released the last ring slots, so
      // no asynchronous arrival can reach this CTA's shared memory after exit
      for (int it = max(0, item - kRing); it < item && ok; ++it) {
        ok = mbar_wait(bar(kBarKvEmpty + it % kRing), (it / kRing) & 1, a.timeout_ns, a.status,
                       kDevTimeoutKvEmpty, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
      }
    }
    const uint64_t drain_ns = a.timeout_ns > kDrainFloorNs ? a.timeout_ns : kDrainFloorNs;
    if (!ok && lane == 0) {
      // let the copies this CTA started land before its shared memory is released
      for (int it = max(0, item - kRing); it < item; ++it)
        mbar_wait(bar(kBarKvFull + it % kRing), (it / kRing) & 1, drain_ns, a.status,
                  kDevTimeoutDrain, nullptr);
      if (fixes > 0) mbar_wait(bar(kBarFix), (fixes - 1) & 1, drain_ns, a.status,
                               kDevTimeoutDrain, nullptr);
    }
    // the last Q tiles requested have landed (at once unless an MMA warp gave
    // up before it waited for them)
    if (q_loads > 0 && lane == 0)
      mbar_wait(bar(kBarQ), (q_loads - 1) & 1, drain_ns, a.status, kDevTimeoutDrain, nullptr);
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ================================================================ MMA
    // Two issue streams, one per Q tile, that take turns: stream t issues
    // PV_t(j) then S_t(j+1) and hands the turn to the other. One thread
    // cannot issue 128x128x16 MMAs much faster than the tensor core retires
    // them, so a barrier wait inside a single stream leaves the pipe idle;
    // here each stream does its waits (V_j, P_t(j), K_j+1) while the other
    // one is issuing. The turn order keeps the pipe order of one stream
    // (S0 S1 | PV0 S0' | PV1 S1' | ...), so one tile's softmax still runs
    // while the tensor core works on the other tile. Each stream is in
    // order, which keeps S_t(j+1) behind the P_t(j) V_j product that reads
    // the aliased columns; the streams share no TMEM. Both streams wait for
    // and release every ring item (kv_empty counts two arrivals), so neither
    // runs a full ring ahead of the other.
    const int t = warp - kMmaWarp;
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, 0, 1);
      const uint32_t q_base = smem_u32(smem + C::kQOff);
      const uint32_t ring_base = smem_u32(smem + C::kRingOff);
      // Descriptor bases built once; an MMA adds a constant to the 14-bit
      // address field (addresses stay below 256 KB, so the add never carries
      // out of the field). K-major tiles advance 32 B per 16-element k-step
      // inside a 128-byte swizzle row and one slab (kBM or kBN rows of 128 B)
      // per 64 columns; the MN-major V operand advances 16 keys = 2 KB per
      // k-step.
      const uint64_t dq = smem_desc_sw128(q_base + t * C::kQTileBytes, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(ring_base, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(ring_base, C::kKvSub, 1024);
      constexpr uint32_t kSlotStep = C::kKvTileBytes >> 4;
      const uint32_t s_tmem = tmem + t * 128;
      const uint32_t o_tmem = tmem + 256 + t * 128;
      auto issue_s = [&](int slot) {
        const uint64_t bk = dk0 + static_cast<uint64_t>(slot) * kSlotStep;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offq = ((kk / 4) * C::kQSub + (kk % 4) * 32) >> 4;
          const uint32_t offk =
              C::kQSub == C::kKvSub ? offq : ((kk / 4) * C::kKvSub + (kk % 4) * 32) >> 4;
          umma_ss(s_tmem, dq + offq, bk + offk, idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int slot, bool first) {
        const uint64_t bv = dv0 + static_cast<uint64_t>(slot) * kSlotStep;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts(o_tmem, s_tmem + kk * 8, bv + ((kk * 16 * 128) >> 4), idesc_pv,
                  (first && kk == 0) ? 0u : 1u);
      };
      // bounded wait for this stream's turn (turn 2u + t in issue round u)
      auto take_turn = [&](int want) -> bool {
        if (*turn == want) return true;
        const uint64_t t0 = globaltimer_ns();
        while (*turn != want) {
          if (*abort_flag) return false;
          if (globaltimer_ns() - t0 > a.timeout_ns) {
            record_error(a.status, kDevTimeoutTurn);
            *abort_flag = 1;
            return false;
          }
        }
        return true;
      };
      if constexpr (C::QT == 1) {
        // One Q tile per item (D = 256): a single issue stream with the S tile
        // double-buffered in TMEM (buffers [0, kBN) and [kBN, 2 kBN), by KV tile
        // parity). S of tile g+2 goes into the buffer of tile g right behind
        // PV of tile g, so the softmax of tile g+1 runs while the tensor core
        // does PV(g) and S(g+2). kBarSFull/kBarPReady + buffer hand the tiles
        // over; kBarOFinal + 1 completes once per P·V (the softmax waits on it
        // before it rescales O). The second issue warp has no work.
        if (t == 0) {
          int item = 0;  // ring items consumed so far
          int g = 0;     // KV tiles processed so far (all work items)
          bool ok = true;
          for (int r = 0; ok; ++r) {
            const int w = item_of(r);
            if (w >= a.n_items) break;
            const WorkItem<D> wi = work_item<D>(a, w);
            const auto& seq = wi.seq;
            ok = mbar_wait(bar(kBarQ), r & 1, a.timeout_ns, a.status, kDevTimeoutQ, abort_flag);
            if (!ok) break;
            tc_fence_after();
            int js = seq.next(0);  // next tile whose S is issued
            int jp = js;           // next tile whose P·V is issued
            int n_s = 0, n_p = 0;  // S and P·V products of this item so far
            auto issue_next_s = [&]() -> bool {
              const int it_k = item + 2 * n_s;  // ring items go K, V, K, V, ...
              const int slot = it_k % kRing;
              if (!mbar_wait(bar(kBarKvFull + slot), (it_k / kRing) & 1, a.timeout_ns, a.status,
                             kDevTimeoutKvFull, abort_flag))
                return false;
              tc_fence_after();
              const int b = (g + n_s) & 1;
              const uint64_t bk = dk0 + static_cast<uint64_t>(slot) * kSlotStep;
              // the 16 Q descriptors are recomputed per tile, not kept live
              // (they would take 32 of this warp's 72 registers)
              uint64_t dqv = dq;
              asm volatile("" : "+l"(dqv));
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t offq = ((kk / 4) * C::kQSub + (kk % 4) * 32) >> 4;
                const uint32_t offk = ((kk / 4) * C::kKvSub + (kk % 4) * 32) >> 4;
                umma_ss(tmem + b * kBN, dqv + offq, bk + offk, idesc_s, kk > 0 ? 1u : 0u);
              }
              umma_commit(bar(kBarSFull + b));
              umma_commit(bar(kBarKvEmpty + slot));  // the slot counts two releases
              umma_commit(bar(kBarKvEmpty + slot));
              ++n_s;
              js = seq.next(js + 1);
              if (!(js < seq.end)) {  // Q is free once the item's last S is issued
                umma_commit(bar(kBarQFree));
                umma_commit(bar(kBarQFree));
              }
              return true;
            };
            if (!(js < seq.end)) {
              // the item sees no key
              umma_commit(bar(kBarQFree));
              umma_commit(bar(kBarQFree));
              umma_commit(bar(kBarOFinal));
              continue;
            }
            ok = issue_next_s();
            if (ok && js < seq.end) ok = issue_next_s();
            while (ok && jp < seq.end) {
              const int b = (g + n_p) & 1;
              const int iv = item + 2 * n_p + 1;
              const int v_slot = iv % kRing;
              ok = mbar_wait(bar(kBarKvFull + v_slot), (iv / kRing) & 1, a.timeout_ns, a.status,
                             kDevTimeoutKvFull, abort_flag);
              if (ok)
                ok = mbar_wait(bar(kBarPReady + b), ((g + n_p) >> 1) & 1, a.timeout_ns, a.status,
                               kDevTimeoutPReady, abort_flag);
              if (ok && n_p == 0 && r > 0)
                // O of the previous item must be read out before it is overwritten
                ok = mbar_wait(bar(kBarODrained), (r - 1) & 1, a.timeout_ns, a.status,
                               kDevTimeoutOFinal, abort_flag);
              if (!ok) break;
              tc_fence_after();
              const uint64_t bv = dv0 + static_cast<uint64_t>(v_slot) * kSlotStep;
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                umma_ts(o_tmem, tmem + b * kBN + kk * 8, bv + ((kk * 16 * 128) >> 4), idesc_pv,
                        (n_p == 0 && kk == 0) ? 0u : 1u);
              umma_commit(bar(kBarOFinal + 1));  // this P·V is done
              umma_commit(bar(kBarKvEmpty + v_slot));
              umma_commit(bar(kBarKvEmpty + v_slot));
              ++n_p;
              jp = seq.next(jp + 1);
              if (!(jp < seq.end)) umma_commit(bar(kBarOFinal));
              if (js < seq.end) ok = issue_next_s();
            }
            item += 2 * n_s;
            g += n_s;
          }
        }
      } else {
      int item = 0;      // ring items consumed so far
      int pv_count = 0;  // P_t tiles consumed so far (all work items)
      int u = 0;         // issue rounds so far (both streams run the same rounds)
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int w = item_of(r);
        if (w >= a.n_items) break;
        const WorkItem<D> wi = work_item<D>(a, w);
        const auto& seq = wi.seq;
        // this stream's KV tiles: those of the item's sequence in [lo, n)
        const int lo = t == 0 ? wi.lo_t[0] : wi.lo_t[1];
        const int n = t == 0 ? wi.n_t[0] : wi.n_t[1];
        auto mine = [&](int jj) { return jj >= lo && jj < n; };
        const bool has_any = seq.next(lo) < n;
        ok = mbar_wait(bar(kBarQ), r & 1, a.timeout_ns, a.status, kDevTimeoutQ, abort_flag);
        if (!ok) break;
        tc_fence_after();
        int j = seq.next(0);
        bool q_freed = false;
        bool first_pv = true;
        // first round of the item: S of the first tile
        if (j < seq.end) {
          const int slot = item % kRing;
          ok = mbar_wait(bar(kBarKvFull + slot), (item / kRing) & 1, a.timeout_ns, a.status,
                         kDevTimeoutKvFull, abort_flag);
          if (ok) ok = take_turn(2 * u + t);
          if (!ok) break;
          tc_fence_after();
          if (mine(j)) issue_s(slot);
          *turn = 2 * u + t + 1;
          ++u;
          if (mine(j)) umma_commit(bar(kBarSFull + t));
          umma_commit(bar(kBarKvEmpty + slot));
        }
        // release Q once this stream's last S product of the item is issued
        if (!has_any || (mine(j) && !(seq.next(j + 1) < n))) {
          umma_commit(bar(kBarQFree));
          q_freed = true;
        }
        if (!has_any) umma_commit(bar(kBarOFinal + t));  // sees no key (or tile absent)
        while (ok && j < seq.end) {
          const int v_item = item + 1;
          const int v_slot = v_item % kRing;
          const int jn = seq.next(j + 1);
          const int k_item = item + 2;
          const int k_slot = k_item % kRing;
          ok = mbar_wait(bar(kBarKvFull + v_slot), (v_item / kRing) & 1, a.timeout_ns, a.status,
                         kDevTimeoutKvFull, abort_flag);
          if (ok && mine(j))
            ok = mbar_wait(bar(kBarPReady + t), pv_count & 1, a.timeout_ns, a.status,
                           kDevTimeoutPReady, abort_flag);
          if (ok && mine(j) && first_pv && r > 0)
            // O_t of the previous item must be read out before it is overwritten
            ok = mbar_wait(bar(kBarODrained + t), (r - 1) & 1, a.timeout_ns, a.status,
                           kDevTimeoutOFinal, abort_flag);
          if (ok && jn < seq.end)
            ok = mbar_wait(bar(kBarKvFull + k_slot), (k_item / kRing) & 1, a.timeout_ns,
                           a.status, kDevTimeoutKvFull, abort_flag);
          if (ok) ok = take_turn(2 * u + t);
          if (!ok) break;
          tc_fence_after();
          if (mine(j)) issue_pv(v_slot, first_pv);
          if (mine(jn)) issue_s(k_slot);
          *turn = 2 * u + t + 1;
          ++u;
          if (mine(j)) {
            ++pv_count;
            first_pv = false;
          }
          if (mine(jn)) umma_commit(bar(kBarSFull + t));
          if (mine(jn) && !q_freed && !(seq.next(jn + 1) < n)) {
            umma_commit(bar(kBarQFree));
            q_freed = true;
          }
          if (mine(j) && !(jn < n)) umma_commit(bar(kBarOFinal + t));
          umma_commit(bar(kBarKvEmpty + v_slot));
          if (jn < seq.end) umma_commit(bar(kBarKvEmpty + k_slot));
          item += 2;
          j = jn;
        }
      }
      }
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kSoftmaxRegs));
    // ============================================================ softmax
    const int t = warp / 4;          // Q tile of this warpgroup
    const int wl = warp % 4;         // TMEM lane quarter
    const int row_in_tile = wl * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(wl * 32) << 16;
    const uint32_t s_tmem_t = tmem + lane_bits + t * 128;
    const uint32_t o_tmem = tmem + lane_bits + 256 + t * 128;
    const float c = a.scale_log2;
    int k = 0;  // S_t tiles consumed so far (all work items)
    bool ok = true;
    // with one Q tile per item (D = 256) the second warpgroup has no rows
    for (int r = 0; ok && (C::QT == 2 || t == 0); ++r) {
      const int w = item_of(r);
      if (w >= a.n_items) break;
      const WorkItem<D> wi = work_item<D>(a, w);
      const auto& seq = wi.seq;
      const int q_row0 = wi.q_row0;
      const int row = q_row0 + t * kBM + row_in_tile;
      float m_run = -INFINITY;  // reference max, log2 domain
      float l_run = 0.f;
      const int lo_mine = t == 0 ? wi.lo_t[0] : wi.lo_t[1];
      const int n_mine = t == 0 ? wi.n_t[0] : wi.n_t[1];
      for (int j = seq.next(lo_mine); j < n_mine; j = seq.next(j + 1), ++k) {
      // S of this tile: the Q tile's buffer, or with one Q tile per item the
      // buffer of this KV tile's parity
      const int sb = C::QT == 1 ? (k & 1) : t;
      const uint32_t s_tmem = C::QT == 1 ? tmem + lane_bits + (k & 1) * kBN : s_tmem_t;
      ok = mbar_wait(bar(kBarSFull + sb), C::QT == 1 ? (k >> 1) & 1 : k & 1, a.timeout_ns, a.status, kDevTimeoutSFull,
                     abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      constexpr int NQ4 = C::NQ4;
      uint32_t sr[NQ4][32];
      // per-element path: masked tiles, and a negative scale (whose row max is
      // the scale times the row min)
      const int r0 = q_row0 + t * kBM;
      const bool masked = (a.win_right >= 0 && j * kBN + kBN - 1 > r0 + a.win_right) ||
                          (a.win_left >= 0 && j * kBN < r0 + kBM - 1 - a.win_left) ||
                          ((j + 1) * kBN > wi.S_kv) || !seq.full(j) || c < 0.f;
      float tmax = -INFINITY;
      if (masked) {
#pragma unroll
        for (int q4 = 0; q4 < NQ4; ++q4) tmem_ld32(s_tmem + q4 * 32, sr[q4]);
        tmem_ld_wait();
        uint32_t words[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
        if (seq.bits != nullptr) {
          const uint4 w = seq.words(j);
          words[0] = w.x; words[1] = w.y; words[2] = w.z; words[3] = w.w;
        }
        // this row's keys of the tile, [lo_k, hi_k) relative to its first key:
        // past S_kv, or outside the window (causal is the window (-1, 0)),
        // folded into the validity words
        {
          const int base = j * kBN;
          int hi_k = wi.S_kv - base;
          if (a.win_right >= 0) hi_k = min(hi_k, row + a.win_right + 1 - base);
          const int lo_k = a.win_left >= 0 ? row - a.win_left - base : 0;
#pragma unroll
          for (int q4 = 0; q4 < NQ4; ++q4) {
            const int lo_i = min(max(lo_k - q4 * 32, 0), 32);
            const int hi_i = min(max(hi_k - q4 * 32, 0), 32);
            const uint32_t below_hi = hi_i >= 32 ? 0xFFFFFFFFu : ((1u << hi_i) - 1u);
            const uint32_t below_lo = lo_i >= 32 ? 0xFFFFFFFFu : ((1u << lo_i) - 1u);
            words[q4] &= below_hi & ~below_lo;
          }
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q4 = 0; q4 < NQ4; ++q4) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const bool valid = (words[q4] >> i) & 1u;
            const float tv = valid ? __uint_as_float(sr[q4][i]) * c : -INFINITY;
            sr[q4][i] = __float_as_uint(tv);
            mx[q4 % 4] = fmaxf(mx[q4 % 4], tv);
          }
        }
        tmax = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
      } else if constexpr (NQ4 == 2) {
        // 64 keys: both halves in one round of TMEM loads
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
        tmem_ld32(s_tmem, sr[0]);
        tmem_ld32(s_tmem + 32, sr[NQ4 - 1]);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < NQ4; ++q4)
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mx[(q4 * 16 + i / 2) % 8] = fmax3(mx[(q4 * 16 + i / 2) % 8], __uint_as_float(sr[q4][i]),
                                              __uint_as_float(sr[q4][i + 1]));
        tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * c;
      } else {
        // row max with 8 independent accumulators; the first half's max runs
        // while the second half is still being read out of TMEM
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
        tmem_ld32(s_tmem, sr[0]);
        tmem_ld32(s_tmem + 32, sr[1]);
        tmem_ld_wait();
        tmem_ld32(s_tmem + 64, sr[2]);
        tmem_ld32(s_tmem + 96, sr[3]);
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4)
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mx[(q4 * 16 + i / 2) % 8] = fmax3(mx[(q4 * 16 + i / 2) % 8], __uint_as_float(sr[q4][i]),
                                              __uint_as_float(sr[q4][i + 1]));
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 2; q4 < 4; ++q4)
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mx[(q4 * 16 + i / 2) % 8] = fmax3(mx[(q4 * 16 + i / 2) % 8], __uint_as_float(sr[q4][i]),
                                              __uint_as_float(sr[q4][i + 1]));
        tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * c;
      }
      // conditional rescale: keep the reference max unless it grows by > 2^8
      const float m_cand = fmaxf(m_run, tmax);
      float alpha = 1.f;
      const bool need = m_cand > m_run + kRescaleThreshold;
      if (need) {
        alpha = ex2(m_run - m_cand);  // 0 when m_run was -inf
        m_run = m_cand;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // p = 2^(s*c - m): packed f32x2 FMA, then ex2; row sum in two packed lanes
      uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};  // independent row-sum chains
      const uint64_t c2 = masked ? pair_f32(1.f, 1.f) : pair_f32(c, c);
      const uint64_t nm2 = pair_f32(-m_use, -m_use);
#pragma unroll
      for (int half = 0; half < NQ4 / 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int q4 = half * 2 + qq;
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 t2 = unpair(ffma2(pair_u32(sr[q4][i], sr[q4][i + 1]), c2, nm2));
            const float p0 = ex2(t2.x);
            const float p1 = ex2(t2.y);
            rs2[(i / 2) % 4] = fadd2(rs2[(i / 2) % 4], pair_f32(p0, p1));
            pk[qq * 16 + i / 2] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st32(s_tmem + half * 32, pk);
      }
      const float2 rsa = unpair(fadd2(rs2[0], rs2[1]));
      const float2 rsb = unpair(fadd2(rs2[2], rs2[3]));
      const float rsum = (rsa.x + rsa.y) + (rsb.x + rsb.y);
      l_run = l_run * alpha + rsum;
      if (k > 0 && __any_sync(0xffffffffu, need)) {
        if constexpr (C::QT == 1) {
          // the previous tile's P·V may still be running: wait until it is done
          ok = mbar_wait(bar(kBarOFinal + 1), (k - 1) & 1, a.timeout_ns, a.status,
                         kDevTimeoutOFinal, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
        }
        // O_t was complete when S_t(j) landed (tcgen05 ops retire in order)
#pragma unroll
        for (int q4 = 0; q4 < D / 32; ++q4) {
          uint32_t orr[32];
          tmem_ld32(o_tmem + q4 * 32, orr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
          tmem_st32(o_tmem + q4 * 32, orr);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarPReady + sb));
      }
      if (!ok) break;
      // ---- epilogue: out = O / l, lse = ln2 * (m + log2 l)
      ok = mbar_wait(bar(kBarOFinal + t), r & 1, a.timeout_ns, a.status, kDevTimeoutOFinal,
                     abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // the O row in rounds of up to 128 columns of TMEM loads (one round
      // unless D = 256); O_t is free for the next item's products as soon as
      // the last round is read
      constexpr int kRound = D < 128 ? D / 32 : D == 256 ? 2 : 4;
      uint32_t orr[kRound][32];
#pragma unroll
      for (int q4 = 0; q4 < kRound; ++q4) tmem_ld32(o_tmem + q4 * 32, orr[q4]);
      tmem_ld_wait();
      if (kRound == D / 32) {
        tc_fence_before();
        mbar_arrive(bar(kBarODrained + t));
      }
      const bool row_ok = row < wi.S_q &&
                          FA_CHECK(wi.q_base + row < (a.varlen != nullptr ? a.T_q : a.S_q),
                                   a.status, kDevCheckPrefillOut);
      const bool invalid = (l_run == 0.f);
      const float inv_l = invalid ? 0.f : 1.f / l_run;
      __nv_bfloat16* dst = a.out + static_cast<long long>(wi.tma_b) * a.out_batch_stride +
                           static_cast<long long>(wi.h) * a.out_head_stride +
                           static_cast<long long>(wi.q_base + row) * a.out_row_stride;
#pragma unroll
      for (int q0 = 0; q0 < D / 32; q0 += kRound) {
        if (q0 > 0) {
#pragma unroll
          for (int q4 = 0; q4 < kRound; ++q4) tmem_ld32(o_tmem + (q0 + q4) * 32, orr[q4]);
          tmem_ld_wait();
          if (q0 + kRound == D / 32) {
            tc_fence_before();
            mbar_arrive(bar(kBarODrained + t));
          }
        }
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < kRound; ++q4) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + (q0 + q4) * 32);
            // an invalid row writes exact zeros: its O columns may never have
            // been written by an MMA
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                f[e] = invalid ? 0.f : __uint_as_float(orr[q4][i + e]) * inv_l;
              d4[i / 8] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                     pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
            }
          }
        }
      }
      if (row_ok && a.lse != nullptr)
        // [B, Hq, S_q], or [T_q, Hq] for packed sequences
        a.lse[a.varlen != nullptr ? static_cast<long long>(wi.q_base + row) * a.Hq + wi.h
                                  : (static_cast<long long>(wi.b) * a.Hq + wi.h) * a.S_q + row] =
            invalid ? INFINITY : (m_run + log2f(l_run)) * 0.69314718055994530942f;
    }
  }

  // ---- teardown: every role is done with TMEM and shared memory
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    tc_fence_after();
    if (*abort_flag && lane == 0) {
      // in-flight MMAs of this stream retire in order: one commit covers them
      const int t = warp - kMmaWarp;
      umma_commit(bar(kBarDrain + t));
      const uint64_t drain_ns = a.timeout_ns > kDrainFloorNs ? a.timeout_ns : kDrainFloorNs;
      mbar_wait(bar(kBarDrain + t), 0, drain_ns, a.status, kDevTimeoutDrain, nullptr);
    }
    __syncwarp();
    asm volatile("bar.sync 1, 64;" ::: "memory");  // both streams drained
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
  }
}

// One 128-bit validity word set per (batch, 128-key tile). Padded layouts:
// key j of batch b is valid iff j < S_kv, j < lens[b] and key_mask[b][j] == 0.
// Packed sequences (varlen = the [5][B] table): key j of sequence b is valid
// iff j < its used kv length and the flag of its packed row (kv offset + j)
// is 0.
__global__ void tile_bits_kernel(const uint8_t* __restrict__ key_mask, const int* __restrict__ lens,
                                 const int32_t* __restrict__ varlen, int B, int S_kv, int n_tiles,
                                 uint32_t* __restrict__ bits) {
  const int tile = blockIdx.x;
  const int b = blockIdx.y;
  const int key = tile * kBitsTile + threadIdx.x;
  bool valid = key < S_kv;
  size_t mask_at = static_cast<size_t>(b) * S_kv + key;
  if (varlen != nullptr) {
    valid = key < __ldg(varlen + 3 * B + b);
    mask_at = static_cast<size_t>(__ldg(varlen + 2 * B + b)) + key;
  }
  if (valid && lens != nullptr) valid = key < lens[b];
  if (valid && key_mask != nullptr) valid = key_mask[mask_at] == 0;
  const uint32_t word = __ballot_sync(0xffffffffu, valid);
  if ((threadIdx.x & 31) == 0)
    bits[(static_cast<size_t>(b) * n_tiles + tile) * 4 + (threadIdx.x >> 5)] = word;
}

// Packed sequences cut by seqused_q: the query rows between a sequence's used
// length and its span get out = 0 and lse = +inf (rows with no valid key,
// FlashAttn guide §1.7). One thread per 16-byte chunk of such a row and head;
// blockIdx.y is the sequence.
template <int D>
__global__ void truncated_rows_kernel(const int32_t* __restrict__ varlen, int B, int Hq,
                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  constexpr int kChunks = D / 8;  // 16-byte chunks of a row of one head
  const int b = blockIdx.y;
  const int q_off = __ldg(varlen + b);
  const int used = __ldg(varlen + B + b);
  const int span = __ldg(varlen + 4 * B + b);
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(span - used) * Hq * kChunks) return;
  const int r = static_cast<int>(idx / (Hq * kChunks));
  const int h = static_cast<int>((idx / kChunks) % Hq);
  const int c = static_cast<int>(idx % kChunks);
  const long long row = static_cast<long long>(q_off) + used + r;  // packed row
  reinterpret_cast<uint4*>(out + (row * Hq + h) * D)[c] = make_uint4(0u, 0u, 0u, 0u);
  if (c == 0 && lse != nullptr) lse[row * Hq + h] = INFINITY;
}

__global__ void wait_probe_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  const uint32_t b = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives: the bounded wait must give up and record the error
  if (threadIdx.x == 0) mbar_wait(b, 0, timeout_ns, status, kDevTimeoutProbe, nullptr);
}

template <int D>
cudaError_t launch_prefill_d(const PrefillLaunch& x, cudaStream_t stream) {
  using C = PCfg<D>;
  constexpr int kBN = C::BN;
  static std::atomic<uint64_t> configured{0};  // devices with the attributes set
  if (setup_needed(configured)) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_kernel<D, Pages>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    setup_done(configured);
  }
  CUtensorMap mq, mk, mv;
  // packed sequences: [T, H, D] tensors, one batch of T rows
  const bool packed = x.varlen != nullptr;
  const bool paged = x.block_table != nullptr;
  const int64_t map_B = packed ? 1 : x.B;
  const int64_t S_q_map = packed ? std::max<int64_t>(x.T_q, 1) : x.S_q;
  const int64_t S_kv_map = packed ? std::max<int64_t>(x.T_kv, 1) : (x.S_kv > 0 ? x.S_kv : 1);
  // a paged cache is a batch of num_blocks sequences of block_size rows
  // (PA_BBND rows as BSND, PA_BNBD as BNSD), loaded in boxes of
  // gcd(block_size, kBN) rows: each box lies inside one block
  const int box_rows = paged ? std::gcd(x.block_size, kBN) : kBN;
  const int kv_layout = !paged ? x.layout
                        : x.kv_layout == FA_LAYOUT_PA_BBND ? FA_LAYOUT_BSND
                                                           : FA_LAYOUT_BNSD;
  const int64_t kv_B = paged ? x.num_blocks : map_B;
  const int64_t kv_S = paged ? x.block_size : S_kv_map;
  if (!encode_bf16_map(&mq, x.q, x.layout, map_B, x.Hq, S_q_map, D, 64, kBM,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_bf16_map(&mk, x.k, kv_layout, kv_B, x.Hkv, kv_S, D, 64, box_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_bf16_map(&mv, x.v, kv_layout, kv_B, x.Hkv, kv_S, D, 64, box_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  PrefillArgs pa;
  pa.out = static_cast<__nv_bfloat16*>(x.out);
  pa.lse = x.lse;
  pa.tile_bits = x.tile_bits;
  pa.sched = x.sched;
  pa.varlen = x.varlen;
  pa.status = x.status;
  pa.timeout_ns = x.timeout_ns;
  pa.B = x.B;
  pa.Hq = x.Hq;
  pa.Hkv = x.Hkv;
  pa.S_q = x.S_q;
  pa.S_kv = x.S_kv;
  pa.win_left = x.win_left;
  pa.win_right = x.win_right;
  pa.n_qpairs = (x.S_q + C::QT * kBM - 1) / (C::QT * kBM);
  pa.n_kv_tiles = (x.S_kv + kBN - 1) / kBN;
  pa.n_items = pa.n_qpairs * x.B * x.Hq;
  if (x.layout == FA_LAYOUT_BNSD) {
    pa.out_row_stride = D;
    pa.out_head_stride = static_cast<long long>(x.S_q) * D;
    pa.out_batch_stride = static_cast<long long>(x.Hq) * x.S_q * D;
  } else {
    pa.out_row_stride = static_cast<long long>(x.Hq) * D;
    pa.out_head_stride = D;
    pa.out_batch_stride = static_cast<long long>(x.S_q) * x.Hq * D;
  }
  pa.scale_log2 = x.scale * 1.4426950408889634f;
#ifdef FA_DEBUG
  pa.T_q = x.T_q;
#endif
  // persistent: one CTA per SM (each CTA holds all 512 TMEM columns)
  const int grid = x.grid;  // the schedule in the workspace was built for this grid
  if (paged)
    prefill_kernel<D, Pages><<<grid, kThreads, C::kSmemBytes, stream>>>(
        mq, mk, mv, pa, Pages{x.block_table, x.max_blocks, x.block_size, box_rows});
  else
    prefill_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, pa, NoPages{});
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& x, cudaStream_t stream) {
  return x.D == 256   ? launch_prefill_d<256>(x, stream)
         : x.D == 128 ? launch_prefill_d<128>(x, stream)
                      : launch_prefill_d<64>(x, stream);
}

cudaError_t launch_tile_bits(const uint8_t* key_mask, const int* lens_dev, const int32_t* varlen,
                             int B, int S_kv, uint32_t* bits, cudaStream_t stream) {
  const int n_tiles = (S_kv + kBitsTile - 1) / kBitsTile;
  tile_bits_kernel<<<dim3(n_tiles, B), kBitsTile, 0, stream>>>(key_mask, lens_dev, varlen, B,
                                                               S_kv, n_tiles, bits);
  return cudaGetLastError();
}

cudaError_t launch_truncated_rows(const int32_t* varlen, int B, int most_rows, int Hq, int D,
                                  void* out, float* lse, cudaStream_t stream) {
  if (B == 0 || most_rows == 0) return cudaSuccess;
  const long long work = static_cast<long long>(most_rows) * Hq * (D / 8);
  const dim3 grid(static_cast<unsigned>((work + 255) / 256), B);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  if (D == 256) truncated_rows_kernel<256><<<grid, 256, 0, stream>>>(varlen, B, Hq, o, lse);
  else if (D == 128) truncated_rows_kernel<128><<<grid, 256, 0, stream>>>(varlen, B, Hq, o, lse);
  else truncated_rows_kernel<64><<<grid, 256, 0, stream>>>(varlen, B, Hq, o, lse);
  return cudaGetLastError();
}

cudaError_t launch_wait_probe(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa
