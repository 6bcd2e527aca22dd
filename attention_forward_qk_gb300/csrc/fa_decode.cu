// Split-KV decode (S_q = 1) for sm_103a.
//
// Stage 1 (decode_chunk_kernel): one CTA per (batch, chunk of KV rows,
// KV head [, group of query heads]). A producer warp streams the chunk's K
// and V rows through a 4-stage shared-memory ring with TMA tensor loads;
// seven consumer warps compute q.k with 128-bit shared loads, packed f32x2
// FMAs and butterfly shuffles over the 8 lanes that share a row (every query
// head of the GQA group reuses the same K/V row), keep
// an online softmax (running max m and sum l, exp2 domain) per head and
// accumulate p*v. The chunk's normalised partial output o/l and its
// log-sum-exp are written to the workspace. This is the FlashDecoding
// tutorial's stage 1 (§3.2) and the FlashAttn guide's FA phase of
// FlashDecode (§1.9), with the scale and the length mask applied.
//
// Stage 2 (decode_merge_kernel): one CTA per (batch, query head) merges the
// chunks by their log-sum-exp with the largest value factored out:
//   M = max_c lse_c, w_c = 2^(lse_c - M), out = sum_c w_c o_c / sum_c w_c,
//   lse = M + log2(sum_c w_c)  (reported as natural log)
// which is aclnnIncreFlashAttention guide §8.3's combine() and the FlashAttn
// guide §10 formula written for normalised partials.
//
// Rows at or past a batch's length are never read by any arithmetic (they
// may be loaded into shared memory with the rest of a box, and are skipped),
// so stale cache contents, NaN included, cannot reach the output.
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

// 7 consumer warps + 1 producer warp: 256 threads keeps the per-thread
// register budget at 255 (larger CTAs are capped at 168).
constexpr int kDecWarps = 7;                       // consumer warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + one producer warp
constexpr int kDecStages = 4;
constexpr int kDecStageBytes = 28672;              // K rows + V rows of one stage
constexpr int kDecSmemBytes = kDecStages * kDecStageBytes + 256;
constexpr int kMergeThreads = 256;

template <int D>
struct DecCfg {
  static constexpr int LPR = 8;                         // lanes per K/V row
  static constexpr int NCH = D / 64;                    // 16-byte chunks of a row per lane
  static constexpr int RPW = 32 / LPR;                  // rows per warp per step
  static constexpr int R = kDecStageBytes / (2 * D * 2);  // rows per stage (56 or 112)
  static constexpr int RPWS = R / kDecWarps;            // rows per warp per stage
  static constexpr int STEPS = RPWS / RPW;
  static constexpr int TILE_BYTES = R * D * 2;
};

struct DecodeArgs {
  const __nv_bfloat16* q;
  const uint8_t* key_mask;
  const int* lens;
  const int2* items;
  float* part_o;
  float* part_lse;
  uint32_t* status;
  uint64_t timeout_ns;
  int Hq, Hkv, S_kv, chunk, max_chunks, head_groups;
  float scale_log2;
};

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_chunk_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  using C = DecCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecStages * kDecStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kDecStages);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int2 item = a.items[blockIdx.x];
  const int b = item.x;
  const int c = item.y;
  const int kvh = blockIdx.y / a.head_groups;
  const int hg = blockIdx.y % a.head_groups;
  const int g_total = a.Hq / a.Hkv;
  const int h0 = kvh * g_total + hg * G;  // first query head of this CTA
  const int L = a.lens[b];
  const int row_begin = c * a.chunk;
  const int row_end = min(row_begin + a.chunk, L);
  const int nstage = (row_end - row_begin + C::R - 1) / C::R;

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kDecStages);
  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kDecWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // per-lane softmax state (consumers); o holds this lane's 8*NCH elements
  // of every head's output as fp32 pairs
  constexpr int NP = 4 * C::NCH;  // fp32 pairs per lane
  float m[G], l[G];
  uint64_t o[G][NP];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int k = 0; k < NP; ++k) o[h][k] = 0ull;
  }
  const int sub = lane % C::LPR;  // this lane owns 16-byte chunks sub, sub+8, ... of a row
  const int rg = lane / C::LPR;   // row group within a warp step

  if (warp == kDecWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      int issued = 0;
      for (int st = 0; st < nstage; ++st) {
        const int slot = st % kDecStages;
        const int use = st / kDecStages;
        if (use > 0 && !mbar_wait(empty0 + 8 * slot, (use - 1) & 1, a.timeout_ns, a.status,
                                  kDevTimeoutDecodeEmpty, abort_flag))
          break;
        const uint32_t dst = smem_u32(smem + slot * kDecStageBytes);
        mbar_expect_tx(full0 + 8 * slot, 2 * C::TILE_BYTES);
        tma_load_4d(dst, &tm_k, full0 + 8 * slot, 0, row_begin + st * C::R, kvh, b);
        tma_load_4d(dst + C::TILE_BYTES, &tm_v, full0 + 8 * slot, 0, row_begin + st * C::R, kvh,
                    b);
        issued = st + 1;
      }
      if (*abort_flag) {
        // let every copy this CTA started land before shared memory is released
        for (int st = max(0, issued - kDecStages); st < issued; ++st)
          mbar_wait(full0 + 8 * (st % kDecStages), (st / kDecStages) & 1, a.timeout_ns, a.status,
                    kDevTimeoutDrain, nullptr);
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    uint64_t qp[G][NP];  // q * scale * log2(e), as fp32 pairs
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const __nv_bfloat16* qh = a.q + (static_cast<size_t>(b) * a.Hq + h0 + h) * D;
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch) {
        const uint4 u = *reinterpret_cast<const uint4*>(qh + (sub + 8 * ch) * 8);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = bf16lo_to_f32(w4[k]) * a.scale_log2;
          const float hi = bf16hi_to_f32(w4[k]) * a.scale_log2;
          qp[h][ch * 4 + k] = pair_f32(lo, hi);
        }
      }
    }
    const uint8_t* mask_row =
        a.key_mask ? a.key_mask + static_cast<size_t>(b) * a.S_kv : nullptr;

    for (int st = 0; st < nstage; ++st) {
      const int slot = st % kDecStages;
      if (!mbar_wait(full0 + 8 * slot, (st / kDecStages) & 1, a.timeout_ns, a.status,
                     kDevTimeoutDecodeFull, abort_flag))
        break;
      const __nv_bfloat16* Ks =
          reinterpret_cast<const __nv_bfloat16*>(smem + slot * kDecStageBytes);
      const __nv_bfloat16* Vs = Ks + C::R * D;
      const int stage_row0 = row_begin + st * C::R;

      float s[C::STEPS][G];
      bool valid[C::STEPS];
#pragma unroll
      for (int i = 0; i < C::STEPS; ++i) {
        const int r = warp * C::RPWS + i * C::RPW + rg;
        const int gr = stage_row0 + r;
        bool ok = gr < row_end;
        if (ok && mask_row != nullptr) ok = mask_row[gr] == 0;
        valid[i] = ok;
        uint64_t kp[NP];
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          const uint4 u = *reinterpret_cast<const uint4*>(Ks + r * D + (sub + 8 * ch) * 8);
          kp[ch * 4 + 0] = bf16x2_pair(u.x);
          kp[ch * 4 + 1] = bf16x2_pair(u.y);
          kp[ch * 4 + 2] = bf16x2_pair(u.z);
          kp[ch * 4 + 3] = bf16x2_pair(u.w);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          uint64_t acc2 = 0ull;
#pragma unroll
          for (int k = 0; k < NP; ++k) acc2 = ffma2(qp[h][k], kp[k], acc2);
          const float2 a2 = unpair(acc2);
          float acc = a2.x + a2.y;
#pragma unroll
          for (int off = C::LPR / 2; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
          s[i][h] = ok ? acc : -INFINITY;
        }
      }
      // online softmax update for this stage's rows (exp2 domain)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = s[0][h];
#pragma unroll
        for (int i = 1; i < C::STEPS; ++i) mx = fmaxf(mx, s[i][h]);
        const float mn = fmaxf(m[h], mx);
        const float m_use = (mn == -INFINITY) ? 0.f : mn;
        const float alpha = ex2(m[h] - m_use);  // 0 when m was -inf
        m[h] = mn;
        l[h] *= alpha;
        const uint64_t a2 = pair_f32(alpha, alpha);
#pragma unroll
        for (int k = 0; k < NP; ++k) o[h][k] = ffma2(o[h][k], a2, 0ull);
#pragma unroll
        for (int i = 0; i < C::STEPS; ++i) {
          s[i][h] = ex2(s[i][h] - m_use);  // -inf -> 0
          l[h] += s[i][h];
        }
      }
#pragma unroll
      for (int i = 0; i < C::STEPS; ++i) {
        const int r = warp * C::RPWS + i * C::RPW + rg;
        uint64_t vp[NP];
#pragma unroll
        for (int ch = 0; ch < C::NCH; ++ch) {
          uint4 u = *reinterpret_cast<const uint4*>(Vs + r * D + (sub + 8 * ch) * 8);
          if (!valid[i]) u = make_uint4(0u, 0u, 0u, 0u);  // stale rows never enter a product
          vp[ch * 4 + 0] = bf16x2_pair(u.x);
          vp[ch * 4 + 1] = bf16x2_pair(u.y);
          vp[ch * 4 + 2] = bf16x2_pair(u.z);
          vp[ch * 4 + 3] = bf16x2_pair(u.w);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const uint64_t p2 = pair_f32(s[i][h], s[i][h]);
#pragma unroll
          for (int k = 0; k < NP; ++k) o[h][k] = ffma2(p2, vp[k], o[h][k]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    }

    // merge the row groups of this warp (lanes with equal `sub`)
#pragma unroll
    for (int off = C::LPR; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m[h], off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l[h], off);
        const float mn = fmaxf(m[h], m2);
        const float m_use = (mn == -INFINITY) ? 0.f : mn;
        const float a1 = ex2(m[h] - m_use);
        const float a2 = ex2(m2 - m_use);
        l[h] = l[h] * a1 + l2 * a2;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const float2 mine = unpair(o[h][k]);
          const float ox = __shfl_xor_sync(0xffffffffu, mine.x, off);
          const float oy = __shfl_xor_sync(0xffffffffu, mine.y, off);
          o[h][k] = pair_f32(mine.x * a1 + ox * a2, mine.y * a1 + oy * a2);
        }
        m[h] = mn;
      }
    }
  }

  __syncthreads();  // every stage consumed: the ring becomes merge scratch
  const bool aborted = *abort_flag != 0;
  float* sm_m = reinterpret_cast<float*>(smem);          // [warps][G]
  float* sm_l = sm_m + kDecWarps * G;                    // [warps][G]
  float* sm_o = sm_l + kDecWarps * G;                    // [warps][G][D]
  if (warp < kDecWarps && lane < C::LPR) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (lane == 0) {
        sm_m[warp * G + h] = m[h];
        sm_l[warp * G + h] = l[h];
      }
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 v2 = unpair(o[h][ch * 4 + k]);
          float* dst = sm_o + (warp * G + h) * D + (sub + 8 * ch) * 8 + 2 * k;
          dst[0] = v2.x;
          dst[1] = v2.y;
        }
    }
  }
  __syncthreads();
  if (aborted) return;
  for (int idx = tid; idx < G * D; idx += kDecThreads) {
    const int h = idx / D;
    const int d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm_m[w * G + h]);
    float Lsum = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = ex2(sm_m[w * G + h] - M);
        Lsum = fmaf(sm_l[w * G + h], f, Lsum);
        O = fmaf(sm_o[(w * G + h) * D + d], f, O);
      }
    }
    const size_t slot = (static_cast<size_t>(b) * a.Hq + h0 + h) * a.max_chunks + c;
    a.part_o[slot * D + d] = (M != -INFINITY) ? O / Lsum : 0.f;
    if (d == 0) a.part_lse[slot] = (M != -INFINITY) ? M + log2f(Lsum) : -INFINITY;
  }
}

struct MergeArgs {
  const float* part_o;
  const float* part_lse;
  const int* lens;
  __nv_bfloat16* out;
  float* lse;
  int Hq, chunk, max_chunks;
};

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const MergeArgs a) {
  constexpr int EPL = D / 32;  // output elements per lane
  constexpr int NW = kMergeThreads / 32;
  __shared__ float red[NW];
  __shared__ float sm_w[NW];
  __shared__ float sm_o[NW][D];
  const int bh = blockIdx.x;
  const int b = bh / a.Hq;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = a.lens[b];
  const int nsp = L > 0 ? (L + a.chunk - 1) / a.chunk : 0;
  const float* pl = a.part_lse + static_cast<size_t>(bh) * a.max_chunks;
  const float* po = a.part_o + static_cast<size_t>(bh) * a.max_chunks * D;

  // 1) M = max over chunks of lse_c
  float M = -INFINITY;
  for (int c = tid; c < nsp; c += kMergeThreads) M = fmaxf(M, pl[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) M = fmaxf(M, red[w]);

  // 2) each warp sums w_c * o_c over its chunks
  float W = 0.f, O[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) O[e] = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int c = warp; c < nsp; c += NW) {
      const float w = ex2(pl[c] - M);  // empty chunk: lse -inf -> 0
      const float* src = po + static_cast<size_t>(c) * D + lane * EPL;
      if constexpr (EPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        O[0] = fmaf(w, v.x, O[0]);
        O[1] = fmaf(w, v.y, O[1]);
        O[2] = fmaf(w, v.z, O[2]);
        O[3] = fmaf(w, v.w, O[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        O[0] = fmaf(w, v.x, O[0]);
        O[1] = fmaf(w, v.y, O[1]);
      }
      W += w;
    }
  }
  if (lane == 0) sm_w[warp] = W;
#pragma unroll
  for (int e = 0; e < EPL; ++e) sm_o[warp][lane * EPL + e] = O[e];
  __syncthreads();
  if (warp == 0) {
    float Wt = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) Wt += sm_w[w];
    const bool invalid = (M == -INFINITY);
    __nv_bfloat16* dst = a.out + static_cast<size_t>(bh) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) acc += sm_o[w][lane * EPL + e];
      dst[e] = __float2bfloat16_rn(invalid ? 0.f : acc / Wt);
    }
    if (lane == 0 && a.lse != nullptr)
      a.lse[bh] = invalid ? INFINITY : (M + log2f(Wt)) * 0.69314718055994530942f;
  }
}

template <int D, int G>
cudaError_t launch_chunks(const DecodeLaunch& x, const CUtensorMap& mk, const CUtensorMap& mv,
                          const DecodeArgs& da, cudaStream_t stream) {
  static bool configured = false;  // benign race: idempotent attribute set
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_chunk_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDecSmemBytes + 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(x.num_items, x.Hkv * da.head_groups);
  decode_chunk_kernel<D, G><<<grid, kDecThreads, kDecSmemBytes + 1024, stream>>>(mk, mv, da);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_chunks_g(int G, const DecodeLaunch& x, const CUtensorMap& mk,
                            const CUtensorMap& mv, const DecodeArgs& da, cudaStream_t s) {
  switch (G) {
    case 8:
      if constexpr (D == 64) return launch_chunks<D, 8>(x, mk, mv, da, s);
      return cudaErrorInvalidValue;
    case 4: return launch_chunks<D, 4>(x, mk, mv, da, s);
    case 2: return launch_chunks<D, 2>(x, mk, mv, da, s);
    default: return launch_chunks<D, 1>(x, mk, mv, da, s);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& x, cudaStream_t stream) {
  const int g_total = x.Hq / x.Hkv;
  const int G = decode_heads_per_cta(g_total, x.D);
  if (x.num_items > 0) {
    CUtensorMap mk, mv;
    const int R = (x.D == 128) ? DecCfg<128>::R : DecCfg<64>::R;
    if (!encode_bf16_map(&mk, x.k, x.layout, x.B, x.Hkv, x.S_kv, x.D, x.D, R,
                         CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_bf16_map(&mv, x.v, x.layout, x.B, x.Hkv, x.S_kv, x.D, x.D, R,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    DecodeArgs da;
    da.q = static_cast<const __nv_bfloat16*>(x.q);
    da.key_mask = x.key_mask;
    da.lens = x.lens_dev;
    da.items = x.items_dev;
    da.part_o = x.part_o;
    da.part_lse = x.part_lse;
    da.status = x.status;
    da.timeout_ns = x.timeout_ns;
    da.Hq = x.Hq;
    da.Hkv = x.Hkv;
    da.S_kv = x.S_kv;
    da.chunk = x.chunk;
    da.max_chunks = x.max_chunks;
    da.head_groups = g_total / G;
    da.scale_log2 = x.scale * 1.4426950408889634f;
    main_kernel_begin(stream);
    cudaError_t e = (x.D == 128) ? launch_chunks_g<128>(G, x, mk, mv, da, stream)
                                 : launch_chunks_g<64>(G, x, mk, mv, da, stream);
    main_kernel_end(stream);
    if (e != cudaSuccess) return e;
    count_launches(1);
  }
  MergeArgs ma;
  ma.part_o = x.part_o;
  ma.part_lse = x.part_lse;
  ma.lens = x.lens_dev;
  ma.out = static_cast<__nv_bfloat16*>(x.out);
  ma.lse = x.lse;
  ma.Hq = x.Hq;
  ma.chunk = x.chunk;
  ma.max_chunks = x.max_chunks;
  if (x.D == 128)
    decode_merge_kernel<128><<<x.B * x.Hq, kMergeThreads, 0, stream>>>(ma);
  else
    decode_merge_kernel<64><<<x.B * x.Hq, kMergeThreads, 0, stream>>>(ma);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace fa
