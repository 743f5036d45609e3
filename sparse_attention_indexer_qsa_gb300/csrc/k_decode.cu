// Decode path and prefill tail persistence over the paged indexer pool
// ("Qsa Indexer Kernels": launchQsaRawKTailWritePrefill, launchQsaIndexerPreDecode,
// launchQsaIndexScoresDecode).  Pool addressing and page-table guards: pool_tail()
// in qsa_launch.h.
//
//   raw_k_tail   tokens t in [ctx - ctx % 4, ctx) copy their raw index-K (indexQk
//                columns [512, 640)) bit for bit to their K-tails.
//   pre_decode   one new token per sequence (pos = ctx - 1): K1a at position pos;
//                then either its raw index-K goes to its K-tail (ctx % 4 != 0), or
//                the just-completed block g = ctx/4 - 1 is compressed from the three
//                K-tails of 4g..4g+2 plus the new row (K1b numerics: the same device
//                routines as the prefill kernels, so the kbar is bit-identical to
//                prefill K1b) and written to the V-tail of 4g.
//   scores_decode  K2's scoring at S = 1 over the V-tails: logits[b][g] for
//                g < ctx/4 only; a block whose page slot is unusable scores -FLT_MAX.
//                FP32 dot products in another order than K2's (eight-term partial
//                dots per lane, then a lane tree), so equal to K2 within the logits
//                tolerance, not bit for bit; relu, the ascending head sum and the
//                scale as in K2.
#include <cfloat>

#include "qsa_common.cuh"
#include "qsa_launch.h"

namespace qsa {
namespace dec {

__device__ __forceinline__ void copy_tail(uint16_t* dst, const uint16_t* src, int lane) {
  if (lane < 16) st_v4(dst + 8 * lane, ld_stream_v4(src + 8 * lane));  // 256 bytes, 16 B per lane
}

// grid (B), 3 warps: warp j handles the j-th token of the open block
__global__ void raw_k_tail_kernel(const uint16_t* __restrict__ index_qk, const int32_t* __restrict__ ctx,
                                  const PoolDev pool, int32_t seq_len) {
  const int32_t b = blockIdx.x;
  const int j = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t c = __ldg(ctx + b);
  if (c <= 0 || j >= c % kRatio) return;
  const int32_t t = c - c % kRatio + j;
  if (t >= seq_len) return;
  uint16_t* dst = pool_tail(pool, b, 0, t);
  if (dst == nullptr) return;
  copy_tail(dst, index_qk + (static_cast<int64_t>(b) * seq_len + t) * kRowWidth + kKCol, lane);
}

// grid (B), 2 warps: warp 0 the q-prep, warp 1 the K-tail write or block compress
template <class T>
__global__ void __launch_bounds__(64) pre_decode_kernel(uint16_t* __restrict__ q_normed,
                                                        const uint16_t* __restrict__ index_qk,
                                                        const float* __restrict__ cos_sin,
                                                        const int32_t* __restrict__ ctx,
                                                        const uint16_t* __restrict__ w_q,
                                                        const uint16_t* __restrict__ w_k, float eps,
                                                        const PoolDev pool) {
  __shared__ __align__(16) float g1q[kHeadDim];
  __shared__ __align__(16) float g1k[kHeadDim];
  stage_gamma<T>(w_q, g1q);
  stage_gamma<T>(w_k, g1k);
  __syncthreads();
  const int32_t b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = lane >> 3, j = lane & 7;
  const int ca = chunk_a(j), cb = chunk_b(j);
  const int32_t c = __ldg(ctx + b);
  const uint16_t* row = index_qk + static_cast<int64_t>(b) * kRowWidth;
  if (warp == 0) {
    uint16_t* dst = q_normed + static_cast<int64_t>(b) * (kNumQHeads * kHeadDim) + h * kHeadDim;
    uint4 oa = make_uint4(0u, 0u, 0u, 0u), ob = oa;
    if (c > 0) {  // block-uniform
      const int32_t pos = c - 1;
      float a[8], bv[8];
      unpack8<T>(ld_stream_v4(row + h * kHeadDim + ca), a);
      unpack8<T>(ld_stream_v4(row + h * kHeadDim + cb), bv);
      RopeCS cs{};
      if (j < 4) cs = load_rope(cos_sin + static_cast<int64_t>(pos) * kCsWidth, j);
      norm_rope_group<T>(a, bv, g1q, eps, cs, j, oa, ob);
    }
    st_v4(dst + ca, oa);
    st_v4(dst + cb, ob);
    return;
  }
  if (c <= 0) return;
  const int32_t pos = c - 1;
  if (c % kRatio != 0) {
    uint16_t* dst = pool_tail(pool, b, 0, pos);
    if (dst != nullptr) copy_tail(dst, row + kKCol, lane);
    return;
  }
  // block g = c/4 - 1 just completed: three K-tails plus the new row; every lane
  // takes part in the group shuffles, lanes of group 0 hold the block
  const int32_t g = c / kRatio - 1;
  const uint16_t* k0 = pool_tail(pool, b, 0, kRatio * g);
  const uint16_t* k1 = pool_tail(pool, b, 0, kRatio * g + 1);
  const uint16_t* k2 = pool_tail(pool, b, 0, kRatio * g + 2);
  uint16_t* out = pool_tail(pool, b, 1, kRatio * g);
  const bool ok = k0 != nullptr && k1 != nullptr && k2 != nullptr && out != nullptr;  // block-uniform
  float a[8], bv[8];
  RopeCS cs{};
  if (ok) {
    const uint16_t* src[kRatio] = {k0, k1, k2, row + kKCol};
    float fa[kRatio][8], fb[kRatio][8];
#pragma unroll
    for (int q = 0; q < kRatio; ++q) {
      unpack8<T>(ld_cached_v4(src[q] + ca), fa[q]);
      unpack8<T>(ld_cached_v4(src[q] + cb), fb[q]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float s = __fadd_rn(__fadd_rn(__fadd_rn(fa[0][e], fa[1][e]), fa[2][e]), fa[3][e]);
      a[e] = T::round_trip(__fmul_rn(s, 0.25f));
      s = __fadd_rn(__fadd_rn(__fadd_rn(fb[0][e], fb[1][e]), fb[2][e]), fb[3][e]);
      bv[e] = T::round_trip(__fmul_rn(s, 0.25f));
    }
    if (j < 4) cs = load_rope(cos_sin + static_cast<int64_t>(kRatio) * g * kCsWidth, j);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) { a[e] = 0.0f; bv[e] = 0.0f; }
  }
  uint4 oa, ob;
  norm_rope_group<T>(a, bv, g1k, eps, cs, j, oa, ob);
  if (ok && h == 0) {
    st_v4(out + ca, oa);
    st_v4(out + cb, ob);
  }
}

// grid (B, ceilDiv(maxBlocks, kDecBlocksPerCta)), kDecThreads threads.  A 16-lane
// half-warp scores one block at a time: lane c holds dims [8c, 8c+8) of the 4 q heads
// in registers, reads the matching 16 bytes of the block's V-tail (the half-warp reads
// the 256-byte row in one coalesced access), forms 4 partial dots, and the half-warp
// reduces them (a reduce-scatter over lane bits 3 and 2, then bits 1 and 0), so that
// lanes 0/4/8/12 hold heads 0/1/2/3; lane 0 sums relu of the heads in ascending order.
constexpr int kDecThreads = 256;
constexpr int kDecUnroll = 4;                                       // blocks in flight a half-warp
constexpr int kDecBlocksPerCta = (kDecThreads / 16) * kDecUnroll * 2;  // two rounds

template <class T>
__global__ void __launch_bounds__(kDecThreads) scores_decode_kernel(float* __restrict__ logits,
                                                                    const uint16_t* __restrict__ q_normed,
                                                                    const int32_t* __restrict__ ctx,
                                                                    const PoolDev pool, int32_t max_blocks,
                                                                    float scale) {
  const int32_t b = blockIdx.x;
  const int32_t c = __ldg(ctx + b);
  const int32_t n_vis = c > 0 ? min(c / kRatio, max_blocks) : 0;
  const int32_t g_begin = blockIdx.y * kDecBlocksPerCta;
  if (g_begin >= n_vis) return;  // only the valid prefix is written
  const int32_t g_end = min(g_begin + kDecBlocksPerCta, n_vis);
  const int lane = threadIdx.x & 31, ch = lane & 15, hw = threadIdx.x >> 4;
  const unsigned half = lane & 16;
  float qf[kNumQHeads][8];
  const uint16_t* q = q_normed + static_cast<int64_t>(b) * (kNumQHeads * kHeadDim) + 8 * ch;
#pragma unroll
  for (int h = 0; h < kNumQHeads; ++h) unpack8<T>(ld_cached_v4(q + h * kHeadDim), qf[h]);
  float* out = logits + static_cast<int64_t>(b) * max_blocks;
  const bool keep_hi = (ch & 8) != 0, keep_odd = (ch & 4) != 0;
#pragma unroll 1
  for (int32_t base = g_begin; base < g_end; base += 16 * kDecUnroll) {  // warp-uniform: shuffles below
    const int32_t g0 = base + hw;
    uint4 raw[kDecUnroll];
    bool ok[kDecUnroll];
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int32_t g = g0 + 16 * u;
      const uint16_t* k = g < g_end ? pool_tail(pool, b, 1, kRatio * g) : nullptr;
      ok[u] = k != nullptr;
      raw[u] = ok[u] ? ld_stream_v4(k + 8 * ch) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      float kf[8];
      unpack8<T>(raw[u], kf);
      float d[kNumQHeads];
#pragma unroll
      for (int h = 0; h < kNumQHeads; ++h) {
        float acc = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(qf[h][e], kf[e], acc);
        d[h] = acc;
      }
      // lane bit 3: keep heads {2,3} or {0,1}; send the other pair to the partner
      const float s0 = keep_hi ? d[0] : d[2], s1 = keep_hi ? d[1] : d[3];
      const float r0 = __shfl_xor_sync(0xffffffffu, s0, 8), r1 = __shfl_xor_sync(0xffffffffu, s1, 8);
      const float e0 = (keep_hi ? d[2] : d[0]) + r0, e1 = (keep_hi ? d[3] : d[1]) + r1;
      // lane bit 2: keep the pair's second or first head
      const float r2 = __shfl_xor_sync(0xffffffffu, keep_odd ? e0 : e1, 4);
      float f = (keep_odd ? e1 : e0) + r2;
      f += __shfl_xor_sync(0xffffffffu, f, 2);
      f += __shfl_xor_sync(0xffffffffu, f, 1);
      const float rel = fmaxf(0.0f, f);  // head ((ch >> 3) & 1) * 2 + ((ch >> 2) & 1)
      const float h1 = __shfl_sync(0xffffffffu, rel, half | 4);
      const float h2 = __shfl_sync(0xffffffffu, rel, half | 8);
      const float h3 = __shfl_sync(0xffffffffu, rel, half | 12);
      const int32_t g = g0 + 16 * u;
      if (ch == 0 && g < g_end) out[g] = ok[u] ? __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(rel, h1), h2), h3), scale)
                                              : -FLT_MAX;
    }
  }
}

}  // namespace dec

cudaError_t launch_raw_k_tail_write_prefill(bool bf16, const void* index_qk, const int32_t* ctx, const PoolDev& pool,
                                            int32_t batch, int32_t seq_len, cudaStream_t stream) {
  (void)bf16;  // a bit copy: the element type does not matter
  dec::raw_k_tail_kernel<<<batch, 32 * (kRatio - 1), 0, stream>>>(static_cast<const uint16_t*>(index_qk), ctx,
                                                                  pool, seq_len);
  return cudaGetLastError();
}

cudaError_t launch_pre_decode(bool bf16, void* q_normed, const void* index_qk, const float* cos_sin,
                              const int32_t* ctx, const void* w_q, const void* w_k, float eps, const PoolDev& pool,
                              int32_t batch, cudaStream_t stream) {
  auto* q = static_cast<uint16_t*>(q_normed);
  auto* iq = static_cast<const uint16_t*>(index_qk);
  auto* wq = static_cast<const uint16_t*>(w_q);
  auto* wk = static_cast<const uint16_t*>(w_k);
  if (bf16) dec::pre_decode_kernel<Bf16><<<batch, 64, 0, stream>>>(q, iq, cos_sin, ctx, wq, wk, eps, pool);
  else dec::pre_decode_kernel<F16><<<batch, 64, 0, stream>>>(q, iq, cos_sin, ctx, wq, wk, eps, pool);
  return cudaGetLastError();
}

cudaError_t launch_scores_decode(bool bf16, float* logits, const void* q_normed, const int32_t* ctx,
                                 const PoolDev& pool, int32_t batch, int32_t max_blocks, float scale,
                                 cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(batch),
                  static_cast<unsigned>((max_blocks + dec::kDecBlocksPerCta - 1) / dec::kDecBlocksPerCta));
  auto* q = static_cast<const uint16_t*>(q_normed);
  if (bf16)
    dec::scores_decode_kernel<Bf16><<<grid, dec::kDecThreads, 0, stream>>>(logits, q, ctx, pool, max_blocks, scale);
  else
    dec::scores_decode_kernel<F16><<<grid, dec::kDecThreads, 0, stream>>>(logits, q, ctx, pool, max_blocks, scale);
  return cudaGetLastError();
}

}  // namespace qsa
