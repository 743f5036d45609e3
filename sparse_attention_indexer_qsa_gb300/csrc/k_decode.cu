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
//   scores_decode  K2 numerics at S = 1 over the V-tails: logits[b][g] for
//                g < ctx/4 only; a block whose page slot is unusable scores -FLT_MAX.
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

// grid (B, ceilDiv(maxBlocks, 256)), one thread per block column
template <class T>
__global__ void __launch_bounds__(256) scores_decode_kernel(float* __restrict__ logits,
                                                            const uint16_t* __restrict__ q_normed,
                                                            const int32_t* __restrict__ ctx, const PoolDev pool,
                                                            int32_t max_blocks, float scale) {
  __shared__ float qs[kNumQHeads * kHeadDim];
  const int32_t b = blockIdx.x;
  const int32_t c = __ldg(ctx + b);
  const int32_t n_vis = c > 0 ? min(c / kRatio, max_blocks) : 0;
  const int32_t g0 = blockIdx.y * blockDim.x;
  if (g0 >= n_vis) return;  // only the valid prefix is written
  const uint16_t* q = q_normed + static_cast<int64_t>(b) * (kNumQHeads * kHeadDim);
  for (int i = threadIdx.x; i < kNumQHeads * kHeadDim / 2; i += blockDim.x) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(q)[i];
    qs[2 * i] = T::lo(w);
    qs[2 * i + 1] = T::hi(w);
  }
  __syncthreads();
  const int32_t g = g0 + threadIdx.x;
  if (g >= n_vis) return;
  float* out = logits + static_cast<int64_t>(b) * max_blocks + g;
  const uint16_t* k = pool_tail(pool, b, 1, kRatio * g);
  if (k == nullptr) {
    *out = -FLT_MAX;
    return;
  }
  float kf[kHeadDim];
#pragma unroll
  for (int ch = 0; ch < kHeadDim / 8; ++ch) {
    float f[8];
    unpack8<T>(ld_cached_v4(k + 8 * ch), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) kf[8 * ch + e] = f[e];
  }
  float sum = 0.0f;
#pragma unroll
  for (int hh = 0; hh < kNumQHeads; ++hh) {
    float dot = 0.0f;
#pragma unroll
    for (int d = 0; d < kHeadDim; ++d) dot = fmaf(qs[hh * kHeadDim + d], kf[d], dot);
    sum = __fadd_rn(sum, fmaxf(0.0f, dot));
  }
  *out = __fmul_rn(sum, scale);
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
  const dim3 grid(static_cast<unsigned>(batch), static_cast<unsigned>((max_blocks + 255) / 256));
  auto* q = static_cast<const uint16_t*>(q_normed);
  if (bf16) dec::scores_decode_kernel<Bf16><<<grid, 256, 0, stream>>>(logits, q, ctx, pool, max_blocks, scale);
  else dec::scores_decode_kernel<F16><<<grid, 256, 0, stream>>>(logits, q, ctx, pool, max_blocks, scale);
  return cudaGetLastError();
}

}  // namespace qsa
