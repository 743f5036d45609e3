// A plain CUDA-core version of K2 ("Qsa Indexer Kernels", launchQsaIndexScores),
// exported only through the testing header.  It exists so that tests can compare
// the tcgen05 kernel against a second, independent device implementation at sizes
// the CPU oracle cannot finish (every one of 537M logits at B=8, S=16384).  It is
// never used by the product entry points.
//
// One CTA per (row, 128 blocks); the row's 4 x 128 q values are staged as FP32 in
// shared memory; thread g forms the four dot products in ascending d with FP32 FMA.
#include <cfloat>

#include "qsa_common.cuh"
#include "qsa_launch.h"

namespace qsa {

template <class T>
__global__ void __launch_bounds__(128)
k2_scores_cc_kernel(float* __restrict__ logits, const uint16_t* __restrict__ q_normed,
                    const uint16_t* __restrict__ kbar, const int32_t* __restrict__ context_lengths,
                    int32_t seq_len, int32_t num_blocks, int32_t row_start, float scale) {
  __shared__ float qs[kNumQHeads * kHeadDim];
  const int64_t r = static_cast<int64_t>(row_start) + blockIdx.x;
  const int32_t b = static_cast<int32_t>(r / seq_len);
  const int32_t t = static_cast<int32_t>(r - static_cast<int64_t>(b) * seq_len);
  const int32_t ctx = __ldg(context_lengths + b);
  const int32_t g = blockIdx.y * 128 + threadIdx.x;
  float* out = logits + static_cast<int64_t>(blockIdx.x) * num_blocks;
  if (ctx <= 0 || t >= ctx) {
    if (g < num_blocks) out[g] = -FLT_MAX;
    return;
  }
  const uint16_t* q = q_normed + r * (kNumQHeads * kHeadDim);
  for (int i = threadIdx.x; i < kNumQHeads * kHeadDim / 2; i += blockDim.x) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(q)[i];
    qs[2 * i] = T::lo(w);
    qs[2 * i + 1] = T::hi(w);
  }
  __syncthreads();
  if (g >= num_blocks) return;
  if (g >= (t + 1) / kRatio) {
    out[g] = -FLT_MAX;
    return;
  }
  const uint16_t* k = kbar + (static_cast<int64_t>(b) * num_blocks + g) * kHeadDim;
  float kf[kHeadDim];
#pragma unroll
  for (int c = 0; c < kHeadDim / 8; ++c) {
    float f[8];
    unpack8<T>(ld_cached_v4(k + 8 * c), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) kf[8 * c + e] = f[e];
  }
  float sum = 0.0f;
#pragma unroll
  for (int h = 0; h < kNumQHeads; ++h) {
    float dot = 0.0f;
#pragma unroll
    for (int d = 0; d < kHeadDim; ++d) dot = fmaf(qs[h * kHeadDim + d], kf[d], dot);
    sum = __fadd_rn(sum, fmaxf(0.0f, dot));
  }
  out[g] = __fmul_rn(sum, scale);
}

cudaError_t launch_scores_cc(const LaunchScores& a) {
  const dim3 grid(static_cast<unsigned>(a.num_rows), static_cast<unsigned>((a.num_blocks + 127) / 128));
  if (a.bf16) {
    k2_scores_cc_kernel<Bf16><<<grid, 128, 0, a.stream>>>(
        a.logits, static_cast<const uint16_t*>(a.q_normed), static_cast<const uint16_t*>(a.kbar),
        a.context_lengths, a.seq_len, a.num_blocks, a.row_start, a.scale);
  } else {
    k2_scores_cc_kernel<F16><<<grid, 128, 0, a.stream>>>(
        a.logits, static_cast<const uint16_t*>(a.q_normed), static_cast<const uint16_t*>(a.kbar),
        a.context_lengths, a.seq_len, a.num_blocks, a.row_start, a.scale);
  }
  return cudaGetLastError();
}

}  // namespace qsa
