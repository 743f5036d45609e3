// K1b: compress the raw index-K of each complete 4-token block into kbar, then the
// K1a norm (with wK) and rope at position 4g ("Qsa Indexer Kernels",
// launchQsaIndexKCompress, including its (blockBegin, blockEnd, pastLen) sub-range
// contract).
//
// One aligned 8-lane group owns one block (b, g): each lane loads its two 16-byte
// chunks of the four K rows (8 loads in flight per lane; in a one-wave launch before
// the CTA stages its gamma), forms the fixed-order
// FP32 mean ((k0+k1)+k2)+k3 times 0.25, casts it to T and re-loads it, then runs
// the same norm_rope_group as K1a.  The block math reads nothing but (b, g), the
// rows and the tables, so a block's bits never depend on the range or pastLen of
// the launch that computed it.
#include "qsa_common.cuh"
#include "qsa_launch.h"

namespace qsa {

// 128-thread CTAs, 6 an SM: small launches spread over more SMs than with 256-thread
// CTAs (2048 blocks: 128 CTAs instead of 64)
#ifndef QSA_K1B_THREADS
#define QSA_K1B_THREADS 128
#endif
#ifndef QSA_K1B_MINB
#define QSA_K1B_MINB (768 / QSA_K1B_THREADS)
#endif

// PAGED (launchQsaIndexKCompressPaged): additionally copy every VALID block's kbar
// row to the pool V-tail of token 4g when that page slot is usable; the dense
// output is the same code path, so it is bit-identical to the unpaged kernel.
// ONE_WAVE: the grid holds a warp for every unit group, so each warp takes one group and
// issues its loads before the CTA stages its gamma (the two round trips overlap); else a
// persistent grid strides over the groups after the gamma stage.
template <class T, bool PAGED, bool ONE_WAVE>
__global__ void __launch_bounds__(QSA_K1B_THREADS, QSA_K1B_MINB)
k1b_compress_kernel(uint16_t* __restrict__ kbar, const uint16_t* __restrict__ index_qk,
                    const float* __restrict__ cos_sin, const int32_t* __restrict__ context_lengths,
                    const uint16_t* __restrict__ w_k, float eps, int32_t batch, int32_t seq_len,
                    int32_t num_blocks, int32_t block_begin, int32_t block_end, int32_t past_len,
                    const PoolDev pool) {
  const int lane = threadIdx.x & 31;
  const int j = lane & 7;
  const int ca = chunk_a(j);
  const int cb = chunk_b(j);
  __shared__ __align__(16) float g1[kHeadDim];
  if constexpr (!ONE_WAVE) {
    stage_gamma<T>(w_k, g1);
    __syncthreads();
  }

  const int32_t nb = block_end - block_begin;
  const int64_t units = static_cast<int64_t>(batch) * nb;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

  // Warp-uniform trip count: all 32 lanes reach the shuffles in norm_rope_group.
  for (int64_t base = warp * 4;; base += nwarps * 4) {
    if (!ONE_WAVE && base >= units) break;
    const int64_t u = base + (lane >> 3);
    const bool active = u < units;
    bool valid = false;
    int32_t b = 0, g = 0;
    if (active) {
      b = static_cast<int32_t>(u / nb);
      g = block_begin + static_cast<int32_t>(u - static_cast<int64_t>(b) * nb);
      const int64_t first = static_cast<int64_t>(kRatio) * g;
      const int64_t last = first + (kRatio - 1);
      valid = last < __ldg(context_lengths + b) && first >= past_len && last - past_len < seq_len;
    }
    float a[8], bv[8];
    RopeCS cs{};
    uint4 ka[kRatio], kb[kRatio];
    if (valid) {
      const uint16_t* src = index_qk +
          (static_cast<int64_t>(b) * seq_len + (static_cast<int64_t>(kRatio) * g - past_len)) * kRowWidth + kKCol;
#pragma unroll
      for (int r = 0; r < kRatio; ++r) {
        ka[r] = ld_stream_v4(src + r * kRowWidth + ca);
        kb[r] = ld_stream_v4(src + r * kRowWidth + cb);
      }
      if (j < 4) cs = load_rope(cos_sin + static_cast<int64_t>(kRatio) * g * kCsWidth, j);
    }
    if constexpr (ONE_WAVE) {  // every warp of the CTA gets here once
      stage_gamma<T>(w_k, g1);
      __syncthreads();
      if (base >= units) break;  // warp-uniform
    }
    if (valid) {
      float fa[kRatio][8], fb[kRatio][8];
#pragma unroll
      for (int r = 0; r < kRatio; ++r) {
        unpack8<T>(ka[r], fa[r]);
        unpack8<T>(kb[r], fb[r]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        // fixed order, each step rounded; x0.25 is exact; bit-critical cast + re-load
        float s = __fadd_rn(__fadd_rn(__fadd_rn(fa[0][e], fa[1][e]), fa[2][e]), fa[3][e]);
        a[e] = T::round_trip(__fmul_rn(s, 0.25f));
        s = __fadd_rn(__fadd_rn(__fadd_rn(fb[0][e], fb[1][e]), fb[2][e]), fb[3][e]);
        bv[e] = T::round_trip(__fmul_rn(s, 0.25f));
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) { a[e] = 0.0f; bv[e] = 0.0f; }
    }
    uint4 oa, ob;
    norm_rope_group<T>(a, bv, g1, eps, cs, j, oa, ob);
    if (active) {
      if (!valid) { oa = make_uint4(0u, 0u, 0u, 0u); ob = oa; }
      uint16_t* dst = kbar + (static_cast<int64_t>(b) * num_blocks + g) * kHeadDim;
      st_v4(dst + ca, oa);
      st_v4(dst + cb, ob);
      if (PAGED && valid) {
        uint16_t* tail = pool_tail(pool, b, 1, kRatio * g);
        if (tail != nullptr) {
          st_v4(tail + ca, oa);
          st_v4(tail + cb, ob);
        }
      }
    }
    if (ONE_WAVE) break;
  }
}

namespace {
constexpr int kK1bThreads = QSA_K1B_THREADS;

template <class T, bool PAGED>
cudaError_t launch_t(const LaunchKCompress& a, const PoolDev& pool) {
  const int64_t units = static_cast<int64_t>(a.batch) * (a.block_end - a.block_begin);
  const int64_t blocks_needed = (units * 8 + kK1bThreads - 1) / kK1bThreads;
  int per_sm = 0;
  cudaError_t e = occupancy_blocks_per_sm(reinterpret_cast<const void*>(k1b_compress_kernel<T, PAGED, false>),
                                          kK1bThreads, 0, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t cap = static_cast<int64_t>(per_sm) * a.num_sms;
  const bool one_wave = blocks_needed <= cap;
  auto kern = one_wave ? k1b_compress_kernel<T, PAGED, true> : k1b_compress_kernel<T, PAGED, false>;
  const int grid = static_cast<int>(one_wave ? blocks_needed : cap);
  kern<<<grid, kK1bThreads, 0, a.stream>>>(
      static_cast<uint16_t*>(a.kbar), static_cast<const uint16_t*>(a.index_qk), a.cos_sin,
      a.context_lengths, static_cast<const uint16_t*>(a.w_k), a.eps, a.batch, a.seq_len,
      a.num_blocks, a.block_begin, a.block_end, a.past_len, pool);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_k_compress(const LaunchKCompress& a) {
  const PoolDev none{};
  return a.bf16 ? launch_t<Bf16, false>(a, none) : launch_t<F16, false>(a, none);
}

cudaError_t launch_k_compress_paged(const LaunchKCompressPaged& a) {
  return a.base.bf16 ? launch_t<Bf16, true>(a.base, a.pool) : launch_t<F16, true>(a.base, a.pool);
}

}  // namespace qsa
