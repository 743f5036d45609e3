// K1a: per-head Gemma-style q-norm + partial neox rope of the packed indexQk rows
// ("Qsa Indexer Kernels", launchQsaIndexQPrep).
//
// HBM-bound stream: a valid row reads its 1024-byte q part and writes 1024 bytes of
// qNormed; a padding row (t >= contextLengths[b]) only writes 1024 zero bytes and
// is never read.  (Large launches go to the staged q mode of k1_stream.cu instead.)
// One warp owns one row: 8-lane group h owns head h, each lane two 16-byte chunks
// (its rope pairs stay in-lane, see qsa_common.cuh).  A persistent grid-stride loop
// keeps ROWS rows of loads in flight per warp before any math; a launch that fits one
// wave issues them before the CTA stages its gamma.
#include "qsa_common.cuh"
#include "qsa_launch.h"

namespace qsa {

#ifndef QSA_K1A_ROWS
#define QSA_K1A_ROWS 2
#endif
#ifndef QSA_K1A_MINB
#define QSA_K1A_MINB 3
#endif

// ONE_WAVE: the grid holds a warp for every ROWS rows, so each warp takes one group and
// issues its loads before the CTA stages its gamma (the two round trips overlap); else a
// persistent grid strides over the groups after the gamma stage.
template <class T, int ROWS, bool ONE_WAVE>
__global__ void __launch_bounds__(256, QSA_K1A_MINB)
k1a_qprep_kernel(uint16_t* __restrict__ q_normed, const uint16_t* __restrict__ index_qk,
                 const float* __restrict__ cos_sin, const int32_t* __restrict__ context_lengths,
                 const uint16_t* __restrict__ w_q, float eps, int32_t batch, int32_t seq_len) {
  const int lane = threadIdx.x & 31;
  const int h = lane >> 3;
  const int j = lane & 7;
  const int ca = chunk_a(j);
  const int cb = chunk_b(j);
  __shared__ __align__(16) float g1[kHeadDim];
  if constexpr (!ONE_WAVE) {
    stage_gamma<T>(w_q, g1);
    __syncthreads();
  }

  const int32_t rows = batch * seq_len;
  const int32_t warp = static_cast<int32_t>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int32_t nwarps = static_cast<int32_t>((gridDim.x * blockDim.x) >> 5);

  for (int32_t base = warp * ROWS;; base += nwarps * ROWS) {
    if (!ONE_WAVE && base >= rows) break;
    uint4 va[ROWS], vb[ROWS];
    RopeCS cs[ROWS] = {};
    bool valid[ROWS];
#pragma unroll
    for (int k = 0; k < ROWS; ++k) {
      const int32_t row = base + k;
      valid[k] = false;
      if (row < rows) {
        const int32_t b = row / seq_len;
        const int32_t t = row - b * seq_len;
        valid[k] = t < __ldg(context_lengths + b);
        if (valid[k]) {
          const uint16_t* src = index_qk + static_cast<int64_t>(row) * kRowWidth + h * kHeadDim;
          va[k] = ld_stream_v4(src + ca);
          vb[k] = ld_stream_v4(src + cb);
          if (j < 4) cs[k] = load_rope(cos_sin + static_cast<int64_t>(t) * kCsWidth, j);
        }
      }
    }
    if constexpr (ONE_WAVE) {  // every warp of the CTA gets here once
      stage_gamma<T>(w_q, g1);
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < ROWS; ++k) {
      const int32_t row = base + k;
      if (row >= rows) break;  // warp-uniform
      uint16_t* dst = q_normed + static_cast<int64_t>(row) * (kNumQHeads * kHeadDim) + h * kHeadDim;
      uint4 oa = make_uint4(0u, 0u, 0u, 0u);
      uint4 ob = make_uint4(0u, 0u, 0u, 0u);
      if (valid[k]) {  // warp-uniform: one row per warp
        float a[8], bv[8];
        unpack8<T>(va[k], a);
        unpack8<T>(vb[k], bv);
        norm_rope_group<T>(a, bv, g1, eps, cs[k], j, oa, ob);
      }
      st_v4(dst + ca, oa);
      st_v4(dst + cb, ob);
    }
    if (ONE_WAVE) break;
  }
}

namespace {
constexpr int kK1aRows = QSA_K1A_ROWS;
constexpr int kK1aThreads = 256;

template <class T>
cudaError_t launch_t(const LaunchQPrep& a) {
  const int64_t rows = static_cast<int64_t>(a.batch) * a.seq_len;
  const int64_t warps_needed = (rows + kK1aRows - 1) / kK1aRows;
  const int64_t blocks_needed = (warps_needed * 32 + kK1aThreads - 1) / kK1aThreads;
  int per_sm = 0;
  cudaError_t e = occupancy_blocks_per_sm(reinterpret_cast<const void*>(k1a_qprep_kernel<T, kK1aRows, false>),
                                          kK1aThreads, 0, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t cap = static_cast<int64_t>(per_sm) * a.num_sms;
  const bool one_wave = blocks_needed <= cap;
  auto kern = one_wave ? k1a_qprep_kernel<T, kK1aRows, true> : k1a_qprep_kernel<T, kK1aRows, false>;
  const int grid = static_cast<int>(one_wave ? blocks_needed : cap);
  kern<<<grid, kK1aThreads, 0, a.stream>>>(
      static_cast<uint16_t*>(a.q_normed), static_cast<const uint16_t*>(a.index_qk), a.cos_sin,
      a.context_lengths, static_cast<const uint16_t*>(a.w_q), a.eps, a.batch, a.seq_len);
  return cudaGetLastError();
}
}  // namespace

// Launches of at least this many rows (batch x seqLen) run through the staged q mode of
// k1_stream.cu (16-row units, each row's q part bulk-copied into shared memory): from 2^17
// rows it streams faster (B=8, S=16384: 5.21 against 5.03 TB/s; 92 against 85 % of the
// copy bandwidth at 2^22 rows), below it this kernel does (1x32768: 17.8 against 19.0 us).
// Both give the same bits: the same norm_rope_group.
#ifndef QSA_K1A_STAGED_MIN_ROWS
#define QSA_K1A_STAGED_MIN_ROWS 131072
#endif

cudaError_t launch_q_prep(const LaunchQPrep& a) {
  if (static_cast<int64_t>(a.batch) * a.seq_len >= QSA_K1A_STAGED_MIN_ROWS) return launch_q_prep_staged(a);
  return a.bf16 ? launch_t<Bf16>(a) : launch_t<F16>(a);
}

}  // namespace qsa
