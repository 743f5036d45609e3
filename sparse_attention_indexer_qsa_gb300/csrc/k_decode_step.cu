// The whole decode step in one launch ("Qsa Indexer Kernels": launchQsaIndexerPreDecode,
// launchQsaIndexScoresDecode and launchQsaTopKExpandDecode, in that order, fused).
//
// grid (B, Y), kDecThreads threads; CTA (b, y) covers blocks [y * perCta, (y + 1) * perCta),
// perCta a multiple of kDecBlocksPerCta chosen so that the grid is about one wave.  CTA (b, y):
//   - warp 0 computes sequence b's q heads into shared memory (CTA y = 0 also writes
//     qNormed[b]); warp 1 either writes the new token's raw K-tail (CTA y = 0), or, in
//     the CTA whose blocks include the just-completed block g, compresses g (the
//     pre-decode routines) into shared memory and the pool's V-tail;
//   - the CTA scores its blocks of the valid prefix, kDecBlocksPerCta at a time (the
//     paged-scores routine; block g is read from shared memory), into logits[b];
//   - the last CTA of sequence b to finish (a per-sequence arrival counter, no waiting)
//     runs the top-512 selection of row b on the logits at L2, writes outIdx[b], zeroes
//     b's split counters and puts the counter back to zero.
// Every value equals the one the three separate kernels give: the same device routines
// compute it.  Arrival counters: kStepSlots sets of kStepMaxBatch, one set a launch in
// turn (so up to kStepSlots launches may run at once on a device), zero at module load
// and left at zero by every launch.
#include <algorithm>
#include <mutex>

#include "qsa_decode.cuh"
#include "qsa_select.cuh"

namespace qsa {

constexpr int kStepSlots = 16;
constexpr int kStepMaxBatch = 4096;
constexpr int kStepCtasPerSm = 3;  // the resident CTAs of decode_step_kernel an SM is sized for
__device__ __align__(256) uint32_t g_decode_step_arrivals[kStepSlots * kStepMaxBatch];

namespace dec {

template <class T, int MW>
__global__ void __launch_bounds__(kDecThreads, kStepCtasPerSm)
decode_step_kernel(int32_t* __restrict__ out_idx, float* __restrict__ logits, uint16_t* __restrict__ q_normed,
                   const uint16_t* __restrict__ index_qk, const float* __restrict__ cos_sin,
                   const int32_t* __restrict__ ctx, const uint16_t* __restrict__ w_q,
                   const uint16_t* __restrict__ w_k, float eps, const PoolDev pool,
                   int32_t* __restrict__ split_counters, int32_t num_kv_heads, int32_t max_blocks, float scale,
                   int32_t per_cta, uint32_t* __restrict__ arrivals) {
  __shared__ __align__(16) float g1q[kHeadDim];
  __shared__ __align__(16) float g1k[kHeadDim];
  __shared__ __align__(16) uint16_t q4[kNumQHeads * kHeadDim];
  __shared__ __align__(16) uint16_t kbar_new[kHeadDim];
  __shared__ __align__(16) sel::SelShared<kDecThreads> sh;
  __shared__ int32_t own_block;  // block scored from kbar_new, or -1
  __shared__ int32_t last;
  const int32_t b = blockIdx.x, y = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t c = __ldg(ctx + b);
  const int32_t n_vis = c > 0 ? min(c / kRatio, max_blocks) : 0;
  const int32_t g_begin = y * per_cta;
  const int32_t g_end = min(g_begin + per_cta, n_vis);
  stage_gamma<T>(w_q, g1q);
  stage_gamma<T>(w_k, g1k);
  if (tid == 0) own_block = -1;
  __syncthreads();
  const uint16_t* row = index_qk + static_cast<int64_t>(b) * kRowWidth;
  const int h = lane >> 3, j = lane & 7;
  const int ca = chunk_a(j), cb = chunk_b(j);
  if (warp == 0) {
    uint4 oa, ob;
    q_heads<T>(row, cos_sin, c, g1q, eps, lane, oa, ob);
    *reinterpret_cast<uint4*>(q4 + h * kHeadDim + ca) = oa;
    *reinterpret_cast<uint4*>(q4 + h * kHeadDim + cb) = ob;
    if (y == 0) {
      uint16_t* dst = q_normed + static_cast<int64_t>(b) * (kNumQHeads * kHeadDim) + h * kHeadDim;
      st_v4(dst + ca, oa);
      st_v4(dst + cb, ob);
    }
  } else if (warp == 1 && c > 0) {
    if (c % kRatio != 0) {
      if (y == 0) {
        uint16_t* dst = pool_tail(pool, b, 0, c - 1);
        if (dst != nullptr) copy_tail(dst, row + kKCol, lane);
      }
    } else if ((c / kRatio - 1) / per_cta == y) {
      uint4 oa, ob;
      uint16_t* vtail = nullptr;
      const bool ok = compress_block<T>(pool, b, c, row, cos_sin, g1k, eps, lane, oa, ob, &vtail);
      if (ok && h == 0) {
        st_v4(vtail + ca, oa);
        st_v4(vtail + cb, ob);
        *reinterpret_cast<uint4*>(kbar_new + ca) = oa;
        *reinterpret_cast<uint4*>(kbar_new + cb) = ob;
      }
      if (ok && lane == 0) own_block = c / kRatio - 1;
    }
  }
  __syncthreads();
  float* lrow = logits + static_cast<int64_t>(b) * max_blocks;
  if (g_begin < g_end) {
    float qf[kNumQHeads][8];
#pragma unroll
    for (int h = 0; h < kNumQHeads; ++h)  // shared memory: a plain (generic) load
      unpack8<T>(*reinterpret_cast<const uint4*>(q4 + h * kHeadDim + 8 * (tid & 15)), qf[h]);
    for (int32_t g0 = g_begin; g0 < g_end; g0 += kDecBlocksPerCta)
      score_range<T>(lrow, qf, pool, b, g0, min(g0 + kDecBlocksPerCta, g_end), scale, own_block, kbar_new);
  }

  // ---- the last CTA of sequence b selects its row
  __syncthreads();
  if (tid == 0) {
    __threadfence();  // this CTA's logits, before its arrival
    last = atomicAdd(arrivals + b, 1u) == gridDim.y - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();  // every CTA's logits of row b, before they are read
  if (tid == 0) arrivals[b] = 0u;
  if (split_counters != nullptr)
    for (int k = tid; k < num_kv_heads; k += kDecThreads) split_counters[static_cast<int64_t>(b) * num_kv_heads + k] = 0;
  int32_t* out = out_idx + static_cast<int64_t>(b) * sel::kWidth;
  const int32_t tail = c > 0 ? c % kRatio : 0;
  if (n_vis <= sel::kTopK) {
    sel::write_unselected<kDecThreads>(out, c <= 0, n_vis, tail);
    return;
  }
  const sel::L2Keys keys{lrow, (reinterpret_cast<uintptr_t>(lrow) & 15u) == 0};
  sel::select_row<kDecThreads, MW>(keys, n_vis, sh);
  sel::write_selected<kDecThreads>(out, sh.win, tail, n_vis);
}

}  // namespace dec

namespace {
std::mutex g_step_mu;
uint32_t* g_step_base[64] = {};
uint32_t g_step_seq[64] = {};
}  // namespace

int32_t decode_step_max_batch() { return kStepMaxBatch; }

cudaError_t launch_decode_step(bool bf16, int32_t* out_idx, float* logits, void* q_normed, const void* index_qk,
                               const float* cos_sin, const int32_t* ctx, const void* w_q, const void* w_k,
                               float eps, const PoolDev& pool, int32_t* split_counters, int32_t num_kv_heads,
                               int32_t batch, int32_t max_blocks, float scale, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  uint32_t* arrivals = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_step_mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_step_base[dev] == nullptr) {  // the symbol's device address, once per device
      void* ptr = nullptr;
      if ((e = cudaGetSymbolAddress(&ptr, g_decode_step_arrivals)) != cudaSuccess) return e;
      g_step_base[dev] = static_cast<uint32_t*>(ptr);
    }
    arrivals = g_step_base[dev] + static_cast<int64_t>(g_step_seq[dev]++ % kStepSlots) * kStepMaxBatch;
  }
  // Y CTAs a sequence, each over per_cta (a multiple of kDecBlocksPerCta) blocks: about one
  // wave of resident CTAs over the batch, so that each CTA computes the q heads once
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int32_t chunks = (max_blocks + dec::kDecBlocksPerCta - 1) / dec::kDecBlocksPerCta;
  const int32_t want_y = std::max<int32_t>(1, sms * kStepCtasPerSm / std::max<int32_t>(batch, 1));
  const int32_t per_chunks = (chunks + want_y - 1) / want_y;
  const int32_t per_cta = std::max<int32_t>(1, per_chunks) * dec::kDecBlocksPerCta;
  const dim3 grid(static_cast<unsigned>(batch), static_cast<unsigned>((max_blocks + per_cta - 1) / per_cta));
  const int32_t words = (max_blocks + dec::kDecThreads * 32 - 1) / (dec::kDecThreads * 32);
  auto* q = static_cast<uint16_t*>(q_normed);
  auto* iq = static_cast<const uint16_t*>(index_qk);
  auto* wq = static_cast<const uint16_t*>(w_q);
  auto* wk = static_cast<const uint16_t*>(w_k);
#define QSA_STEP_LAUNCH(T, MW)                                                                             \
  dec::decode_step_kernel<T, MW><<<grid, dec::kDecThreads, 0, stream>>>(                                   \
      out_idx, logits, q, iq, cos_sin, ctx, wq, wk, eps, pool, split_counters, num_kv_heads, max_blocks, scale, \
      per_cta, arrivals)
#define QSA_STEP_DISPATCH(T)                 \
  do {                                       \
    if (words <= 1) QSA_STEP_LAUNCH(T, 1);   \
    else if (words <= 2) QSA_STEP_LAUNCH(T, 2); \
    else if (words <= 4) QSA_STEP_LAUNCH(T, 4); \
    else QSA_STEP_LAUNCH(T, 8);              \
  } while (0)
  if (bf16) QSA_STEP_DISPATCH(Bf16);
  else QSA_STEP_DISPATCH(F16);
#undef QSA_STEP_DISPATCH
#undef QSA_STEP_LAUNCH
  return cudaGetLastError();
}

}  // namespace qsa
