// The whole decode step in one launch ("Qsa Indexer Kernels": launchQsaIndexerPreDecode,
// launchQsaIndexScoresDecode and launchQsaTopKExpandDecode, in that order, fused).
//
// grid (B, Y), kDecThreads threads; CTA (b, y) covers the run of blocks [y * perCta,
// (y + 1) * perCta), perCta chosen so that the grid is about one wave.  CTA (b, y):
//   - warp 0 stages the run's page entries (for the whole run, without waiting for the
//     context length) and issues the first tiles' TMA copies at once;
//   - warp 2 computes sequence b's q heads straight into the tensor-core B operand
//     (CTA y = 0 also writes qNormed[b]); warp 3 either writes the new token's raw
//     K-tail (CTA y = 0), or, in the CTA whose run holds the just-completed block g
//     (the last CTA if g lies past maxBlocks), compresses g (the pre-decode
//     routines) into the pool's V-tail.  Both issue their loads before the gamma
//     barrier.  If g's tile is one of the first copied, its copy holds g's stale
//     V-tail row, and warp 3 writes the compressed row into that A stage once the copy
//     has landed; a later tile is copied after the V-tail store and reads it from L2;
//   - the tensor-core paged-scores engine scores the run's blocks of the valid prefix
//     into logits[b];
//   - the last CTA of sequence b to finish (a per-sequence arrival counter, no waiting)
//     runs the top-512 selection of row b on the logits at L2, writes outIdx[b], zeroes
//     b's split counters and puts the counter back to zero.  Its shared memory for the
//     selection reuses the engine's operand stages.  For batches of up to kHistBatch
//     sequences with more than 512 visible blocks, the scoring CTAs also count each
//     logit they write into the row's first-digit histogram, so that the last CTA
//     copies it instead of counting the row again, and zeroes it.
// Every value equals the one the three separate kernels give: the same device routines
// compute it.  Arrival counters and histograms: kStepSlots sets, one set a launch in
// turn (so up to kStepSlots launches may run at once on a device), zero at module load
// and left at zero by every launch.
#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>

#include "qsa_decode.cuh"
#include "qsa_decode_tc.cuh"
#include "qsa_select.cuh"

namespace qsa {

constexpr int kStepSlots = 16;
constexpr int kStepMaxBatch = 4096;
constexpr int kHistBatch = 64;     // batches up to this size count the rows' histograms while scoring
constexpr int kStepCtasPerSm = 2;  // the resident CTAs of decode_step_kernel an SM is sized for
__device__ __align__(256) uint32_t g_decode_step_arrivals[kStepSlots * kStepMaxBatch];
__device__ __align__(256) uint32_t g_decode_step_hist[kStepSlots * kHistBatch * sel::kBins1];
__device__ uint32_t g_step_fault_flags;

namespace dec {

constexpr uint32_t kStepSmem = dtc::kEngineBytes + 1024;  // + slack to align the base to 1024
static_assert(sizeof(sel::SelShared<kDecThreads>) <= dtc::kStages * dtc::kABytes,
              "the selection's shared memory reuses the engine's A stages");

template <class T, int MW>
__global__ void __launch_bounds__(kDecThreads, kStepCtasPerSm)
decode_step_kernel(const __grid_constant__ CUtensorMap pool_map, int32_t* __restrict__ out_idx,
                   float* __restrict__ logits, uint16_t* __restrict__ q_normed,
                   const uint16_t* __restrict__ index_qk, const float* __restrict__ cos_sin,
                   const int32_t* __restrict__ ctx, const uint16_t* __restrict__ w_q,
                   const uint16_t* __restrict__ w_k, float eps, const PoolDev pool,
                   int32_t* __restrict__ split_counters, int32_t num_kv_heads, int32_t max_blocks, float scale,
                   int32_t per_cta, uint32_t* __restrict__ arrivals, uint32_t* __restrict__ hists) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(16) float g1q[kHeadDim];
  __shared__ __align__(16) float g1k[kHeadDim];
  __shared__ int32_t vpages[kPageWindow];
  __shared__ int32_t last;
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const dtc::Engine en{base, smem_raw + (base - raw), &g_step_fault_flags};
  const int32_t b = blockIdx.x, y = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t c = __ldg(ctx + b);
  const int32_t n_vis = c > 0 ? min(c / kRatio, max_blocks) : 0;
  const int32_t g_begin = y * per_cta;
  const int32_t g_end = min(g_begin + per_cta, n_vis);
  uint32_t* const hist = hists != nullptr && n_vis > sel::kTopK ? hists + static_cast<int64_t>(b) * sel::kBins1 : nullptr;
  // the CTA that compresses block g_new = c/4 - 1 (if this step completes one): the
  // one whose run holds it, or the last one if g_new lies past maxBlocks
  const int32_t g_new = c > 0 && c % kRatio == 0 ? c / kRatio - 1 : -1;
  const bool owner = g_new >= 0 && min(g_new / per_cta, static_cast<int32_t>(gridDim.y) - 1) == y;
  // The owning CTA scores g_new itself when g_new < g_end.  If g_new's tile is one of the
  // first kStages (copied before the CTA barrier, with g_new's stale V-tail row), the
  // compressed row is written into that tile's A stage once the copy has landed; a later
  // tile is copied after the V-tail is written and fenced, and reads it from L2.
  const int t_patch = owner && g_new < g_end ? (g_new - g_begin) / dtc::kTile : dtc::kStages;
  const bool patch = t_patch < dtc::kStages;
  constexpr int pre_limit = dtc::kStages;
  const uint16_t* row = index_qk + static_cast<int64_t>(b) * kRowWidth;
  QHeadsIn qin{};
  CompressIn cin{};
  if (warp == 0) {
    if (lane == 0) ptx::prefetch_tensormap(&pool_map);  // its fetch overlaps the page-table loads
    stage_vpages(vpages, pool, b, g_begin, min(g_begin + per_cta, max_blocks), tid, 32);
    __syncwarp();
    dtc::engine_start(en, &pool_map, vpages, pool.head_size, g_begin, g_end, pre_limit);
  } else {
    // the q heads' and the block compress's loads, in flight across the barrier
    if (warp == 2) qin = q_heads_load(row, cos_sin, c, lane);
    if (warp == 3 && owner) cin = compress_load(pool, b, c, row, cos_sin, lane);
    stage_gamma<T>(w_q, g1q, tid - 32, kDecThreads - 32);
    stage_gamma<T>(w_k, g1k, tid - 32, kDecThreads - 32);
    dtc::zero_b_padding(en, tid - 32, kDecThreads - 32);
  }
  __syncthreads();
  const int h = lane >> 3, j = lane & 7;
  const int ca = chunk_a(j), cb = chunk_b(j);
  if (warp == 2) {
    uint4 oa, ob;
    q_heads_finish<T>(qin, c, g1q, eps, lane, oa, ob);
    dtc::put_q_chunk(en, h, ca / 8, oa);
    dtc::put_q_chunk(en, h, cb / 8, ob);
    if (y == 0) {
      uint16_t* dst = q_normed + static_cast<int64_t>(b) * (kNumQHeads * kHeadDim) + h * kHeadDim;
      st_v4(dst + ca, oa);
      st_v4(dst + cb, ob);
    }
  } else if (warp == 3 && c > 0) {
    if (c % kRatio != 0) {
      if (y == 0) {
        uint16_t* dst = pool_tail(pool, b, 0, c - 1);
        if (dst != nullptr) copy_tail(dst, row + kKCol, lane);
      }
    } else if (owner) {
      uint4 oa, ob;
      compress_finish<T>(cin, g1k, eps, lane, oa, ob);
      if (cin.ok && h == 0) {
        st_v4(cin.vtail + ca, oa);
        st_v4(cin.vtail + cb, ob);
      }
      ptx::fence_proxy_async_global();  // the V-tail, before a TMA copy issued later reads it
      if (patch && cin.ok)  // warp-uniform
        dtc::patch_a_row(en, t_patch, g_new - g_begin - dtc::kTile * t_patch, lane, ca, cb, oa, ob);
    }
  }
  ptx::fence_proxy_async_shared();  // the B operand, before the MMAs read it
  const uint32_t tmem = dtc::engine_setup(en);
  if (tid == 0) ptx::fence_proxy_async_global();
  float* lrow = logits + static_cast<int64_t>(b) * max_blocks;
  dtc::engine_run<T::kIsBf16>(en, tmem, &pool_map, vpages, pool.head_size, g_begin, g_end, lrow, scale,
                              pre_limit, hist);
  dtc::engine_teardown(tmem);

  // ---- the last CTA of sequence b selects its row.  The arrival releases this CTA's
  // logits and histogram counts (ordered before it by the teardown's CTA barrier) and
  // acquires those of the CTAs that arrived before.
  if (tid == 0) last = ptx::atom_add_acq_rel_gpu(arrivals + b, 1u) == gridDim.y - 1 ? 1 : 0;
  __syncthreads();
  if (!last) return;
  if (tid == 0) arrivals[b] = 0u;
  if (split_counters != nullptr)
    for (int k = tid; k < num_kv_heads; k += kDecThreads) split_counters[static_cast<int64_t>(b) * num_kv_heads + k] = 0;
  int32_t* out = out_idx + static_cast<int64_t>(b) * sel::kWidth;
  const int32_t tail = c > 0 ? c % kRatio : 0;
  if (n_vis <= sel::kTopK) {
    sel::write_unselected<kDecThreads>(out, c <= 0, n_vis, tail);
    return;
  }
  sel::SelShared<kDecThreads>& sh = *reinterpret_cast<sel::SelShared<kDecThreads>*>(en.ptr + dtc::kOffA);
  const sel::L2Keys keys{lrow, (reinterpret_cast<uintptr_t>(lrow) & 15u) == 0};
  sel::select_row<kDecThreads, MW, MW == 1>(keys, n_vis, sh, hist);
  sel::write_selected<kDecThreads>(out, sh.win(), tail, n_vis);
}

}  // namespace dec

namespace {
std::mutex g_step_mu;
uint32_t* g_step_base[64] = {};
uint32_t* g_step_hist_base[64] = {};
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
  uint32_t* hists = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_step_mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_step_base[dev] == nullptr) {  // the symbols' device addresses, once per device
      void* ptr = nullptr;
      if ((e = cudaGetSymbolAddress(&ptr, g_decode_step_arrivals)) != cudaSuccess) return e;
      void* hptr = nullptr;
      if ((e = cudaGetSymbolAddress(&hptr, g_decode_step_hist)) != cudaSuccess) return e;
      g_step_base[dev] = static_cast<uint32_t*>(ptr);
      g_step_hist_base[dev] = static_cast<uint32_t*>(hptr);
    }
    const int64_t slot = g_step_seq[dev]++ % kStepSlots;
    arrivals = g_step_base[dev] + slot * kStepMaxBatch;
    if (batch <= kHistBatch) hists = g_step_hist_base[dev] + slot * kHistBatch * sel::kBins1;
  }
  // Y CTAs a sequence, each over a run of per_cta blocks: about one wave of resident CTAs
  // over the batch, so that each CTA computes the q heads once
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int32_t per_cta = dec::decode_run_blocks(sms, kStepCtasPerSm, batch, max_blocks);
  const dim3 grid(static_cast<unsigned>(batch), static_cast<unsigned>((max_blocks + per_cta - 1) / per_cta));
  const int32_t words = (max_blocks + dec::kDecThreads * 32 - 1) / (dec::kDecThreads * 32);
  const int mw_index = words <= 1 ? 0 : words <= 2 ? 1 : words <= 4 ? 2 : 3;
  {
    static std::mutex mu;
    static bool attr_set[64][2][4] = {};
    std::lock_guard<std::mutex> lk(mu);
    bool& done = attr_set[dev][bf16 ? 1 : 0][mw_index];
    if (!done) {
      const void* fns[2][4] = {
          {reinterpret_cast<const void*>(dec::decode_step_kernel<F16, 1>),
           reinterpret_cast<const void*>(dec::decode_step_kernel<F16, 2>),
           reinterpret_cast<const void*>(dec::decode_step_kernel<F16, 4>),
           reinterpret_cast<const void*>(dec::decode_step_kernel<F16, 8>)},
          {reinterpret_cast<const void*>(dec::decode_step_kernel<Bf16, 1>),
           reinterpret_cast<const void*>(dec::decode_step_kernel<Bf16, 2>),
           reinterpret_cast<const void*>(dec::decode_step_kernel<Bf16, 4>),
           reinterpret_cast<const void*>(dec::decode_step_kernel<Bf16, 8>)}};
      e = cudaFuncSetAttribute(fns[bf16 ? 1 : 0][mw_index], cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(dec::kStepSmem));
      if (e != cudaSuccess) return e;
      done = true;
    }
  }
  CUtensorMap map;
  if ((e = encode_vtail_map(&map, pool)) != cudaSuccess) return e;
  auto* q = static_cast<uint16_t*>(q_normed);
  auto* iq = static_cast<const uint16_t*>(index_qk);
  auto* wq = static_cast<const uint16_t*>(w_q);
  auto* wk = static_cast<const uint16_t*>(w_k);
#define QSA_STEP_LAUNCH(T, MW)                                                                             \
  dec::decode_step_kernel<T, MW><<<grid, dec::kDecThreads, dec::kStepSmem, stream>>>(                     \
      map, out_idx, logits, q, iq, cos_sin, ctx, wq, wk, eps, pool, split_counters, num_kv_heads, max_blocks,     \
      scale, per_cta, arrivals, hists)
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

namespace dec {
// bin 0 of each of n histograms (kBins1 words apart) += add
__global__ void hist_offset_kernel(uint32_t* __restrict__ hist, int32_t n, uint32_t add) {
  const int32_t i = static_cast<int32_t>(blockIdx.x * blockDim.x + threadIdx.x);
  if (i < n) hist[static_cast<int64_t>(i) * sel::kBins1] += add;
}
}  // namespace dec

cudaError_t testing_decode_step_histograms(int32_t add, cudaStream_t stream) {
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_step_hist);
  if (e != cudaSuccess) return e;
  if (add == 0) return cudaMemsetAsync(ptr, 0, sizeof(g_decode_step_hist), stream);
  constexpr int32_t n = kStepSlots * kHistBatch;
  dec::hist_offset_kernel<<<(n + 255) / 256, 256, 0, stream>>>(static_cast<uint32_t*>(ptr), n,
                                                              static_cast<uint32_t>(add));
  return cudaGetLastError();
}

cudaError_t read_step_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_step_fault_flags, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_step_fault_flags, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  }
  return e;
}

}  // namespace qsa
