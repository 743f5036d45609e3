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
//                On the tensor cores (qsa_decode_tc.cuh): the dots are formed as in
//                K2, then relu, the ascending head sum and the scale as in K2.
#include <mutex>

#include <cudaTypedefs.h>

#include "qsa_decode.cuh"
#include "qsa_decode_tc.cuh"

namespace qsa {

__device__ uint32_t g_dec_fault_flags;

namespace dec {

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
    uint4 oa, ob;
    q_heads<T>(row, cos_sin, c, g1q, eps, lane, oa, ob);
    uint16_t* dst = q_normed + static_cast<int64_t>(b) * (kNumQHeads * kHeadDim) + h * kHeadDim;
    st_v4(dst + ca, oa);
    st_v4(dst + cb, ob);
    return;
  }
  if (c <= 0) return;
  if (c % kRatio != 0) {
    uint16_t* dst = pool_tail(pool, b, 0, c - 1);
    if (dst != nullptr) copy_tail(dst, row + kKCol, lane);
    return;
  }
  uint4 oa, ob;
  uint16_t* vtail = nullptr;
  const bool ok = compress_block<T>(pool, b, c, row, cos_sin, g1k, eps, lane, oa, ob, &vtail);
  if (ok && h == 0) {
    st_v4(vtail + ca, oa);
    st_v4(vtail + cb, ob);
  }
}

constexpr int kScoresThreads = 32 * dtc::kEngineWarps;
constexpr uint32_t kScoresSmem = dtc::kEngineBytes + 1024;  // + slack to align the base to 1024

// grid (B, ceilDiv(maxBlocks, run)), kScoresThreads threads: the tensor-core engine
// over the CTA's run of blocks of the valid prefix, q read from qNormed.
template <bool kBf16>
__global__ void __launch_bounds__(kScoresThreads, kScoresCtasPerSm)
    scores_decode_kernel(const __grid_constant__ CUtensorMap pool_map, float* __restrict__ logits,
                         const uint16_t* __restrict__ q_normed, const int32_t* __restrict__ ctx,
                         const PoolDev pool, int32_t max_blocks, float scale, int32_t run) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int32_t vpages[kPageWindow];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const dtc::Engine en{base, smem_raw + (base - raw), &g_dec_fault_flags};
  const int32_t b = blockIdx.x;
  const int32_t c = __ldg(ctx + b);
  const int32_t n_vis = c > 0 ? min(c / kRatio, max_blocks) : 0;
  const int32_t g_begin = blockIdx.y * run;
  const int32_t g_end = min(g_begin + run, n_vis);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    // the page entries of the whole run (their loads need not wait for the context
    // length), then the first tiles' copies, before the CTA barrier
    if (tid == 0) ptx::prefetch_tensormap(&pool_map);  // its fetch overlaps the page-table loads
    stage_vpages(vpages, pool, b, g_begin, min(g_begin + run, max_blocks), tid, 32);
    __syncwarp();
    if (g_begin < n_vis) dtc::engine_start(en, &pool_map, vpages, pool.head_size, g_begin, g_end, dtc::kStages);
  } else if (g_begin < n_vis) {
    const int k = tid - 32;
    if (k < kNumQHeads * 16) {
      const int h = k >> 4, ch = k & 15;
      dtc::put_q_chunk(en, h, ch,
                       ld_cached_v4(q_normed + static_cast<int64_t>(b) * (kNumQHeads * kHeadDim) + h * kHeadDim +
                                    8 * ch));
    }
    dtc::zero_b_padding(en, k, kScoresThreads - 32);
    ptx::fence_proxy_async_shared();
  }
  if (g_begin >= n_vis) return;  // only the valid prefix is written (the whole CTA leaves)
  const uint32_t tmem = dtc::engine_setup(en);
  dtc::engine_run<kBf16>(en, tmem, &pool_map, vpages, pool.head_size, g_begin, g_end,
                         logits + static_cast<int64_t>(b) * max_blocks, scale, dtc::kStages);
  dtc::engine_teardown(tmem);
}

// Test-only: the engine's bounded wait on an mbarrier that nothing arrives on.  Every
// thread of one warp waits; the wait runs out after limit_ns, sets the epilogue fault
// bit of this module's fault word and the CTA's abort flag, and the kernel returns.
__global__ void bounded_wait_probe_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar_word;
  __shared__ int abort_flag;
  const uint32_t bar = ptx::smem_u32(&bar_word);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncwarp();
  dtc::wait_bounded_raw(bar, 0, &abort_flag, &g_dec_fault_flags, dtc::kFaultEpilogue, limit_ns);
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
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  {
    static std::mutex mu;
    static bool attr_set[64][2] = {};
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev][bf16 ? 1 : 0]) {
      e = bf16 ? cudaFuncSetAttribute(dec::scores_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(dec::kScoresSmem))
               : cudaFuncSetAttribute(dec::scores_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(dec::kScoresSmem));
      if (e != cudaSuccess) return e;
      attr_set[dev][bf16 ? 1 : 0] = true;
    }
  }
  CUtensorMap map;
  if ((e = encode_vtail_map(&map, pool)) != cudaSuccess) return e;
  const int32_t run = dec::decode_run_blocks(sms, dec::kScoresCtasPerSm, batch, max_blocks);
  const dim3 grid(static_cast<unsigned>(batch), static_cast<unsigned>((max_blocks + run - 1) / run));
  auto* q = static_cast<const uint16_t*>(q_normed);
  if (bf16)
    dec::scores_decode_kernel<true>
        <<<grid, dec::kScoresThreads, dec::kScoresSmem, stream>>>(map, logits, q, ctx, pool, max_blocks, scale, run);
  else
    dec::scores_decode_kernel<false>
        <<<grid, dec::kScoresThreads, dec::kScoresSmem, stream>>>(map, logits, q, ctx, pool, max_blocks, scale, run);
  return cudaGetLastError();
}

// The pool's V-tails as a 3-D map {poolHeadDim, 4 x numKVHeads, 2 x numPages x 32}
// (element within a token-head row, token-head row within a 4-token block, block),
// box {64, 1, 32}: one page's 32 V-tail halves per copy, 128-byte swizzle.
cudaError_t encode_vtail_map(void* map, const PoolDev& pool) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (status == cudaSuccess && q != cudaDriverEntryPointSuccess) status = cudaErrorNotSupported;
    if (status == cudaSuccess) encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  if (status != cudaSuccess) return status;
  const uint64_t phd = static_cast<uint64_t>(pool.pool_head_dim);
  const uint64_t rows = 4ull * static_cast<uint64_t>(pool.num_kv_heads);
  cuuint64_t dims[3] = {phd, rows, 2ull * static_cast<uint64_t>(pool.num_pages) * 32ull};
  cuuint64_t strides[2] = {phd * 2, rows * phd * 2};
  cuuint32_t box[3] = {64, 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, pool.pool, dims, strides,
                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_bounded_wait_probe(uint64_t limit_ns, cudaStream_t stream) {
  dec::bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_dec_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_dec_fault_flags, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_dec_fault_flags, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  }
  return e;
}

}  // namespace qsa
