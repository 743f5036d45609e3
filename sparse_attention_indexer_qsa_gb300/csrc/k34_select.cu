// Prefill block selection ("Qsa Indexer Kernels": launchQsaIndexIdsFill,
// launchQsaIndexExpand, and the stable descending segmented sort between them).
//
//   ids_fill      K3: ids[r * numBlocks + c] = c
//   expand        K4: top kSel = min(512, nVis) sorted block ids -> token ids
//                 4*id + j, then the causal tail, then -1 to width 2051
//   topk_expand   the whole selection of a row in one CTA, without a segmented
//                 sort or its workspace: an MSB-first 8-bit radix select over the
//                 order-preserving u32 map of the FP32 logits finds the kSel-th
//                 largest key; keys above it, and keys equal to it in ascending
//                 block order until kSel are reached, are selected.  That is the
//                 set the page's stable descending sort puts first, and the rule of
//                 its decode top-k (launchQsaTopKExpandDecode); like the decode
//                 path, the selected blocks are emitted in ascending block order
//                 (the page's token ids are "unsorted"), then expanded.
#include <cstdint>

#include "qsa_launch.h"

namespace qsa {
namespace sel {

constexpr int kTopK = 512;
constexpr int kRatio = 4;
constexpr int kWidth = kTopK * kRatio + kRatio - 1;  // 2051

__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__global__ void ids_fill_kernel(int32_t* __restrict__ ids, int64_t total, int32_t num_blocks) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    ids[i] = static_cast<int32_t>(i % num_blocks);
}

// one CTA per row; rows [row_start, row_start + num_rows), sorted_ids chunk-local
__global__ void expand_kernel(int32_t* __restrict__ out_idx, const int32_t* __restrict__ sorted_ids,
                              const int32_t* __restrict__ ctx, int32_t seq_len, int32_t num_blocks,
                              int32_t row_start) {
  const int64_t r = static_cast<int64_t>(row_start) + blockIdx.x;
  const int32_t b = static_cast<int32_t>(r / seq_len);
  const int32_t t = static_cast<int32_t>(r - static_cast<int64_t>(b) * seq_len);
  const int32_t c = __ldg(ctx + b);
  int32_t* out = out_idx + r * kWidth;
  const bool padded = c <= 0 || t >= c;
  const int32_t n_vis = (t + 1) / kRatio;
  const int32_t k_sel = padded ? 0 : min(kTopK, n_vis);
  const int32_t tail = padded ? 0 : (t + 1) % kRatio;
  const int32_t* ids = sorted_ids + static_cast<int64_t>(blockIdx.x) * num_blocks;
  for (int i = threadIdx.x; i < kWidth; i += blockDim.x) {
    int32_t v = -1;
    if (i < kRatio * k_sel) v = __ldg(ids + i / kRatio) * kRatio + (i % kRatio);
    else if (i < kRatio * k_sel + tail) v = kRatio * n_vis + (i - kRatio * k_sel);
    out[i] = v;
  }
}

// One CTA (kSelThreads threads) per row.  Shared memory: the row's keys
// (num_blocks u32), per-warp histograms, the winners' block ids, scan scratch.
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

__device__ __forceinline__ uint32_t* keys_smem(uint8_t* base) { return reinterpret_cast<uint32_t*>(base); }

// exclusive scan of one value per thread over the CTA; returns the CTA total too
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += x;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint32_t base = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const uint32_t x = warp_tot[w];
    if (w < warp) base += x;
    total += x;
  }
  __syncthreads();  // warp_tot may be reused by the caller's next scan
  return base + incl - v;
}

// DECODE (launchQsaTopKExpandDecode): row b is sequence b's one new token at
// t = ctx_b - 1, logits [B, num_blocks = maxBlocks], outIdx [B, 2051], and the
// decode attention's split-K counters of b are zeroed first when given.
template <bool DECODE>
__global__ void __launch_bounds__(kSelThreads)
topk_expand_kernel(int32_t* __restrict__ out_idx, const float* __restrict__ logits,
                   const int32_t* __restrict__ ctx, int32_t seq_len, int32_t num_blocks,
                   int32_t row_start, int32_t* __restrict__ split_counters, int32_t num_kv_heads) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t hist[kSelWarps][256];
  __shared__ uint32_t warp_tot[kSelWarps];
  __shared__ int32_t win[kTopK];
  __shared__ uint32_t sh_bin, sh_above, sh_count;
  uint32_t* keys = keys_smem(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = lanemask_lt();

  const int32_t i = blockIdx.x;
  int64_t r;
  int32_t b, t, c;
  if (DECODE) {
    r = i;
    b = i;
    c = __ldg(ctx + b);
    t = c - 1;
    if (split_counters != nullptr)
      for (int k = tid; k < num_kv_heads; k += kSelThreads) split_counters[static_cast<int64_t>(b) * num_kv_heads + k] = 0;
  } else {
    r = static_cast<int64_t>(row_start) + i;
    b = static_cast<int32_t>(r / seq_len);
    t = static_cast<int32_t>(r - static_cast<int64_t>(b) * seq_len);
    c = __ldg(ctx + b);
  }
  int32_t* out = out_idx + r * kWidth;
  if (c <= 0 || t >= c) {  // padded row: all -1, logits not read
    for (int k = tid; k < kWidth; k += kSelThreads) out[k] = -1;
    return;
  }
  const int32_t n_vis = min((t + 1) / kRatio, num_blocks);
  const int32_t k_sel = min(kTopK, n_vis);
  const int32_t tail = (t + 1) % kRatio;

  if (n_vis <= kTopK) {
    // every visible block is selected, in ascending order
    for (int k = tid; k < kWidth; k += kSelThreads) {
      int32_t v = -1;
      if (k < kRatio * k_sel) v = k;                       // block k/4, token 4*(k/4) + k%4
      else if (k < kRatio * k_sel + tail) v = kRatio * n_vis + (k - kRatio * k_sel);
      out[k] = v;
    }
    return;
  }

  const float* row = logits + static_cast<int64_t>(i) * num_blocks;
  for (int32_t g = tid; g < n_vis; g += kSelThreads) keys[g] = orderable(__ldg(row + g));

  // ---- MSB-first radix select of the k_sel-th largest key
  uint32_t prefix = 0, mask = 0;
  int32_t remaining = k_sel;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int k = lane; k < 256; k += 32) hist[warp][k] = 0;
    __syncthreads();  // keys staged (first pass) / previous pass's reads done
    for (int32_t base = warp * 32; base < n_vis; base += kSelThreads) {
      const int32_t g = base + lane;
      const uint32_t u = g < n_vis ? keys[g] : 0u;
      const bool cand = g < n_vis && (u & mask) == prefix;
      const uint32_t active = __ballot_sync(0xffffffffu, cand);
      if (cand) {
        const uint32_t d = (u >> shift) & 255u;
        const uint32_t same = __match_any_sync(active, d);
        if ((same & lt) == 0) atomicAdd(&hist[warp][d], static_cast<uint32_t>(__popc(same)));
      }
    }
    __syncthreads();
    // thread d totals bin (255 - d): descending bin order, then an exclusive scan
    const uint32_t cnt = [&] {
      uint32_t s = 0;
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) s += hist[w][255 - tid];
      return s;
    }();
    uint32_t total;
    const uint32_t above = block_exclusive_scan(cnt, warp_tot, total);
    if (above < static_cast<uint32_t>(remaining) && static_cast<uint32_t>(remaining) <= above + cnt) {
      sh_bin = 255u - tid;
      sh_above = above;
      sh_count = cnt;
    }
    __syncthreads();
    remaining -= static_cast<int32_t>(sh_above);
    prefix |= sh_bin << shift;
    mask |= 255u << shift;
    const bool exact = sh_count == static_cast<uint32_t>(remaining);
    __syncthreads();  // everyone has read sh_*
    if (exact) break;  // the whole bin is selected
  }

  // ---- ordered gather: winners in ascending block order.  Thread k owns the
  // contiguous keys [k*C, k*C + C); a winner is above the threshold bin, or one
  // of the first `remaining` keys inside it (in block order).
  const int32_t chunk = (n_vis + kSelThreads - 1) / kSelThreads;
  const int32_t g0 = tid * chunk;
  const int32_t g1 = min(g0 + chunk, n_vis);
  uint32_t my_ties = 0;
  for (int32_t g = g0; g < g1; ++g) my_ties += (keys[g] & mask) == prefix;
  uint32_t tot;
  uint32_t tie_rank = block_exclusive_scan(my_ties, warp_tot, tot);
  uint32_t my_wins = 0;
  {
    uint32_t tr = tie_rank;
    for (int32_t g = g0; g < g1; ++g) {
      const uint32_t m = keys[g] & mask;
      if (m > prefix) ++my_wins;
      else if (m == prefix) { my_wins += tr < static_cast<uint32_t>(remaining); ++tr; }
    }
  }
  uint32_t pos = block_exclusive_scan(my_wins, warp_tot, tot);
  for (int32_t g = g0; g < g1; ++g) {
    const uint32_t m = keys[g] & mask;
    bool w = m > prefix;
    if (m == prefix) { w = tie_rank < static_cast<uint32_t>(remaining); ++tie_rank; }
    if (w) win[pos++] = g;
  }
  __syncthreads();

  // ---- expand
  for (int k = tid; k < kWidth; k += kSelThreads) {
    int32_t v = -1;
    if (k < kRatio * k_sel) v = win[k / kRatio] * kRatio + (k % kRatio);
    else if (k < kRatio * k_sel + tail) v = kRatio * n_vis + (k - kRatio * k_sel);
    out[k] = v;
  }
}

}  // namespace sel

cudaError_t launch_ids_fill(int32_t* ids, int32_t num_rows, int32_t num_blocks, int num_sms, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(num_rows) * num_blocks;
  const int64_t blocks = (total + 255) / 256;
  const int grid = static_cast<int>(blocks < 8LL * num_sms ? blocks : 8LL * num_sms);
  sel::ids_fill_kernel<<<grid, 256, 0, stream>>>(ids, total, num_blocks);
  return cudaGetLastError();
}

cudaError_t launch_expand(int32_t* out_idx, const int32_t* sorted_ids, const int32_t* ctx, int32_t seq_len,
                          int32_t num_blocks, int32_t row_start, int32_t num_rows, cudaStream_t stream) {
  sel::expand_kernel<<<num_rows, 256, 0, stream>>>(out_idx, sorted_ids, ctx, seq_len, num_blocks, row_start);
  return cudaGetLastError();
}

size_t topk_smem_bytes(int32_t num_blocks) { return (static_cast<size_t>(num_blocks) * 4 + 15) & ~size_t{15}; }

cudaError_t launch_topk_expand(int32_t* out_idx, const float* logits, const int32_t* ctx, int32_t seq_len,
                               int32_t num_blocks, int32_t row_start, int32_t num_rows, int num_sms,
                               cudaStream_t stream) {
  (void)num_sms;
  const size_t smem = topk_smem_bytes(num_blocks);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(sel::topk_expand_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  sel::topk_expand_kernel<false><<<num_rows, sel::kSelThreads, smem, stream>>>(out_idx, logits, ctx, seq_len,
                                                                               num_blocks, row_start, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_topk_expand_decode(int32_t* out_idx, const float* logits, const int32_t* ctx,
                                      int32_t* split_counters, int32_t num_kv_heads, int32_t batch,
                                      int32_t max_blocks, cudaStream_t stream) {
  const size_t smem = topk_smem_bytes(max_blocks);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(sel::topk_expand_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  sel::topk_expand_kernel<true><<<batch, sel::kSelThreads, smem, stream>>>(out_idx, logits, ctx, 1, max_blocks, 0,
                                                                          split_counters, num_kv_heads);
  return cudaGetLastError();
}

}  // namespace qsa
