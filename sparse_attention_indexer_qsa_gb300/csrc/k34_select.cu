// Prefill block selection ("Qsa Indexer Kernels": launchQsaIndexIdsFill,
// launchQsaIndexExpand, and the stable descending segmented sort between them).
//
//   ids_fill      K3: ids[r * numBlocks + c] = c
//   expand        K4: top kSel = min(512, nVis) sorted block ids -> token ids
//                 4*id + j, then the causal tail, then -1 to width 2051
//   topk          the whole selection of a row in one CTA, without a segmented
//                 sort or its workspace: an MSB-first radix select (a 1024-bin first
//                 digit, then 8-bit digits over the candidates it leaves) on the
//                 order-preserving u32 map of the FP32 logits finds the kSel-th
//                 largest key; keys above it, and keys equal to it in ascending
//                 block order until kSel are reached, are selected.  That is the
//                 set the page's stable descending sort puts first, and the rule of
//                 its decode top-k (launchQsaTopKExpandDecode); like the decode
//                 path, the selected blocks are emitted in ascending block order
//                 (the page's token ids are "unsorted"), then expanded.
#include <cstdint>

#include "qsa_launch.h"
#include "qsa_select.cuh"

namespace qsa {

namespace sel {

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

struct RowInfo {
  int64_t r;      // global row
  int32_t n_vis, tail;
  bool padded;
};

template <bool DECODE>
__device__ __forceinline__ RowInfo row_info(int32_t i, const int32_t* ctx, int32_t seq_len, int32_t num_blocks,
                                            int32_t row_start) {
  RowInfo ri;
  int32_t b, t;
  if (DECODE) {
    ri.r = i;
    b = i;
    t = __ldg(ctx + b) - 1;
  } else {
    ri.r = static_cast<int64_t>(row_start) + i;
    if (ri.r <= 0xffffffffLL) {
      const uint32_t ru = static_cast<uint32_t>(ri.r);
      b = static_cast<int32_t>(ru / static_cast<uint32_t>(seq_len));
      t = static_cast<int32_t>(ru - static_cast<uint32_t>(b) * static_cast<uint32_t>(seq_len));
    } else {
      b = static_cast<int32_t>(ri.r / seq_len);
      t = static_cast<int32_t>(ri.r - static_cast<int64_t>(b) * seq_len);
    }
  }
  const int32_t c = __ldg(ctx + b);
  ri.padded = c <= 0 || t >= c;
  ri.n_vis = ri.padded ? 0 : min((t + 1) / kRatio, num_blocks);
  ri.tail = ri.padded ? 0 : (t + 1) % kRatio;
  return ri;
}

// QSA_SEL_CODES: rows of at most 32 * T * 2 blocks keep each key's first digit >> 2 in
// shared memory, so the ordered pass re-reads only the keys whose code is the
// threshold bin's (0.591 -> 0.530 ms at B=8, S=16384)
#ifndef QSA_SEL_CODES
#define QSA_SEL_CODES 1
#endif

// Resident CTAs a kernel is compiled for: QSA_SEL_WARPS_PER_SM warps for the small
// prefill CTAs with short rows, 32 warps (64 registers a thread) otherwise.
constexpr int sel_min_blocks(int T, int MW) { return (T == 64 && MW < 8 ? QSA_SEL_WARPS_PER_SM : 32) * 32 / T; }

// DECODE (launchQsaTopKExpandDecode): row b is sequence b's one new token at
// t = ctx_b - 1, logits [B, num_blocks = maxBlocks], outIdx [B, 2051], and the
// decode attention's split-K counters of b are zeroed first when given.
// T: threads a row; MW: 32-bit mask words a thread owns, num_blocks <= T * 32 * MW.
template <int T, int MW, bool DECODE>
__global__ void __launch_bounds__(T, sel_min_blocks(T, MW))
topk_kernel(int32_t* __restrict__ out_idx, const float* __restrict__ logits, const int32_t* __restrict__ ctx,
            int32_t seq_len, int32_t num_blocks, int32_t row_start, int32_t* __restrict__ split_counters,
            int32_t num_kv_heads) {
  __shared__ __align__(16) SelShared<T> sh;
  // each visible key's first digit >> 2, for rows of at most 32 * T * MW blocks
  constexpr bool kCodes = QSA_SEL_CODES && !DECODE && MW <= 2;
  __shared__ __align__(16) uint8_t codes[kCodes ? 32 * T * MW : 16];
  const int32_t i = blockIdx.x;
  if (DECODE && split_counters != nullptr)
    for (int k = threadIdx.x; k < num_kv_heads; k += T) split_counters[static_cast<int64_t>(i) * num_kv_heads + k] = 0;
  const RowInfo ri = row_info<DECODE>(i, ctx, seq_len, num_blocks, row_start);
  int32_t* out = out_idx + ri.r * kWidth;
  if (ri.n_vis <= kTopK) {
    write_unselected<T>(out, ri.padded, ri.n_vis, ri.tail);
    return;
  }
  const float* row = logits + static_cast<int64_t>(i) * num_blocks;
  const GlobalKeys keys{row, (reinterpret_cast<uintptr_t>(row) & 15u) == 0};
  select_row<T, MW, DECODE && MW == 1>(keys, ri.n_vis, sh, nullptr, kCodes ? codes : nullptr);
  write_selected<T>(out, sh.win(), ri.tail, ri.n_vis);
}

#ifndef QSA_SEL_THREADS
#define QSA_SEL_THREADS 64
#endif
#ifndef QSA_SEL_DECODE_THREADS
#define QSA_SEL_DECODE_THREADS 128
#endif

template <int T, bool DECODE>
cudaError_t launch_plain(int32_t* out_idx, const float* logits, const int32_t* ctx, int32_t seq_len,
                         int32_t num_blocks, int32_t row_start, int32_t rows, int32_t* split_counters,
                         int32_t num_kv_heads, cudaStream_t stream) {
  const int32_t words = (num_blocks + T * 32 - 1) / (T * 32);
#define QSA_SEL_LAUNCH(MW)                                                                          \
  topk_kernel<T, MW, DECODE><<<rows, T, 0, stream>>>(out_idx, logits, ctx, seq_len, num_blocks, row_start, \
                                                      split_counters, num_kv_heads)
  if (words <= 1) QSA_SEL_LAUNCH(1);
  else if (words <= 2) QSA_SEL_LAUNCH(2);
  else if (words <= 4) QSA_SEL_LAUNCH(4);
  else if (words <= 8) QSA_SEL_LAUNCH(8);
  else QSA_SEL_LAUNCH(16);
#undef QSA_SEL_LAUNCH
  return cudaGetLastError();
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

int32_t topk_max_blocks() { return sel::kMaxBlocks; }

cudaError_t launch_topk_expand(int32_t* out_idx, const float* logits, const int32_t* ctx, int32_t seq_len,
                               int32_t num_blocks, int32_t row_start, int32_t num_rows, int num_sms,
                               cudaStream_t stream) {
  (void)num_sms;
  using namespace sel;
  if (num_blocks <= QSA_SEL_THREADS * 32 * 16)
    return launch_plain<QSA_SEL_THREADS, false>(out_idx, logits, ctx, seq_len, num_blocks, row_start, num_rows,
                                                nullptr, 0, stream);
  return launch_plain<128, false>(out_idx, logits, ctx, seq_len, num_blocks, row_start, num_rows, nullptr, 0,
                                  stream);
}


cudaError_t launch_topk_expand_decode(int32_t* out_idx, const float* logits, const int32_t* ctx,
                                      int32_t* split_counters, int32_t num_kv_heads, int32_t batch,
                                      int32_t max_blocks, cudaStream_t stream) {
  return sel::launch_plain<QSA_SEL_DECODE_THREADS, true>(out_idx, logits, ctx, 1, max_blocks, 0, batch,
                                                        split_counters, num_kv_heads, stream);
}

}  // namespace qsa
