// Internal launcher interface between the C ABI (qsa_abi.cpp) and the kernels.
// Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace qsa {

// Paged indexer state ("Qsa Indexer Kernels", QsaIndexerPoolState): pool
// [2*numPages, 128, numKVHeads, poolHeadDim] T; page table [B, 2, maxPagesPerSeq]
// (plane 0: K pages, plane 1: V pages with ids already offset by +numPages; -1 =
// unused).  Token t's raw index-K tail: K page table[b][0][t >> 7], row t & 127,
// head 0, columns [headSize, headSize + 128); block g's kbar: V page
// table[b][1][(4g) >> 7], row (4g) & 127, head 0, same columns.
struct PoolDev {
  uint16_t* pool;
  const int32_t* table;
  int32_t max_pages, num_pages, num_kv_heads, pool_head_dim, head_size;
};

#ifdef __CUDACC__
// The tail of `token` in `plane` (0 = K, 1 = V), or nullptr when the page slot is past
// maxPagesPerSeq, unused (-1) or outside the pool: such entries are never dereferenced.
__device__ __forceinline__ uint16_t* pool_tail(const PoolDev& p, int32_t b, int plane, int32_t token) {
  if (token < 0) return nullptr;
  const int32_t slot = token >> 7;
  if (slot >= p.max_pages) return nullptr;
  const int32_t page = __ldg(p.table + (static_cast<int64_t>(b) * 2 + plane) * p.max_pages + slot);
  if (page < 0 || page >= 2 * p.num_pages) return nullptr;
  const int64_t row = token & 127;
  return p.pool + ((static_cast<int64_t>(page) * 128 + row) * p.num_kv_heads) * p.pool_head_dim + p.head_size;
}
#endif

struct LaunchQPrep {
  bool bf16;
  void* q_normed;
  const void* index_qk;
  const float* cos_sin;
  const int32_t* context_lengths;
  const void* w_q;
  float eps;
  int32_t batch, seq_len;
  int num_sms;
  cudaStream_t stream;
};

struct LaunchKCompress {
  bool bf16;
  void* kbar;
  const void* index_qk;
  const float* cos_sin;
  const int32_t* context_lengths;
  const void* w_k;
  float eps;
  int32_t batch, seq_len, num_blocks, block_begin, block_end, past_len;
  int num_sms;
  cudaStream_t stream;
};

struct LaunchKCompressPaged {
  LaunchKCompress base;
  PoolDev pool;
};

struct LaunchQKPrep {
  bool bf16;
  void* q_normed;
  void* kbar;
  const void* index_qk;
  const float* cos_sin;
  const int32_t* context_lengths;
  const void* w_q;
  const void* w_k;
  float eps;
  int32_t batch, seq_len, num_blocks;
  int num_sms;
  cudaStream_t stream;
};

struct LaunchScores {
  bool bf16;
  float* logits;
  const void* q_normed;
  const void* kbar;
  const int32_t* context_lengths;
  int32_t batch, seq_len, num_blocks, row_start, num_rows;
  float scale;  // 1.0f / sqrtf(128.0f), evaluated on the host in binary32
  int num_sms;
  cudaStream_t stream;
};

// K2 and the top-512 selection + expand in one kernel, no logits written
// (k2_topk_fused.cu); num_blocks <= scores_topk_max_blocks().
struct LaunchScoresTopk {
  bool bf16;
  int32_t* out_idx;
  const void* q_normed;
  const void* kbar;
  const int32_t* context_lengths;
  int32_t batch, seq_len, num_blocks, row_start, num_rows;
  float scale;
  int num_sms;
  cudaStream_t stream;
};

cudaError_t launch_q_prep(const LaunchQPrep& a);         // K1a (k1a_qprep.cu)
cudaError_t launch_qk_prep(const LaunchQKPrep& a);       // fused K1a + prefill K1b (k1_stream.cu)
cudaError_t launch_q_prep_staged(const LaunchQPrep& a);  // K1a through k1_stream.cu's staged q mode
cudaError_t launch_k_compress(const LaunchKCompress& a);
cudaError_t launch_scores_tc(const LaunchScores& a);
cudaError_t launch_scores_cc(const LaunchScores& a);  // CUDA-core cross-check (testing only)
// K2 with its scheduler scratch in one fixed static array (qsa_index_scores_no_alloc)
cudaError_t launch_scores_tc_no_alloc(const LaunchScores& a);
int64_t scores_work_units(int32_t batch, int32_t seq_len, int32_t num_blocks, int32_t row_start,
                          int32_t num_rows);
int64_t scores_no_alloc_max_units();

cudaError_t launch_k_compress_paged(const LaunchKCompressPaged& a);

// Decode path and prefill tail persistence (k_decode.cu)
cudaError_t launch_raw_k_tail_write_prefill(bool bf16, const void* index_qk, const int32_t* ctx, const PoolDev& pool,
                                            int32_t batch, int32_t seq_len, cudaStream_t stream);
cudaError_t launch_pre_decode(bool bf16, void* q_normed, const void* index_qk, const float* cos_sin,
                              const int32_t* ctx, const void* w_q, const void* w_k, float eps, const PoolDev& pool,
                              int32_t batch, cudaStream_t stream);
cudaError_t launch_scores_decode(bool bf16, float* logits, const void* q_normed, const int32_t* ctx,
                                 const PoolDev& pool, int32_t batch, int32_t max_blocks, float scale,
                                 cudaStream_t stream);

// Prefill selection (k34_select.cu)
cudaError_t launch_ids_fill(int32_t* ids, int32_t num_rows, int32_t num_blocks, int num_sms, cudaStream_t stream);
cudaError_t launch_expand(int32_t* out_idx, const int32_t* sorted_ids, const int32_t* ctx, int32_t seq_len,
                          int32_t num_blocks, int32_t row_start, int32_t num_rows, cudaStream_t stream);
cudaError_t launch_topk_expand(int32_t* out_idx, const float* logits, const int32_t* ctx, int32_t seq_len,
                               int32_t num_blocks, int32_t row_start, int32_t num_rows, int num_sms,
                               cudaStream_t stream);
int32_t topk_max_blocks();  // longest row the selection kernels take
cudaError_t launch_topk_expand_decode(int32_t* out_idx, const float* logits, const int32_t* ctx,
                                      int32_t* split_counters, int32_t num_kv_heads, int32_t batch,
                                      int32_t max_blocks, cudaStream_t stream);

// The decode step fused into one launch (k_decode_step.cu); batch <= decode_step_max_batch().
cudaError_t launch_decode_step(bool bf16, int32_t* out_idx, float* logits, void* q_normed, const void* index_qk,
                               const float* cos_sin, const int32_t* ctx, const void* w_q, const void* w_k,
                               float eps, const PoolDev& pool, int32_t* split_counters, int32_t num_kv_heads,
                               int32_t batch, int32_t max_blocks, float scale, cudaStream_t stream);
int32_t decode_step_max_batch();

// Device fault flags: bits set by bounded waits that ran out (k2_scores_tc.cu,
// k1_stream.cu, k_decode.cu, k_decode_step.cu).
cudaError_t read_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream);
cudaError_t read_k1_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream);
cudaError_t read_dec_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream);
// Test-only: one warp's bounded wait on an mbarrier nothing arrives on (k_decode.cu).
cudaError_t launch_bounded_wait_probe(uint64_t limit_ns, cudaStream_t stream);
cudaError_t read_step_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream);
// Testing: add `add` to bin 0 of every first-digit histogram of the one-launch decode
// step (every slot, every sequence), or zero them all when add == 0.
cudaError_t testing_decode_step_histograms(int32_t add, cudaStream_t stream);
cudaError_t read_fused_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream);

cudaError_t launch_scores_topk_fused(const LaunchScoresTopk& a);
int32_t scores_topk_max_blocks();

// Test-only plain streaming kernel with a K1 kernel's byte pattern (yardstick.cu).
cudaError_t launch_stream_yardstick(void* dst, const void* src, int64_t units, int rows, int64_t row_pitch,
                                    int64_t unit_pitch, int64_t offset, int bytes, cudaStream_t stream);
int yardstick_max_rows();
// Test-only plain kernel with the paged decode scoring's byte pattern (yardstick.cu);
// bytes a power of two in [16, 512].
cudaError_t launch_gather_yardstick(void* dst, const void* src, int64_t units, int64_t unit_pitch, int64_t offset,
                                    int bytes, cudaStream_t stream);

// TMA map (a CUtensorMap, 64-byte aligned) over the pool's V-tails for the tensor-core
// decode scoring (k_decode.cu).
cudaError_t encode_vtail_map(void* map, const PoolDev& pool);

// Cached cudaOccupancyMaxActiveBlocksPerMultiprocessor for (kernel, device).
cudaError_t occupancy_blocks_per_sm(const void* kernel, int threads, size_t smem, int* out);

}  // namespace qsa
