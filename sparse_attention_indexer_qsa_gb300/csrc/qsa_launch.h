// Internal launcher interface between the C ABI (qsa_abi.cpp) and the kernels.
// Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace qsa {

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

cudaError_t launch_q_prep(const LaunchQPrep& a);         // K1a (k1a_qprep.cu)
cudaError_t launch_qk_prep(const LaunchQKPrep& a);       // fused K1a + prefill K1b (k1_stream.cu)
cudaError_t launch_k_compress(const LaunchKCompress& a);
cudaError_t launch_scores_tc(const LaunchScores& a);
cudaError_t launch_scores_cc(const LaunchScores& a);  // CUDA-core cross-check (testing only)
// K2 with its scheduler scratch in one fixed static array (qsa_index_scores_no_alloc)
cudaError_t launch_scores_tc_no_alloc(const LaunchScores& a);
int64_t scores_work_units(int32_t batch, int32_t seq_len, int32_t num_blocks, int32_t row_start,
                          int32_t num_rows);
int64_t scores_no_alloc_max_units();

// Prefill selection (k34_select.cu)
cudaError_t launch_ids_fill(int32_t* ids, int32_t num_rows, int32_t num_blocks, int num_sms, cudaStream_t stream);
cudaError_t launch_expand(int32_t* out_idx, const int32_t* sorted_ids, const int32_t* ctx, int32_t seq_len,
                          int32_t num_blocks, int32_t row_start, int32_t num_rows, cudaStream_t stream);
cudaError_t launch_topk_expand(int32_t* out_idx, const float* logits, const int32_t* ctx, int32_t seq_len,
                               int32_t num_blocks, int32_t row_start, int32_t num_rows, int num_sms,
                               cudaStream_t stream);
size_t topk_smem_bytes(int32_t num_blocks);

// Device fault flags: bits set by bounded waits that ran out (k2_scores_tc.cu, k1_stream.cu).
cudaError_t read_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream);
cudaError_t read_k1_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream);

// Cached cudaOccupancyMaxActiveBlocksPerMultiprocessor for (kernel, device).
cudaError_t occupancy_blocks_per_sm(const void* kernel, int threads, size_t smem, int* out);

}  // namespace qsa
