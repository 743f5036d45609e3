/*
 * qsa_indexer_testing.h -- entry points that exist only for the test suite.
 *
 * Not part of the product interface: nothing in the library's own call paths
 * uses them, and they may change without an ABI version bump.
 */
#ifndef QSA_INDEXER_TESTING_H
#define QSA_INDEXER_TESTING_H

#include "qsa_indexer.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * The K2 scores of qsa_index_scores ("Qsa Indexer Kernels", launchQsaIndexScores)
 * computed by a plain CUDA-core kernel (FP32 FMA dot products in ascending d, one
 * CTA per row and 128 blocks) instead of the tensor cores.  Same arguments,
 * layouts, validation and error codes as qsa_index_scores.  Tests hold it to the
 * oracle under the same tolerance as the tensor-core kernel; it is a second,
 * independent device implementation of the same formula.
 */
int qsa_testing_index_scores_cuda_core(qsa_dtype_t dtype, float* logits, const void* qNormed,
                                       const void* kbar, const int32_t* contextLengths,
                                       int32_t batchSize, int32_t seqLen, int32_t numBlocks,
                                       int32_t rowStart, int32_t numRows, qsa_stream_t stream);

/*
 * Exercises the bounded-wait error path of the tensor-core decode scoring: one warp
 * waits, through the same device routine the decode engine uses, on an mbarrier that
 * nothing arrives on.  After timeoutMs milliseconds (1..10000) the wait gives up, sets
 * bit 2 of the paged-decode-scores field of qsa_device_fault_flags (bit 18 of the
 * word) and the kernel returns; the context stays usable.  No fault, trap or
 * unbounded spin is involved.
 * Errors: QSA_E_RANGE (timeoutMs), QSA_E_CUDA.
 */
int qsa_testing_bounded_wait_probe(int32_t timeoutMs, qsa_stream_t stream);

/*
 * A plain streaming kernel for same-size bandwidth comparisons (no computation of
 * the page).  Unit u < units reads `rows` slices of `bytes` bytes at
 *   src + u*unitPitch + r*rowPitch + offset,  r < rows,
 * XORs them and writes `bytes` bytes at dst + u*bytes, one 16-byte chunk per
 * thread with every row's load issued first.  With rows = 4, rowPitch = 1280,
 * unitPitch = 5120, offset = 1024, bytes = 256 it moves what qsa_index_k_compress
 * moves for B*numBlocks valid blocks; with rows = 1, rowPitch = unitPitch = 1280,
 * offset = 0, bytes = 1024, what qsa_index_q_prep moves for B*seqLen valid rows.
 * Limits: 1 <= rows <= 8, bytes a multiple of 16 in [16, 1024], pitches and offset
 * multiples of 16, src/dst 16-byte aligned.
 * Errors: QSA_E_NULL, QSA_E_SHAPE, QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_testing_stream_yardstick(void* dst, const void* src, int64_t units, int32_t rows, int64_t rowPitch,
                                 int64_t unitPitch, int64_t offset, int32_t bytes, qsa_stream_t stream);

/*
 * A plain gathering kernel for same-size bandwidth comparisons with the paged decode
 * scoring (qsa_index_scores_decode, "Qsa Indexer Kernels": launchQsaIndexScoresDecode),
 * which reads one 256-byte V-tail a block at the pool's block pitch and writes one FP32
 * logit a block.  Unit u < units reads `bytes` bytes at
 *   src + u*unitPitch + offset
 * and writes the XOR of their 32-bit words (4 bytes) at dst + 4u; bytes/16
 * consecutive threads share a unit, and each such group issues the 16-byte loads of
 * 4 consecutive units before using any.  With unitPitch = 6144, bytes = 256 and src +
 * offset the first V-tail of a pool whose V pages are consecutive, it reads what
 * qsa_index_scores_decode reads for units valid blocks.  The caller owns both buffers:
 * every read must lie in src's allocation.
 * Limits: bytes a power of two in [16, 512]; src, unitPitch and offset 16-byte
 * aligned, dst 4-byte aligned.
 * Errors: QSA_E_NULL, QSA_E_SHAPE, QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_testing_gather_yardstick(void* dst, const void* src, int64_t units, int64_t unitPitch, int64_t offset,
                                 int32_t bytes, qsa_stream_t stream);

/*
 * The one-launch decode step (qsa_indexer_decode_step) keeps, for batches of up to 64
 * sequences, a first-digit histogram per sequence that its scoring CTAs fill and its
 * selection copies and leaves zeroed.  The selection checks that the copied counts total
 * the row's visible blocks and counts the row itself when they do not (as after a launch
 * whose waits ran out).  This entry adds `add` (> 0) to bin 0 of every such histogram,
 * in every one of the 16 launch slots, so that the next launches exercise that check; add
 * = 0 zeroes them all again.  Enqueued on `stream`.
 * Errors: QSA_E_RANGE (add < 0), QSA_E_CUDA.
 */
int qsa_testing_decode_step_histograms(int32_t add, qsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_INDEXER_TESTING_H */
