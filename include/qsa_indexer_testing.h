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

#ifdef __cplusplus
}
#endif

#endif /* QSA_INDEXER_TESTING_H */
