// The C ABI (include/qsa_indexer.h): host-side validation, device checks,
// dtype dispatch and error reporting.  Every check here runs before anything is
// enqueued; device data is never read on the host.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdint>
#include <mutex>

#include "../../include/qsa_indexer.h"
#include "../../include/qsa_indexer_testing.h"
#include "qsa_launch.h"

#define QSA_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct DeviceInfo {
  bool known = false;
  int num_sms = 0;
  int major = 0, minor = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

// SM count and compute capability of the current device (cached per device).
int current_device(const char* fn, DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(QSA_E_CUDA, "%s: cudaGetDevice: %s", fn, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(QSA_E_DEVICE, "%s: device ordinal %d unsupported", fn, dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.known) {
    if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return fail(QSA_E_CUDA, "%s: cudaDeviceGetAttribute: %s", fn, cudaGetErrorString(e));
    d.known = true;
  }
  if (d.major != 10 || d.minor != 3)
    return fail(QSA_E_DEVICE, "%s: the library is built for sm_103a only; device %d is sm_%d%d", fn,
                dev, d.major, d.minor);
  *out = d;
  return QSA_OK;
}

int check_dtype(const char* fn, qsa_dtype_t dt) {
  if (dt != QSA_BF16 && dt != QSA_F16) return fail(QSA_E_DTYPE, "%s: unknown dtype %d", fn, static_cast<int>(dt));
  return QSA_OK;
}

int launched(const char* fn, cudaError_t e) {
  if (e != cudaSuccess) return fail(QSA_E_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  g_last_error[0] = '\0';
  return QSA_OK;
}

int validate_scores(const char* fn, qsa_dtype_t dtype, const float* logits, const void* qNormed,
                    const void* kbar, const int32_t* ctx, int32_t B, int32_t S, int32_t NB,
                    int32_t rowStart, int32_t numRows) {
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!logits || !qNormed || !kbar || !ctx) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (B < 1 || S < 1) return fail(QSA_E_SHAPE, "%s: batchSize=%d seqLen=%d must be >= 1", fn, B, S);
  if (static_cast<int64_t>(B) * S > INT32_MAX) return fail(QSA_E_SHAPE, "%s: batchSize*seqLen exceeds INT32_MAX", fn);
  if (NB < (S + 3) / 4) return fail(QSA_E_SHAPE, "%s: numBlocks=%d < ceilDiv(seqLen=%d, 4)", fn, NB, S);
  if (rowStart < 0 || numRows < 0 || static_cast<int64_t>(rowStart) + numRows > static_cast<int64_t>(B) * S)
    return fail(QSA_E_RANGE, "%s: rows [%d, %d + %d) outside [0, %lld)", fn, rowStart, rowStart, numRows,
                static_cast<long long>(B) * S);
  if (!aligned(qNormed, 16) || !aligned(kbar, 16) || !aligned(logits, 4) || !aligned(ctx, 4))
    return fail(QSA_E_ALIGN, "%s: qNormed/kbar must be 16-byte aligned, logits/contextLengths 4-byte", fn);
  return QSA_OK;
}

float score_scale() {
  volatile float root = std::sqrt(128.0f);  // binary32 sqrt, then a binary32 division
  return 1.0f / root;
}

}  // namespace

QSA_API int qsa_abi_version(void) { return QSA_ABI_VERSION; }

QSA_API const char* qsa_last_error(void) { return g_last_error; }

QSA_API int qsa_index_q_prep(qsa_dtype_t dtype, void* qNormed, const void* indexQk, const float* cosSin,
                             const int32_t* contextLengths, const void* wQ, float rmsEps,
                             int32_t batchSize, int32_t seqLen, qsa_stream_t stream) {
  static const char* fn = "qsa_index_q_prep";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!qNormed || !indexQk || !cosSin || !contextLengths || !wQ) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (batchSize < 1 || seqLen < 1)
    return fail(QSA_E_SHAPE, "%s: batchSize=%d seqLen=%d must be >= 1", fn, batchSize, seqLen);
  if (static_cast<int64_t>(batchSize) * seqLen > INT32_MAX)
    return fail(QSA_E_SHAPE, "%s: batchSize*seqLen exceeds INT32_MAX", fn);
  if (!aligned(qNormed, 16) || !aligned(indexQk, 16) || !aligned(cosSin, 16) || !aligned(wQ, 16) ||
      !aligned(contextLengths, 4))
    return fail(QSA_E_ALIGN, "%s: T and FP32 arrays must be 16-byte aligned, contextLengths 4-byte", fn);
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  qsa::LaunchQPrep a{dtype == QSA_BF16, qNormed, indexQk, cosSin, contextLengths, wQ, rmsEps,
                     batchSize, seqLen, d.num_sms, reinterpret_cast<cudaStream_t>(stream)};
  return launched(fn, qsa::launch_q_prep(a));
}

QSA_API int qsa_index_qk_prep(qsa_dtype_t dtype, void* qNormed, void* kbar, const void* indexQk,
                              const float* cosSin, const int32_t* contextLengths, const void* wQ,
                              const void* wK, float rmsEps, int32_t batchSize, int32_t seqLen,
                              int32_t numBlocks, qsa_stream_t stream) {
  static const char* fn = "qsa_index_qk_prep";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!qNormed || !kbar || !indexQk || !cosSin || !contextLengths || !wQ || !wK)
    return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (batchSize < 1 || seqLen < 1)
    return fail(QSA_E_SHAPE, "%s: batchSize=%d seqLen=%d must be >= 1", fn, batchSize, seqLen);
  if (static_cast<int64_t>(batchSize) * seqLen > INT32_MAX)
    return fail(QSA_E_SHAPE, "%s: batchSize*seqLen exceeds INT32_MAX", fn);
  if (numBlocks < (seqLen + 3) / 4)
    return fail(QSA_E_SHAPE, "%s: numBlocks=%d < ceilDiv(seqLen=%d, 4)", fn, numBlocks, seqLen);
  if (!aligned(qNormed, 16) || !aligned(kbar, 16) || !aligned(indexQk, 16) || !aligned(cosSin, 16) ||
      !aligned(wQ, 16) || !aligned(wK, 16) || !aligned(contextLengths, 4))
    return fail(QSA_E_ALIGN, "%s: T and FP32 arrays must be 16-byte aligned, contextLengths 4-byte", fn);
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  qsa::LaunchQKPrep a{dtype == QSA_BF16, qNormed, kbar, indexQk, cosSin, contextLengths, wQ, wK, rmsEps,
                      batchSize, seqLen, numBlocks, d.num_sms, reinterpret_cast<cudaStream_t>(stream)};
  return launched(fn, qsa::launch_qk_prep(a));
}

QSA_API int qsa_index_k_compress(qsa_dtype_t dtype, void* kbar, const void* indexQk, const float* cosSin,
                                 const int32_t* contextLengths, const void* wK, float rmsEps,
                                 int32_t batchSize, int32_t seqLen, int32_t numBlocks, int32_t blockBegin,
                                 int32_t blockEnd, int32_t pastLen, qsa_stream_t stream) {
  static const char* fn = "qsa_index_k_compress";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!kbar || !indexQk || !cosSin || !contextLengths || !wK) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (batchSize < 1 || seqLen < 1 || numBlocks < 1)
    return fail(QSA_E_SHAPE, "%s: batchSize=%d seqLen=%d numBlocks=%d must be >= 1", fn, batchSize, seqLen, numBlocks);
  if (static_cast<int64_t>(batchSize) * seqLen > INT32_MAX)
    return fail(QSA_E_SHAPE, "%s: batchSize*seqLen exceeds INT32_MAX", fn);
  if (blockBegin < 0 || blockBegin > blockEnd || blockEnd > numBlocks || pastLen < 0)
    return fail(QSA_E_RANGE, "%s: need 0 <= blockBegin=%d <= blockEnd=%d <= numBlocks=%d and pastLen=%d >= 0", fn,
                blockBegin, blockEnd, numBlocks, pastLen);
  if (static_cast<int64_t>(numBlocks) * 4 > INT32_MAX)
    return fail(QSA_E_SHAPE, "%s: 4*numBlocks exceeds INT32_MAX", fn);
  if (!aligned(kbar, 16) || !aligned(indexQk, 16) || !aligned(cosSin, 16) || !aligned(wK, 16) ||
      !aligned(contextLengths, 4))
    return fail(QSA_E_ALIGN, "%s: T and FP32 arrays must be 16-byte aligned, contextLengths 4-byte", fn);
  if (blockBegin == blockEnd) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  qsa::LaunchKCompress a{dtype == QSA_BF16, kbar, indexQk, cosSin, contextLengths, wK, rmsEps, batchSize, seqLen,
                         numBlocks, blockBegin, blockEnd, pastLen, d.num_sms,
                         reinterpret_cast<cudaStream_t>(stream)};
  return launched(fn, qsa::launch_k_compress(a));
}

QSA_API int qsa_index_scores(qsa_dtype_t dtype, float* logits, const void* qNormed, const void* kbar,
                             const int32_t* contextLengths, int32_t batchSize, int32_t seqLen,
                             int32_t numBlocks, int32_t rowStart, int32_t numRows, qsa_stream_t stream) {
  static const char* fn = "qsa_index_scores";
  int st = validate_scores(fn, dtype, logits, qNormed, kbar, contextLengths, batchSize, seqLen, numBlocks,
                           rowStart, numRows);
  if (st != QSA_OK) return st;
  if (numRows == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  qsa::LaunchScores a{dtype == QSA_BF16, logits, qNormed, kbar, contextLengths, batchSize, seqLen,
                      numBlocks, rowStart, numRows, score_scale(), d.num_sms,
                      reinterpret_cast<cudaStream_t>(stream)};
  return launched(fn, qsa::launch_scores_tc(a));
}

QSA_API int qsa_index_scores_no_alloc(qsa_dtype_t dtype, float* logits, const void* qNormed, const void* kbar,
                                      const int32_t* contextLengths, int32_t batchSize, int32_t seqLen,
                                      int32_t numBlocks, int32_t rowStart, int32_t numRows,
                                      qsa_stream_t stream) {
  static const char* fn = "qsa_index_scores_no_alloc";
  int st = validate_scores(fn, dtype, logits, qNormed, kbar, contextLengths, batchSize, seqLen, numBlocks,
                           rowStart, numRows);
  if (st != QSA_OK) return st;
  if (numRows == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  const int64_t units = qsa::scores_work_units(batchSize, seqLen, numBlocks, rowStart, numRows);
  if (units > qsa::scores_no_alloc_max_units())
    return fail(QSA_E_SHAPE, "%s: %lld work units exceed the static scratch counter's maximum of %lld", fn,
                static_cast<long long>(units), static_cast<long long>(qsa::scores_no_alloc_max_units()));
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  qsa::LaunchScores a{dtype == QSA_BF16, logits, qNormed, kbar, contextLengths, batchSize, seqLen,
                      numBlocks, rowStart, numRows, score_scale(), d.num_sms,
                      reinterpret_cast<cudaStream_t>(stream)};
  return launched(fn, qsa::launch_scores_tc_no_alloc(a));
}

QSA_API int qsa_index_ids_fill(int32_t* ids, int32_t numRows, int32_t numBlocks, qsa_stream_t stream) {
  static const char* fn = "qsa_index_ids_fill";
  if (!ids) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (numRows < 0 || numBlocks < 1) return fail(QSA_E_SHAPE, "%s: numRows=%d >= 0, numBlocks=%d >= 1 required", fn, numRows, numBlocks);
  if (!aligned(ids, 4)) return fail(QSA_E_ALIGN, "%s: ids must be 4-byte aligned", fn);
  if (numRows == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  int st = current_device(fn, &d);
  if (st != QSA_OK) return st;
  return launched(fn, qsa::launch_ids_fill(ids, numRows, numBlocks, d.num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
int validate_selection(const char* fn, const void* outIdx, const void* in, const int32_t* ctx, int32_t B,
                       int32_t S, int32_t NB, int32_t rowStart, int32_t numRows) {
  if (!outIdx || !in || !ctx) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (B < 1 || S < 1) return fail(QSA_E_SHAPE, "%s: batchSize=%d seqLen=%d must be >= 1", fn, B, S);
  if (static_cast<int64_t>(B) * S > INT32_MAX) return fail(QSA_E_SHAPE, "%s: batchSize*seqLen exceeds INT32_MAX", fn);
  if (NB < (S + 3) / 4) return fail(QSA_E_SHAPE, "%s: numBlocks=%d < ceilDiv(seqLen=%d, 4)", fn, NB, S);
  if (rowStart < 0 || numRows < 0 || static_cast<int64_t>(rowStart) + numRows > static_cast<int64_t>(B) * S)
    return fail(QSA_E_RANGE, "%s: rows [%d, %d + %d) outside [0, %lld)", fn, rowStart, rowStart, numRows,
                static_cast<long long>(B) * S);
  if (!aligned(outIdx, 4) || !aligned(in, 4) || !aligned(ctx, 4))
    return fail(QSA_E_ALIGN, "%s: arrays must be 4-byte aligned", fn);
  return QSA_OK;
}
}  // namespace

QSA_API int qsa_index_expand(int32_t* outIdx, const int32_t* sortedIds, const int32_t* contextLengths,
                             int32_t batchSize, int32_t seqLen, int32_t numBlocks, int32_t rowStart,
                             int32_t numRows, qsa_stream_t stream) {
  static const char* fn = "qsa_index_expand";
  int st = validate_selection(fn, outIdx, sortedIds, contextLengths, batchSize, seqLen, numBlocks, rowStart, numRows);
  if (st != QSA_OK) return st;
  if (numRows == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  return launched(fn, qsa::launch_expand(outIdx, sortedIds, contextLengths, seqLen, numBlocks, rowStart, numRows,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_index_topk_expand(int32_t* outIdx, const float* logits, const int32_t* contextLengths,
                                  int32_t batchSize, int32_t seqLen, int32_t numBlocks, int32_t rowStart,
                                  int32_t numRows, qsa_stream_t stream) {
  static const char* fn = "qsa_index_topk_expand";
  int st = validate_selection(fn, outIdx, logits, contextLengths, batchSize, seqLen, numBlocks, rowStart, numRows);
  if (st != QSA_OK) return st;
  if (numBlocks > qsa::topk_max_blocks())
    return fail(QSA_E_SHAPE, "%s: numBlocks=%d above %d", fn, numBlocks, qsa::topk_max_blocks());
  if (numRows == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  return launched(fn, qsa::launch_topk_expand(outIdx, logits, contextLengths, seqLen, numBlocks, rowStart, numRows,
                                              d.num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_index_scores_topk_expand(qsa_dtype_t dtype, int32_t* outIdx, const void* qNormed,
                                         const void* kbar, const int32_t* contextLengths, int32_t batchSize,
                                         int32_t seqLen, int32_t numBlocks, int32_t rowStart, int32_t numRows,
                                         qsa_stream_t stream) {
  static const char* fn = "qsa_index_scores_topk_expand";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!qNormed || !kbar) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if ((st = validate_selection(fn, outIdx, qNormed, contextLengths, batchSize, seqLen, numBlocks, rowStart,
                               numRows)) != QSA_OK)
    return st;
  if (numBlocks > qsa::scores_topk_max_blocks())
    return fail(QSA_E_SHAPE, "%s: numBlocks=%d above %d (use qsa_index_scores + qsa_index_topk_expand)", fn,
                numBlocks, qsa::scores_topk_max_blocks());
  if (!aligned(qNormed, 16) || !aligned(kbar, 16))
    return fail(QSA_E_ALIGN, "%s: qNormed/kbar must be 16-byte aligned", fn);
  if (numRows == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  qsa::LaunchScoresTopk a{dtype == QSA_BF16, outIdx, qNormed, kbar, contextLengths, batchSize, seqLen, numBlocks,
                          rowStart, numRows, score_scale(), d.num_sms, reinterpret_cast<cudaStream_t>(stream)};
  return launched(fn, qsa::launch_scores_topk_fused(a));
}

namespace {
int validate_pool(const char* fn, const qsa_pool_state_t* ps, qsa::PoolDev* out) {
  if (!ps || !ps->poolPtr || !ps->pageTable) return fail(QSA_E_NULL, "%s: null pool state or pool pointer", fn);
  if (ps->maxPagesPerSeq < 1 || ps->numPages < 1 || ps->numKVHeads < 1 || ps->headSize < 0 ||
      ps->headSize + 128 > ps->poolHeadDim)
    return fail(QSA_E_SHAPE, "%s: pool needs maxPagesPerSeq, numPages, numKVHeads >= 1 and headSize + 128 <= poolHeadDim", fn);
  if (ps->headSize % 8 != 0 || ps->poolHeadDim % 8 != 0 || !aligned(ps->poolPtr, 16) || !aligned(ps->pageTable, 4))
    return fail(QSA_E_ALIGN, "%s: pool tails must be 16-byte aligned (headSize, poolHeadDim multiples of 8)", fn);
  *out = qsa::PoolDev{static_cast<uint16_t*>(ps->poolPtr), ps->pageTable, ps->maxPagesPerSeq, ps->numPages,
                      ps->numKVHeads, ps->poolHeadDim, ps->headSize};
  return QSA_OK;
}
}  // namespace

QSA_API int qsa_index_k_compress_paged(qsa_dtype_t dtype, void* kbar, const void* indexQk, const float* cosSin,
                                       const int32_t* contextLengths, const void* wK, float rmsEps,
                                       const qsa_pool_state_t* pool, int32_t batchSize, int32_t seqLen,
                                       int32_t numBlocks, int32_t blockBegin, int32_t blockEnd, int32_t pastLen,
                                       qsa_stream_t stream) {
  static const char* fn = "qsa_index_k_compress_paged";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!kbar || !indexQk || !cosSin || !contextLengths || !wK) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  qsa::PoolDev pd;
  if ((st = validate_pool(fn, pool, &pd)) != QSA_OK) return st;
  if (batchSize < 1 || seqLen < 1 || numBlocks < 1)
    return fail(QSA_E_SHAPE, "%s: batchSize=%d seqLen=%d numBlocks=%d must be >= 1", fn, batchSize, seqLen, numBlocks);
  if (static_cast<int64_t>(batchSize) * seqLen > INT32_MAX)
    return fail(QSA_E_SHAPE, "%s: batchSize*seqLen exceeds INT32_MAX", fn);
  if (blockBegin < 0 || blockBegin > blockEnd || blockEnd > numBlocks || pastLen < 0)
    return fail(QSA_E_RANGE, "%s: need 0 <= blockBegin=%d <= blockEnd=%d <= numBlocks=%d and pastLen=%d >= 0", fn,
                blockBegin, blockEnd, numBlocks, pastLen);
  if (!aligned(kbar, 16) || !aligned(indexQk, 16) || !aligned(cosSin, 16) || !aligned(wK, 16) ||
      !aligned(contextLengths, 4))
    return fail(QSA_E_ALIGN, "%s: T and FP32 arrays must be 16-byte aligned, contextLengths 4-byte", fn);
  if (blockBegin == blockEnd) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  qsa::LaunchKCompressPaged a{{dtype == QSA_BF16, kbar, indexQk, cosSin, contextLengths, wK, rmsEps, batchSize, seqLen,
                               numBlocks, blockBegin, blockEnd, pastLen, d.num_sms,
                               reinterpret_cast<cudaStream_t>(stream)},
                              pd};
  return launched(fn, qsa::launch_k_compress_paged(a));
}

QSA_API int qsa_raw_k_tail_write_prefill(qsa_dtype_t dtype, const void* indexQk, const int32_t* contextLengths,
                                         const qsa_pool_state_t* pool, int32_t batchSize, int32_t seqLen,
                                         qsa_stream_t stream) {
  static const char* fn = "qsa_raw_k_tail_write_prefill";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!indexQk || !contextLengths) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  qsa::PoolDev pd;
  if ((st = validate_pool(fn, pool, &pd)) != QSA_OK) return st;
  if (batchSize < 1 || seqLen < 1) return fail(QSA_E_SHAPE, "%s: batchSize=%d seqLen=%d must be >= 1", fn, batchSize, seqLen);
  if (static_cast<int64_t>(batchSize) * seqLen > INT32_MAX)
    return fail(QSA_E_SHAPE, "%s: batchSize*seqLen exceeds INT32_MAX", fn);
  if (!aligned(indexQk, 16) || !aligned(contextLengths, 4))
    return fail(QSA_E_ALIGN, "%s: indexQk must be 16-byte aligned, contextLengths 4-byte", fn);
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  return launched(fn, qsa::launch_raw_k_tail_write_prefill(dtype == QSA_BF16, indexQk, contextLengths, pd, batchSize,
                                                           seqLen, reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_indexer_pre_decode(qsa_dtype_t dtype, void* qNormed, const void* indexQk, const float* cosSin,
                                   const int32_t* contextLengths, const void* wQ, const void* wK, float rmsEps,
                                   const qsa_pool_state_t* pool, int32_t batchSize, qsa_stream_t stream) {
  static const char* fn = "qsa_indexer_pre_decode";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!qNormed || !indexQk || !cosSin || !contextLengths || !wQ || !wK)
    return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  qsa::PoolDev pd;
  if ((st = validate_pool(fn, pool, &pd)) != QSA_OK) return st;
  if (batchSize < 1) return fail(QSA_E_SHAPE, "%s: batchSize=%d must be >= 1", fn, batchSize);
  if (!aligned(qNormed, 16) || !aligned(indexQk, 16) || !aligned(cosSin, 16) || !aligned(wQ, 16) ||
      !aligned(wK, 16) || !aligned(contextLengths, 4))
    return fail(QSA_E_ALIGN, "%s: T and FP32 arrays must be 16-byte aligned, contextLengths 4-byte", fn);
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  return launched(fn, qsa::launch_pre_decode(dtype == QSA_BF16, qNormed, indexQk, cosSin, contextLengths, wQ, wK,
                                             rmsEps, pd, batchSize, reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_index_scores_decode(qsa_dtype_t dtype, float* logits, const void* qNormed,
                                    const int32_t* contextLengths, const qsa_pool_state_t* pool, int32_t batchSize,
                                    int32_t maxBlocks, qsa_stream_t stream) {
  static const char* fn = "qsa_index_scores_decode";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!logits || !qNormed || !contextLengths) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  qsa::PoolDev pd;
  if ((st = validate_pool(fn, pool, &pd)) != QSA_OK) return st;
  if (batchSize < 1 || maxBlocks < 1 || maxBlocks > 65535 * 256)
    return fail(QSA_E_SHAPE, "%s: batchSize=%d >= 1 and 1 <= maxBlocks=%d <= 16776960 required", fn, batchSize, maxBlocks);
  if (!aligned(qNormed, 16) || !aligned(logits, 4) || !aligned(contextLengths, 4))
    return fail(QSA_E_ALIGN, "%s: qNormed must be 16-byte aligned, logits/contextLengths 4-byte", fn);
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  return launched(fn, qsa::launch_scores_decode(dtype == QSA_BF16, logits, qNormed, contextLengths, pd, batchSize,
                                                maxBlocks, score_scale(), reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_topk_expand_decode(int32_t* outIdx, const float* logits, const int32_t* contextLengths,
                                   int32_t* splitCounters, int32_t numKVHeads, int32_t batchSize, int32_t maxBlocks,
                                   qsa_stream_t stream) {
  static const char* fn = "qsa_topk_expand_decode";
  if (!outIdx || !logits || !contextLengths) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (batchSize < 1 || maxBlocks < 1) return fail(QSA_E_SHAPE, "%s: batchSize=%d maxBlocks=%d must be >= 1", fn, batchSize, maxBlocks);
  if (splitCounters && numKVHeads < 0) return fail(QSA_E_SHAPE, "%s: numKVHeads=%d must be >= 0", fn, numKVHeads);
  if (maxBlocks > qsa::topk_max_blocks())
    return fail(QSA_E_SHAPE, "%s: maxBlocks=%d above %d", fn, maxBlocks, qsa::topk_max_blocks());
  if (!aligned(outIdx, 4) || !aligned(logits, 4) || !aligned(contextLengths, 4) || !aligned(splitCounters, 4))
    return fail(QSA_E_ALIGN, "%s: arrays must be 4-byte aligned", fn);
  DeviceInfo d;
  int st = current_device(fn, &d);
  if (st != QSA_OK) return st;
  return launched(fn, qsa::launch_topk_expand_decode(outIdx, logits, contextLengths, splitCounters,
                                                     splitCounters ? numKVHeads : 0, batchSize, maxBlocks,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_indexer_decode_step(qsa_dtype_t dtype, int32_t* outIdx, float* logits, void* qNormed,
                                    const void* indexQk, const float* cosSin, const int32_t* contextLengths,
                                    const void* wQ, const void* wK, float rmsEps, const qsa_pool_state_t* pool,
                                    int32_t* splitCounters, int32_t numKVHeads, int32_t batchSize,
                                    int32_t maxBlocks, qsa_stream_t stream) {
  static const char* fn = "qsa_indexer_decode_step";
  int st;
  if ((st = check_dtype(fn, dtype)) != QSA_OK) return st;
  if (!outIdx || !logits || !qNormed || !indexQk || !cosSin || !contextLengths || !wQ || !wK)
    return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  qsa::PoolDev pd;
  if ((st = validate_pool(fn, pool, &pd)) != QSA_OK) return st;
  if (batchSize < 1 || batchSize > qsa::decode_step_max_batch())
    return fail(QSA_E_SHAPE, "%s: batchSize=%d must be in [1, %d]", fn, batchSize, qsa::decode_step_max_batch());
  if (maxBlocks < 1 || maxBlocks > qsa::topk_max_blocks())
    return fail(QSA_E_SHAPE, "%s: maxBlocks=%d must be in [1, %d]", fn, maxBlocks, qsa::topk_max_blocks());
  if (splitCounters && numKVHeads < 0) return fail(QSA_E_SHAPE, "%s: numKVHeads=%d must be >= 0", fn, numKVHeads);
  if (!aligned(qNormed, 16) || !aligned(indexQk, 16) || !aligned(cosSin, 16) || !aligned(wQ, 16) ||
      !aligned(wK, 16) || !aligned(contextLengths, 4) || !aligned(logits, 4) || !aligned(outIdx, 4) ||
      !aligned(splitCounters, 4))
    return fail(QSA_E_ALIGN, "%s: T and cosSin arrays must be 16-byte aligned, the others 4-byte", fn);
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  return launched(fn, qsa::launch_decode_step(dtype == QSA_BF16, outIdx, logits, qNormed, indexQk, cosSin,
                                              contextLengths, wQ, wK, rmsEps, pd, splitCounters,
                                              splitCounters ? numKVHeads : 0, batchSize, maxBlocks, score_scale(),
                                              reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_testing_bounded_wait_probe(int32_t timeoutMs, qsa_stream_t stream) {
  static const char* fn = "qsa_testing_bounded_wait_probe";
  if (timeoutMs < 1 || timeoutMs > 10000) return fail(QSA_E_RANGE, "%s: timeoutMs must be in [1, 10000]", fn);
  DeviceInfo d;
  int st = current_device(fn, &d);
  if (st != QSA_OK) return st;
  return launched(fn, qsa::launch_bounded_wait_probe(static_cast<uint64_t>(timeoutMs) * 1000000ull,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_testing_index_scores_cuda_core(qsa_dtype_t dtype, float* logits, const void* qNormed,
                                               const void* kbar, const int32_t* contextLengths,
                                               int32_t batchSize, int32_t seqLen, int32_t numBlocks,
                                               int32_t rowStart, int32_t numRows, qsa_stream_t stream) {
  static const char* fn = "qsa_testing_index_scores_cuda_core";
  int st = validate_scores(fn, dtype, logits, qNormed, kbar, contextLengths, batchSize, seqLen, numBlocks,
                           rowStart, numRows);
  if (st != QSA_OK) return st;
  if (numRows == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  if (numBlocks > 65535 * 128) return fail(QSA_E_SHAPE, "%s: numBlocks too large for the CUDA-core grid", fn);
  DeviceInfo d;
  if ((st = current_device(fn, &d)) != QSA_OK) return st;
  qsa::LaunchScores a{dtype == QSA_BF16, logits, qNormed, kbar, contextLengths, batchSize, seqLen,
                      numBlocks, rowStart, numRows, score_scale(), d.num_sms,
                      reinterpret_cast<cudaStream_t>(stream)};
  return launched(fn, qsa::launch_scores_cc(a));
}

QSA_API int qsa_testing_stream_yardstick(void* dst, const void* src, int64_t units, int32_t rows, int64_t rowPitch,
                                         int64_t unitPitch, int64_t offset, int32_t bytes, qsa_stream_t stream) {
  static const char* fn = "qsa_testing_stream_yardstick";
  if (!dst || !src) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (units < 0 || rows < 1 || rows > qsa::yardstick_max_rows() || bytes < 16 || bytes > 1024 || bytes % 16 != 0 ||
      rowPitch < 0 || unitPitch < 0 || offset < 0)
    return fail(QSA_E_SHAPE, "%s: need units >= 0, 1 <= rows <= %d, bytes a multiple of 16 in [16, 1024]", fn,
                qsa::yardstick_max_rows());
  if (!aligned(dst, 16) || !aligned(src, 16) || rowPitch % 16 != 0 || unitPitch % 16 != 0 || offset % 16 != 0)
    return fail(QSA_E_ALIGN, "%s: pointers, pitches and offset must be 16-byte aligned", fn);
  if (units == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  int st = current_device(fn, &d);
  if (st != QSA_OK) return st;
  return launched(fn, qsa::launch_stream_yardstick(dst, src, units, rows, rowPitch, unitPitch, offset, bytes,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_testing_gather_yardstick(void* dst, const void* src, int64_t units, int64_t unitPitch, int64_t offset,
                                         int32_t bytes, qsa_stream_t stream) {
  static const char* fn = "qsa_testing_gather_yardstick";
  if (!dst || !src) return fail(QSA_E_NULL, "%s: null pointer argument", fn);
  if (units < 0 || bytes < 16 || bytes > 512 || (bytes & (bytes - 1)) != 0 || unitPitch < 0 || offset < 0)
    return fail(QSA_E_SHAPE, "%s: need units >= 0, bytes a power of two in [16, 512]", fn);
  if (!aligned(dst, 4) || !aligned(src, 16) || unitPitch % 16 != 0 || offset % 16 != 0)
    return fail(QSA_E_ALIGN, "%s: src, unitPitch and offset must be 16-byte aligned, dst 4-byte", fn);
  if (units == 0) {
    g_last_error[0] = '\0';
    return QSA_OK;
  }
  DeviceInfo d;
  int st = current_device(fn, &d);
  if (st != QSA_OK) return st;
  return launched(fn, qsa::launch_gather_yardstick(dst, src, units, unitPitch, offset, bytes,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_testing_decode_step_histograms(int32_t add, qsa_stream_t stream) {
  static const char* fn = "qsa_testing_decode_step_histograms";
  if (add < 0) return fail(QSA_E_RANGE, "%s: add must be >= 0", fn);
  DeviceInfo d;
  int st = current_device(fn, &d);
  if (st != QSA_OK) return st;
  return launched(fn, qsa::testing_decode_step_histograms(add, reinterpret_cast<cudaStream_t>(stream)));
}

QSA_API int qsa_device_fault_flags(uint32_t* flags, int clear, qsa_stream_t stream) {
  static const char* fn = "qsa_device_fault_flags";
  if (!flags) return fail(QSA_E_NULL, "%s: null flags pointer", fn);
  DeviceInfo d;
  int st = current_device(fn, &d);
  if (st != QSA_OK) return st;
  uint32_t k2 = 0, k1 = 0, dec = 0, step = 0, fused = 0;
  const auto cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = qsa::read_fault_flags(&k2, clear != 0, cs);
  if (e == cudaSuccess) e = qsa::read_k1_fault_flags(&k1, clear != 0, cs);
  if (e == cudaSuccess) e = qsa::read_dec_fault_flags(&dec, clear != 0, cs);
  if (e == cudaSuccess) e = qsa::read_step_fault_flags(&step, clear != 0, cs);
  if (e == cudaSuccess) e = qsa::read_fused_fault_flags(&fused, clear != 0, cs);
  if (e != cudaSuccess) return fail(QSA_E_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  *flags = k2 | (k1 << 8) | (dec << 16) | (step << 20) | (fused << 24);
  g_last_error[0] = '\0';
  return QSA_OK;
}

namespace qsa {

cudaError_t occupancy_blocks_per_sm(const void* kernel, int threads, size_t smem, int* out) {
  struct Entry {
    const void* kernel;
    int device, threads;
    size_t smem;
    int blocks;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < used; ++i) {
    if (cache[i].kernel == kernel && cache[i].device == dev && cache[i].threads == threads && cache[i].smem == smem) {
      *out = cache[i].blocks;
      return cudaSuccess;
    }
  }
  int blocks = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (blocks < 1) blocks = 1;
  if (used < 64) cache[used++] = Entry{kernel, dev, threads, smem, blocks};
  *out = blocks;
  return cudaSuccess;
}

}  // namespace qsa
