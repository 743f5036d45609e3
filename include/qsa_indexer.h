/*
 * qsa_indexer.h -- C ABI of the GB300 (sm_103a) QSA sparse-attention indexer.
 *
 * Operations are those of the "Qsa Indexer Kernels" page (TensorRT-Edge-LLM C++
 * API, cpp_api/kernels/qsaIndexerKernels.html): launchQsaIndexQPrep (K1a),
 * launchQsaIndexKCompress (K1b) and launchQsaIndexScores (K2).  Arguments mirror
 * the page one for one; a dtype enum replaces the C++ template parameter T and a
 * status code replaces std::runtime_error.
 *
 * Conventions shared by every entry point
 *  - T is the 2-byte activation type named by `dtype`: QSA_BF16 or QSA_F16.
 *  - Every array argument is a DEVICE pointer owned by the caller; scalars are
 *    host values.  The library allocates nothing, never synchronises (except
 *    qsa_device_fault_flags), and enqueues its kernels on `stream` only
 *    (0 = the legacy default stream).  Kernels are compiled ahead of time for
 *    sm_103a: there is no JIT step.  The first scoring call on a device does a
 *    one-time host-side set-up (kernel attribute, static-array address).
 *  - Arguments are validated on the host before anything is enqueued; device
 *    data (contextLengths) is never read on the host.  On a non-zero status
 *    nothing was enqueued (except QSA_E_CUDA from a failed launch) and
 *    qsa_last_error() returns a message for the calling thread.
 *  - Every array must be 16-byte aligned (torch allocations are); a misaligned
 *    pointer returns QSA_E_ALIGN.
 *  - Empty work (blockBegin == blockEnd, numRows == 0) returns QSA_OK and
 *    enqueues nothing.
 *  - "Exact zeros" are +0.0 in every element.  -FLT_MAX is the binary32 pattern
 *    0xFF7FFFFF.
 */
#ifndef QSA_INDEXER_H
#define QSA_INDEXER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* qsa_stream_t;

typedef enum {
  QSA_BF16 = 0, /* __nv_bfloat16 */
  QSA_F16 = 1   /* half */
} qsa_dtype_t;

typedef enum {
  QSA_OK = 0,
  QSA_E_NULL = -1,  /* a required pointer is null */
  QSA_E_SHAPE = -2, /* a size is out of range (batchSize, seqLen, numBlocks) */
  QSA_E_RANGE = -3, /* a block/row range or pastLen is out of range */
  QSA_E_DTYPE = -4, /* dtype is not QSA_BF16 or QSA_F16 */
  QSA_E_ALIGN = -5, /* a pointer is not 16-byte aligned */
  QSA_E_CUDA = -6,  /* a CUDA runtime call or kernel launch failed */
  QSA_E_DEVICE = -7 /* the current device is not an sm_103 GPU */
} qsa_status_t;

#define QSA_ABI_VERSION 1
#define QSA_HEAD_DIM 128
#define QSA_NUM_Q_HEADS 4
#define QSA_INDEX_QK_WIDTH 640 /* 4 q heads x 128, then the raw index-K x 128 */
#define QSA_COMPRESS_RATIO 4   /* tokens per compressed block */

/* QSA_ABI_VERSION of the loaded library. */
int qsa_abi_version(void);

/* Message for the calling thread's most recent non-OK status ("" if none). */
const char* qsa_last_error(void);

/*
 * K1a, launchQsaIndexQPrep: Gemma-style q-norm plus partial neox rope.
 *
 *  qNormed        [out] T [batchSize, seqLen, 4, 128], contiguous.
 *  indexQk        [in]  T [batchSize, seqLen, 640]; per row 4 q heads x 128, then
 *                       the raw k x 128 (unused here).
 *  cosSin         [in]  FP32 [maxPositions, 64], maxPositions >= seqLen; cos in
 *                       columns 0..31, sin in 32..63; row t is rope position t.
 *  contextLengths [in]  INT32 [batchSize], 0 <= contextLengths[b] <= seqLen.
 *  wQ             [in]  T [128], the RAW checkpoint gamma (the kernel applies 1+w).
 *  rmsEps         RMS-norm epsilon.
 *
 * Per row (b, t) with t < contextLengths[b] and per head h, in FP32:
 *   meanSq = sum_d x_d^2 / 128 (warp reduction), r = rsqrtf(meanSq + rmsEps),
 *   y_d = x_d * r * (1 + w_d); for i < 32 the pair (y_i, y_{i+32}) becomes
 *   (y_i*cos - y_{i+32}*sin, y_{i+32}*cos + y_i*sin) with cos = cosSin[t][i],
 *   sin = cosSin[t][32+i]; dims 64..127 pass through; one cast to T at the end.
 * Rows with t >= contextLengths[b] are written as exact zeros and never read.
 *
 * Errors: QSA_E_NULL, QSA_E_DTYPE, QSA_E_SHAPE (batchSize < 1, seqLen < 1),
 *         QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_index_q_prep(qsa_dtype_t dtype, void* qNormed, const void* indexQk,
                     const float* cosSin, const int32_t* contextLengths, const void* wQ,
                     float rmsEps, int32_t batchSize, int32_t seqLen, qsa_stream_t stream);

/*
 * K1b, launchQsaIndexKCompress: 4-token block compression of the raw index-K,
 * then the K1a norm (with wK) and rope at position 4g.
 *
 *  kbar           [out] T [batchSize, numBlocks, 128]; only rows g in
 *                       [blockBegin, blockEnd) are written, the rest untouched.
 *  indexQk        [in]  T [batchSize, seqLen, 640]; the raw k is columns 512..639.
 *                       Row i holds token pastLen + i.
 *  cosSin         [in]  FP32 [maxPositions, 64], maxPositions >= 4*blockEnd - 3.
 *  contextLengths [in]  INT32 [batchSize], the TOTAL length (past + new).
 *  wK             [in]  T [128], raw checkpoint gamma.
 *  numBlocks      row stride of kbar: ceilDiv(maxTotalLen, 4).
 *  blockBegin, blockEnd  0 <= blockBegin <= blockEnd <= numBlocks.
 *  pastLen        tokens already cached before indexQk row 0 (0 in prefill), >= 0.
 *
 * Block (b, g) is valid iff 4g+3 < contextLengths[b], 4g >= pastLen and
 * 4g+3-pastLen < seqLen (complete and fully inside the provided rows).  A valid
 * block computes per dim m = T((((k0+k1)+k2)+k3) * 0.25f) in FP32 in that fixed
 * order, with k_j the raw k of indexQk row 4g+j-pastLen; then the K1a math on
 * the re-loaded m with wK at rope position 4g; one cast.  Invalid blocks are
 * exact zeros and their rows are never read.  The result of a block does not
 * depend on the range or pastLen it was computed in (sub-range bit-parity).
 *
 * Errors: QSA_E_NULL, QSA_E_DTYPE, QSA_E_SHAPE (batchSize < 1, seqLen < 1,
 *         numBlocks < 1), QSA_E_RANGE (block range, pastLen < 0), QSA_E_ALIGN,
 *         QSA_E_CUDA.
 */
int qsa_index_k_compress(qsa_dtype_t dtype, void* kbar, const void* indexQk,
                         const float* cosSin, const int32_t* contextLengths, const void* wK,
                         float rmsEps, int32_t batchSize, int32_t seqLen, int32_t numBlocks,
                         int32_t blockBegin, int32_t blockEnd, int32_t pastLen,
                         qsa_stream_t stream);

/*
 * K2, launchQsaIndexScores: causal block-relevance logits for a chunk of rows,
 * on the tcgen05 tensor cores (FP32 accumulation of T products).
 *
 *  logits         [out] FP32 [numRows, numBlocks], chunk-local: row r - rowStart.
 *  qNormed        [in]  T [batchSize, seqLen, 4, 128] (from qsa_index_q_prep).
 *  kbar           [in]  T [batchSize, numBlocks, 128] (from qsa_index_k_compress).
 *  contextLengths [in]  INT32 [batchSize].
 *  numBlocks      ceilDiv(seqLen, 4) or more (extra columns are masked).
 *  rowStart, numRows  global rows r = b*seqLen + t in [rowStart, rowStart+numRows),
 *                 rowStart >= 0, rowStart + numRows <= batchSize*seqLen.
 *
 * For a row with 0 < contextLengths[b] and t < contextLengths[b]:
 *   logits[g] = (1/sqrtf(128)) * sum_{h=0..3, ascending} max(0, q_h . kbar[b][g])
 *   for g < (t+1)/4 (block fully before or at t), else -FLT_MAX.
 * Padded rows are -FLT_MAX everywhere and their q rows are ignored.
 *
 * Work is handed out by a device-side counter pair; calls take turns through 64
 * such pairs per device and each launch resets its pair when it ends, so at most
 * 64 launches may be in flight on one device at a time.  A CUDA graph that
 * captured a launch keeps that launch's pair on every replay, so one captured
 * graph must not be replayed concurrently with itself (for example on two
 * streams at once); replays in stream order are fine.
 *
 * Errors: QSA_E_NULL, QSA_E_DTYPE, QSA_E_SHAPE (batchSize < 1, seqLen < 1,
 *         numBlocks < ceilDiv(seqLen, 4)), QSA_E_RANGE (row range), QSA_E_ALIGN,
 *         QSA_E_CUDA, QSA_E_DEVICE.
 */
int qsa_index_scores(qsa_dtype_t dtype, float* logits, const void* qNormed, const void* kbar,
                     const int32_t* contextLengths, int32_t batchSize, int32_t seqLen,
                     int32_t numBlocks, int32_t rowStart, int32_t numRows,
                     qsa_stream_t stream);

/*
 * qsa_index_qk_prep: qsa_index_q_prep and the prefill qsa_index_k_compress
 * (blockBegin = 0, blockEnd = ceilDiv(seqLen, 4), pastLen = 0) in one pass over
 * indexQk ("Qsa Indexer Kernels": launchQsaIndexQPrep and launchQsaIndexKCompress
 * as the prefill pipeline calls them).  Outputs are bit-identical to the two
 * separate calls; each 1280-byte indexQk row is read once instead of in two
 * slices.
 *
 *  qNormed  [out] T [batchSize, seqLen, 4, 128]
 *  kbar     [out] T [batchSize, numBlocks, 128]; rows [0, ceilDiv(seqLen, 4)) written,
 *                 numBlocks >= ceilDiv(seqLen, 4) is the row stride
 *  other arguments as qsa_index_q_prep / qsa_index_k_compress; contextLengths[b]
 *  is the length of sequence b (0 <= ctx <= seqLen).
 *
 * Errors: QSA_E_NULL, QSA_E_DTYPE, QSA_E_SHAPE, QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_index_qk_prep(qsa_dtype_t dtype, void* qNormed, void* kbar, const void* indexQk,
                      const float* cosSin, const int32_t* contextLengths, const void* wQ,
                      const void* wK, float rmsEps, int32_t batchSize, int32_t seqLen,
                      int32_t numBlocks, qsa_stream_t stream);

#define QSA_TOPK_BLOCKS 512
#define QSA_INDEX_WIDTH 2051 /* QSA_TOPK_BLOCKS * 4 + 3 */

/*
 * K3, launchQsaIndexIdsFill: ids[r * numBlocks + c] = c for r < numRows, the value
 * array of a segmented sort.  ids: [out] INT32 [numRows, numBlocks].
 * Errors: QSA_E_NULL, QSA_E_SHAPE, QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_index_ids_fill(int32_t* ids, int32_t numRows, int32_t numBlocks, qsa_stream_t stream);

/*
 * K4, launchQsaIndexExpand: for global rows r = b*seqLen + t in [rowStart,
 * rowStart + numRows), with nVis = (t+1)/4, kSel = min(512, nVis),
 * tail = (t+1) % 4:
 *   outIdx[r][4i + j]    = sortedIds[r - rowStart][i] * 4 + j   for i < kSel, j < 4
 *   outIdx[r][4kSel + j] = 4*nVis + j                           for j < tail
 *   outIdx[r][k]         = -1                                   elsewhere (width 2051)
 * Padded rows (t >= contextLengths[b] or contextLengths[b] <= 0) are all -1 and
 * sortedIds is not read for them.
 *  outIdx    [out] INT32 [batchSize*seqLen, 2051]; only the chunk's rows are written
 *  sortedIds [in]  INT32 [numRows, numBlocks], chunk-local, block ids by descending logit
 * Errors: QSA_E_NULL, QSA_E_SHAPE, QSA_E_RANGE, QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_index_expand(int32_t* outIdx, const int32_t* sortedIds, const int32_t* contextLengths,
                     int32_t batchSize, int32_t seqLen, int32_t numBlocks, int32_t rowStart,
                     int32_t numRows, qsa_stream_t stream);

/*
 * The prefill selection of the page (qsa_index_ids_fill, a stable descending
 * segmented sort of the chunk's logits with the ids as values, qsa_index_expand)
 * in one kernel, with no sort and no workspace.  Per row: the FP32 logits of the
 * visible blocks g < nVis are mapped to order-preserving u32 keys
 * (bits >= 0 ? bits | 0x80000000 : ~bits); an MSB-first radix select finds
 * the kSel-th largest key; keys above it are selected, and keys equal to it in
 * ascending block order until kSel are selected.  That is exactly the set of
 * blocks the three-step pipeline puts first (and the rule of the page's decode
 * top-k).  The selected blocks are emitted in ascending block order, as the
 * decode path emits them (the page's token ids are "unsorted"), then expanded:
 * out[4i + j] = sel[i]*4 + j, the causal tail, -1 to width 2051.
 *  outIdx [out] INT32 [batchSize*seqLen, 2051] (chunk rows written)
 *  logits [in]  FP32 [numRows, numBlocks], chunk-local (qsa_index_scores' output)
 * Limit: numBlocks <= 65536.
 * Errors: QSA_E_NULL, QSA_E_SHAPE, QSA_E_RANGE, QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_index_topk_expand(int32_t* outIdx, const float* logits, const int32_t* contextLengths,
                          int32_t batchSize, int32_t seqLen, int32_t numBlocks, int32_t rowStart,
                          int32_t numRows, qsa_stream_t stream);

/*
 * The prefill scores of qsa_index_scores and the selection of qsa_index_topk_expand
 * in one kernel, which never writes the FP32 logits ("Qsa Indexer Kernels":
 * launchQsaIndexScores, then launchQsaIndexIdsFill, the stable descending segmented
 * sort and launchQsaIndexExpand; the fusion is an addition of this library).  For
 * the same arguments outIdx equals, bit for bit, what qsa_index_scores into a
 * logits buffer followed by qsa_index_topk_expand on that buffer writes: every
 * logit is computed by the same tensor-core tile and epilogue arithmetic, and the
 * same 512 blocks a row are selected (largest keys, equal keys by ascending block
 * id), emitted in ascending block order and expanded to 2051 token ids.
 * The kernel computes each 64-token tile's scores twice or more on the tensor cores
 * and keeps per-row histograms and bit masks in shared memory instead of the logits.
 *  outIdx  [out] INT32 [batchSize*seqLen, 2051]; only the rows [rowStart,
 *               rowStart + numRows) are written
 *  qNormed [in]  T [batchSize, seqLen, 4, 128], kbar [in] T [batchSize, numBlocks, 128]
 *               (16-byte aligned), as for qsa_index_scores
 * Limit: numBlocks <= 4096 (larger problems: the two calls).  Up to 64 launches may
 * be in flight on one device (device-side scheduler counters taken in turn), and one
 * captured graph must not be replayed concurrently with itself.
 * Errors: QSA_E_NULL, QSA_E_DTYPE, QSA_E_SHAPE, QSA_E_RANGE, QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_index_scores_topk_expand(qsa_dtype_t dtype, int32_t* outIdx, const void* qNormed, const void* kbar,
                                 const int32_t* contextLengths, int32_t batchSize, int32_t seqLen,
                                 int32_t numBlocks, int32_t rowStart, int32_t numRows, qsa_stream_t stream);

/*
 * QsaIndexerPoolState ("Qsa Indexer Kernels"): where the decode state lives.
 *  poolPtr      [2*numPages, 128, numKVHeads, poolHeadDim] T, element (page, row, head,
 *               col) at ((page*128 + row)*numKVHeads + head)*poolHeadDim + col
 *  pageTable    INT32 [B, 2, maxPagesPerSeq]: plane 0 = K pages, plane 1 = V pages
 *               (ids already offset by +numPages); -1 = unused
 * Token t's raw index-K tail: K page pageTable[b][0][t >> 7], row t & 127, head 0,
 * columns [headSize, headSize + 128).  Block g's kbar: V page pageTable[b][1][(4g) >> 7],
 * row (4g) & 127, head 0, same columns.  A slot past maxPagesPerSeq, an entry of -1 or
 * an id outside [0, 2*numPages) is never dereferenced: writes there are skipped.
 * Requirements: headSize + 128 <= poolHeadDim, headSize and poolHeadDim multiples of
 * 8, poolPtr 16-byte aligned.  The struct is a host object; its pointers are device
 * pointers.
 */
typedef struct {
  void* poolPtr;
  const int32_t* pageTable;
  int32_t maxPagesPerSeq;
  int32_t numPages;   /* K-plane page count */
  int32_t numKVHeads;
  int32_t poolHeadDim;
  int32_t headSize;   /* tail column offset */
} qsa_pool_state_t;

/*
 * launchQsaIndexKCompressPaged: qsa_index_k_compress, and every VALID block's kbar
 * row is also written to the V-tail of token 4g.  The dense kbar output is
 * bit-identical to qsa_index_k_compress; invalid blocks write dense zeros and never
 * touch the pool; unusable page slots skip the pool write only.
 * Errors: those of qsa_index_k_compress, plus QSA_E_NULL / QSA_E_SHAPE / QSA_E_ALIGN
 * for the pool state.
 */
int qsa_index_k_compress_paged(qsa_dtype_t dtype, void* kbar, const void* indexQk,
                               const float* cosSin, const int32_t* contextLengths, const void* wK,
                               float rmsEps, const qsa_pool_state_t* pool, int32_t batchSize,
                               int32_t seqLen, int32_t numBlocks, int32_t blockBegin,
                               int32_t blockEnd, int32_t pastLen, qsa_stream_t stream);

/*
 * launchQsaRawKTailWritePrefill: for each sequence, tokens t in
 * [ctx - ctx % 4, ctx) (the trailing incomplete block) copy indexQk row (b, t)
 * columns [512, 640) BIT-UNMODIFIED to their K-tails.  Nothing else in the pool is
 * touched.  0 <= contextLengths[b] <= seqLen.
 * Errors: QSA_E_NULL (indexQk, contextLengths, the pool state or its pointers),
 *         QSA_E_DTYPE, QSA_E_SHAPE (batchSize < 1, seqLen < 1, the pool sizes),
 *         QSA_E_ALIGN (indexQk 16-byte, contextLengths 4-byte, the pool tails),
 *         QSA_E_CUDA.
 */
int qsa_raw_k_tail_write_prefill(qsa_dtype_t dtype, const void* indexQk, const int32_t* contextLengths,
                                 const qsa_pool_state_t* pool, int32_t batchSize, int32_t seqLen,
                                 qsa_stream_t stream);

/*
 * launchQsaIndexerPreDecode: one new token per sequence; contextLengths[b] is the
 * TOTAL length including it, pos = ctx - 1.
 *  qNormed  [out] T [batchSize, 1, 4, 128]: qsa_index_q_prep numerics at rope
 *           position pos; exact zeros when ctx <= 0 (and nothing else is done).
 *  indexQk  [in]  T [batchSize, 1, 640]
 *  ctx % 4 != 0: the row's raw index-K goes bit for bit to the K-tail of pos.
 *  ctx % 4 == 0: block g = ctx/4 - 1 is complete: the raw keys of 4g..4g+2 are read
 *           from their K-tails, 4g+3 is the new row; qsa_index_k_compress numerics
 *           (bit-identical to prefill); the kbar row goes to the V-tail of 4g.  If
 *           any of those page slots is unusable the block is not written.
 *  cosSin   FP32 [maxPositions, 64], maxPositions >= max ctx.
 * Errors: QSA_E_NULL (any array, the pool state or its pointers), QSA_E_DTYPE,
 *         QSA_E_SHAPE (batchSize < 1, the pool sizes), QSA_E_ALIGN (T and FP32
 *         arrays 16-byte, contextLengths 4-byte, the pool tails), QSA_E_CUDA.
 */
int qsa_indexer_pre_decode(qsa_dtype_t dtype, void* qNormed, const void* indexQk, const float* cosSin,
                           const int32_t* contextLengths, const void* wQ, const void* wK, float rmsEps,
                           const qsa_pool_state_t* pool, int32_t batchSize, qsa_stream_t stream);

/*
 * launchQsaIndexScoresDecode: logits[b][g] = (1/sqrtf(128)) * sum_h relu(q[b][h] .
 * kbar[b][g]) (FP32, ascending h, scale after the sum) for g < nVis = ctx/4, with
 * kbar read from the V-tail of token 4g.  ONLY [0, nVis) of each row is written.  A
 * block whose V page slot is unusable scores -FLT_MAX.  The dots run on the tensor
 * cores with qsa_index_scores' MMA shape along K and K order, so each logit equals,
 * bit for bit, qsa_index_scores' logit of the same token given the same q and kbar.
 *  logits   [out] FP32 [batchSize, maxBlocks]; maxBlocks >= ceilDiv(max ctx, 4)
 *  qNormed  [in]  T [batchSize, 1, 4, 128] (qsa_indexer_pre_decode's output)
 * Limit: maxBlocks <= 16776960 (65535 * 256).
 * Errors: QSA_E_NULL (logits, qNormed, contextLengths, the pool state or its
 *         pointers), QSA_E_DTYPE, QSA_E_SHAPE (batchSize < 1, maxBlocks outside
 *         [1, 16776960], the pool sizes), QSA_E_ALIGN (qNormed 16-byte, logits and
 *         contextLengths 4-byte, the pool tails), QSA_E_CUDA.
 */
int qsa_index_scores_decode(qsa_dtype_t dtype, float* logits, const void* qNormed,
                            const int32_t* contextLengths, const qsa_pool_state_t* pool,
                            int32_t batchSize, int32_t maxBlocks, qsa_stream_t stream);

/*
 * launchQsaTopKExpandDecode, per sequence b (ctx = contextLengths[b], nVis = ctx/4,
 * kSel = min(512, nVis), tail = ctx % 4):
 *  splitCounters[b*numKVHeads .. +numKVHeads) are zeroed when splitCounters != NULL;
 *  nVis <= 512 selects every block (logits not read); otherwise keys above the
 *  kSel-th largest logit (order-preserving u32 map) and keys equal to it in
 *  ascending block order until kSel are selected (the set the prefill selection
 *  picks for identical logits); outIdx[b][4i + j] = sel[i]*4 + j with sel in
 *  ascending order, then tokens 4*nVis + j for j < tail, then -1 to width 2051.
 *  Deterministic: identical inputs give identical bits.
 *  outIdx  [out] INT32 [batchSize, 1, 2051];  logits [in] FP32 [batchSize, maxBlocks]
 *  (only [0, nVis) read).
 * Limit: maxBlocks <= 65536.
 * Errors: QSA_E_NULL (outIdx, logits, contextLengths; splitCounters may be NULL),
 *         QSA_E_SHAPE (batchSize < 1, maxBlocks outside [1, 65536], numKVHeads < 0
 *         with split counters), QSA_E_ALIGN (4-byte), QSA_E_CUDA.
 */
int qsa_topk_expand_decode(int32_t* outIdx, const float* logits, const int32_t* contextLengths,
                           int32_t* splitCounters, int32_t numKVHeads, int32_t batchSize, int32_t maxBlocks,
                           qsa_stream_t stream);

/*
 * The decode step in one launch: qsa_indexer_pre_decode, qsa_index_scores_decode and
 * qsa_topk_expand_decode, in that order, over the same arguments ("Qsa Indexer
 * Kernels": launchQsaIndexerPreDecode, launchQsaIndexScoresDecode,
 * launchQsaTopKExpandDecode).  Every output equals, bit for bit, the output of the three
 * calls: qNormed [B, 1, 4, 128], the pool's K- or V-tail of the new token, logits
 * [B, maxBlocks] (only g < nVis written), outIdx [B, 1, 2051] and the zeroed split
 * counters.  (The fusion is an addition of this library; the page has three launches.)
 * Each CTA computes its sequence's q heads once and scores a run of 128-block chunks
 * of that sequence (the run length sizes the grid to about one wave of resident
 * CTAs); the CTA that completes a sequence last runs its selection, so no CTA waits
 * for another.  For batches of up to 64 sequences, the scoring CTAs also count every
 * logit they write into the row's first-digit histogram of the selection, which the
 * last CTA copies instead of counting the row again (and leaves zeroed); if the copied
 * counts do not total the row's visible blocks (as after a launch whose waits ran out),
 * that CTA counts the row itself.  Sequences
 * report completion through a device-side set of counters (and of histograms), one of
 * 16 taken in turn by each launch: at most 16 launches may be in flight on one device
 * at a time, and a CUDA graph that captured a launch keeps its set on every replay, so
 * one captured graph must not be replayed concurrently with itself.  The sets are
 * module memory of the library (256 KB of counters, 4 MB of histograms a device),
 * zero at load; no call allocates.
 * Limits: batchSize <= 4096, maxBlocks <= 65536.
 * Errors: QSA_E_NULL, QSA_E_DTYPE, QSA_E_SHAPE, QSA_E_ALIGN, QSA_E_CUDA.
 */
int qsa_indexer_decode_step(qsa_dtype_t dtype, int32_t* outIdx, float* logits, void* qNormed,
                            const void* indexQk, const float* cosSin, const int32_t* contextLengths,
                            const void* wQ, const void* wK, float rmsEps, const qsa_pool_state_t* pool,
                            int32_t* splitCounters, int32_t numKVHeads, int32_t batchSize, int32_t maxBlocks,
                            qsa_stream_t stream);

/*
 * qsa_index_scores_no_alloc: the K2 scores of qsa_index_scores, for callers that
 * must not allocate device memory.  (No counterpart on the "Qsa Indexer Kernels"
 * page; an addition of this library.)
 *
 * Who needs it: code that cannot call cudaMalloc at the point of the call, such
 * as an inference engine whose memory manager owns every device allocation, code
 * recording work into a stream that is being captured (cudaMalloc is not a stream
 * operation and may synchronise the device), or a latency-critical path that
 * cannot afford the implicit synchronisation of cudaMalloc/cudaFree.
 *
 * Arguments, layouts, results, validation and error codes are those of
 * qsa_index_scores; the caller still passes every input and output.  The kernel's
 * scratch (its work-scheduler counters) lives in one fixed 256-byte static device
 * array that every GPU loading this library holds until the process exits; this
 * entry point never calls cudaMalloc, cudaFree or any allocating routine.
 *  - Every call on a device shares that array, which keeps the last call's
 *    contents.  Each call zeroes the counters on `stream` before its kernel, so
 *    calls that overlap on the GPU (for example on two streams) race on them and
 *    produce undefined logits: serialise them.
 *  - The first call on a device does a one-time set-up (looks up the array's
 *    device address and sets the kernel's shared-memory attribute) with that
 *    device current; make that first call before any stream capture begins.
 *  - Limit: the work-unit count, ceilDiv of the chunk's token tiles (64 tokens)
 *    times ceilDiv(numBlocks, 1024), must not exceed 2^31 - 65537; larger
 *    problems return QSA_E_SHAPE with a message.
 */
int qsa_index_scores_no_alloc(qsa_dtype_t dtype, float* logits, const void* qNormed,
                              const void* kbar, const int32_t* contextLengths, int32_t batchSize,
                              int32_t seqLen, int32_t numBlocks, int32_t rowStart, int32_t numRows,
                              qsa_stream_t stream);

/*
 * Device-side fault flags.  Kernels that wait on their own asynchronous copies
 * bound every wait (about two seconds); a wait that runs out sets a bit here
 * (bits 0-3: scoring kernel, bits 8-11: staged q-prep kernels, bits 16-19: paged
 * decode scores, bits 20-23: the one-launch decode step, bits 24-27: the fused
 * scores + selection)
 * instead of hanging, the kernel drains and returns, and the outputs of that
 * launch are undefined.  This call synchronises `stream`, copies the flags of
 * the current device into *flags (0 = no fault since the last clear) and clears
 * them when `clear` is non-zero.
 *
 * Errors: QSA_E_NULL (flags), QSA_E_CUDA.
 */
int qsa_device_fault_flags(uint32_t* flags, int clear, qsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_INDEXER_H */
