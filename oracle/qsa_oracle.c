/*
 * QSA indexer oracle: a plain, slow, single-threaded CPU restatement of what the
 * indexer hot path computes.  TEST INFRASTRUCTURE ONLY: it is used by tests/,
 * by __graft_entry__.smoke() and by bench.py's CPU-baseline leg, never by the
 * product path.  It shares no code, header or table with the CUDA library.
 *
 * Source of every formula: "Qsa Indexer Kernels" (TensorRT-Edge-LLM C++ API,
 * cpp_api/kernels/qsaIndexerKernels.html), the entries
 *   launchQsaIndexQPrep      (K1a: q-norm + partial neox rope),
 *   launchQsaIndexKCompress  (K1b: 4-token block mean, cast, norm, rope at 4g),
 *   launchQsaIndexScores     (K2: causal block-relevance logits).
 *
 * Arithmetic: IEEE binary32, one rounding per written operation, no fused
 * multiply-add (built with -ffp-contract=off), no reassociation.  Where the page
 * leaves an order open (the sum of squares of a "warp reduction", the order of
 * the 128-term dot product) this file sums sequentially in ascending index; the
 * GPU may use another order and is compared within a tolerance.  rsqrtf is read
 * as the correctly rounded 1.0f / sqrtf(v).  The single casts to T (bf16 or
 * fp16) are round-to-nearest-even, written out from the IEEE definitions below.
 *
 * Parity pins (tests/test_oracle_pins.py): the conversions are checked against
 * numpy/torch on every bf16/fp16 pattern; the norm against torch's rms_norm;
 * the rope against complex rotation; closed forms for one-hot inputs; the
 * zero-gamma, gamma=-1 and gamma=1 invariants; the 4-identical-rows and
 * (a,-a,b,-b) block cases; sub-range equivalence; relu-per-head, scale and
 * homogeneity of the scores; float64 brute force on tiny shapes.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <float.h>

#define QSA_HEAD_DIM 128
#define QSA_NUM_Q_HEADS 4
#define QSA_ROW_WIDTH 640          /* 4 q heads x 128, then raw k x 128 */
#define QSA_K_COL 512              /* first column of the raw index-K */
#define QSA_ROPE_HALF 32           /* rope pairs (i, i + 32) for i < 32 */
#define QSA_COMPRESS_RATIO 4       /* tokens per compressed block */

enum { ORACLE_BF16 = 0, ORACLE_F16 = 1 };

/* ---------------------------------------------------------------- conversions */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 is the upper half of a binary32: widening is exact. */
static float bf16_to_f32(uint16_t v) { return bits_f32((uint32_t)v << 16); }

/* binary32 -> bf16, round to nearest, ties to even; NaN stays a (quiet) NaN. */
static uint16_t f32_to_bf16(float f) {
  uint32_t u = f32_bits(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;  /* a carry into the exponent is the correct rounding, up to inf */
}

/* IEEE binary16 -> binary32, exact (normals, subnormals, zeros, inf, NaN). */
static float f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  uint32_t exp = (h >> 10) & 0x1fu;
  uint32_t man = h & 0x3ffu;
  if (exp == 0x1fu) return bits_f32(sign | 0x7f800000u | (man << 13));
  if (exp == 0) {
    /* subnormal or zero: value = man * 2^-24, exact in binary32 */
    float mag = (float)man * 0x1p-24f;
    return sign ? -mag : mag;
  }
  return bits_f32(sign | ((exp + 112u) << 23) | (man << 13));
}

/* binary32 -> binary16, round to nearest, ties to even, with subnormal results. */
static uint16_t f32_to_f16(float f) {
  uint32_t u = f32_bits(f);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  uint32_t a = u & 0x7fffffffu;
  if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u | ((a >> 13) & 0x3ffu));
  if (a >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u); /* >= 65520: rounds to inf */
  int32_t e = (int32_t)(a >> 23) - 127;                   /* unbiased exponent */
  uint32_t m = (a & 0x7fffffu) | (a >= 0x00800000u ? 0x800000u : 0u);
  if (a < 0x00800000u) e = -126;                          /* binary32 subnormal input */
  /* The result's quantum is 2^-24 for e < -14 (binary16 subnormal), else 2^(e-10).
     Express the input as m * 2^(e-23) and shift right by (quantum_exp - (e-23)). */
  int32_t q = (e < -14) ? -24 : e - 10;
  int32_t shift = q - (e - 23);                           /* >= 13 */
  uint32_t r;
  if (shift >= 32) {
    r = 0;                                                /* far below half a quantum */
  } else {
    uint32_t kept = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (kept & 1u))) kept += 1u;
    r = kept;
  }
  /* r counts quanta: for subnormal range it is the mantissa field directly (it may
     carry into the smallest normal, which the encoding handles); for normals it is
     1.mmmmmmmmmm with an implicit leading bit that may carry into the next binade. */
  if (e < -14) return (uint16_t)(sign | r);
  uint32_t biased = (uint32_t)(e + 15);
  uint32_t enc = (biased << 10) + (r - 0x400u);           /* carry into exponent is exact */
  return (uint16_t)(sign | enc);
}

float qsa_oracle_t_to_f32(int dtype, uint16_t v) {
  return dtype == ORACLE_BF16 ? bf16_to_f32(v) : f16_to_f32(v);
}

uint16_t qsa_oracle_f32_to_t(int dtype, float f) {
  return dtype == ORACLE_BF16 ? f32_to_bf16(f) : f32_to_f16(f);
}

void qsa_oracle_t_to_f32_array(int dtype, const uint16_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = qsa_oracle_t_to_f32(dtype, in[i]);
}

void qsa_oracle_f32_to_t_array(int dtype, const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = qsa_oracle_f32_to_t(dtype, in[i]);
}

/* ------------------------------------------------------ shared per-vector math */

/*
 * Gemma-style RMS norm with raw gamma plus one, then partial neox rope, then one
 * cast (launchQsaIndexQPrep, "Exact numerics"; reused verbatim by
 * launchQsaIndexKCompress after its block mean):
 *   meanSq = sum_d x_d^2 / 128
 *   y_d    = (x_d * (1 / sqrt(meanSq + eps))) * (1 + w_d)
 *   for i < 32: out_i = y_i*cos_i - y_{i+32}*sin_i ; out_{i+32} = y_{i+32}*cos_i + y_i*sin_i
 *   dims 64..127 pass through;  cos_i = cs[i], sin_i = cs[32 + i].
 */
void qsa_oracle_norm_rope(int dtype, const float* x, const uint16_t* w, float eps,
                          const float* cs, uint16_t* out) {
  float sumsq = 0.0f;
  for (int d = 0; d < QSA_HEAD_DIM; ++d) {
    float sq = x[d] * x[d];
    sumsq = sumsq + sq;
  }
  float meanSq = sumsq / 128.0f;
  float r = 1.0f / sqrtf(meanSq + eps);
  float y[QSA_HEAD_DIM];
  for (int d = 0; d < QSA_HEAD_DIM; ++d) {
    float g = 1.0f + qsa_oracle_t_to_f32(dtype, w[d]);
    float xr = x[d] * r;
    y[d] = xr * g;
  }
  float o[QSA_HEAD_DIM];
  for (int i = 0; i < QSA_ROPE_HALF; ++i) {
    float c = cs[i];
    float s = cs[QSA_ROPE_HALF + i];
    float x0 = y[i];
    float x1 = y[i + QSA_ROPE_HALF];
    float a = x0 * c;
    float b = x1 * s;
    float e = x1 * c;
    float f = x0 * s;
    o[i] = a - b;
    o[i + QSA_ROPE_HALF] = e + f;
  }
  for (int d = 2 * QSA_ROPE_HALF; d < QSA_HEAD_DIM; ++d) o[d] = y[d];
  for (int d = 0; d < QSA_HEAD_DIM; ++d) out[d] = qsa_oracle_f32_to_t(dtype, o[d]);
}

/*
 * Fixed-order block mean of four raw K rows and its bit-critical cast
 * (launchQsaIndexKCompress): m_d = T( (((k0+k1)+k2)+k3) * 0.25f ).
 */
void qsa_oracle_block_mean(int dtype, const uint16_t* k0, const uint16_t* k1,
                           const uint16_t* k2, const uint16_t* k3, uint16_t* m) {
  for (int d = 0; d < QSA_HEAD_DIM; ++d) {
    float s = qsa_oracle_t_to_f32(dtype, k0[d]) + qsa_oracle_t_to_f32(dtype, k1[d]);
    s = s + qsa_oracle_t_to_f32(dtype, k2[d]);
    s = s + qsa_oracle_t_to_f32(dtype, k3[d]);
    float mean = s * 0.25f;
    m[d] = qsa_oracle_f32_to_t(dtype, mean);
  }
}

/* ------------------------------------------------------------------------ K1a */

/*
 * launchQsaIndexQPrep: for each row (b, t) of indexQk [B, S, 640] write
 * qNormed [B, S, 4, 128].  Rows with t >= contextLengths[b] are exact zeros and
 * are never read.  The rope position is t.
 */
int qsa_oracle_q_prep(int dtype, uint16_t* qNormed, const uint16_t* indexQk,
                      const float* cosSin, const int32_t* contextLengths,
                      const uint16_t* wQ, float eps, int32_t B, int32_t S) {
  if (B < 0 || S < 0) return -2;
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t t = 0; t < S; ++t) {
      int64_t row = (int64_t)b * S + t;
      uint16_t* out = qNormed + row * (QSA_NUM_Q_HEADS * QSA_HEAD_DIM);
      if (t >= contextLengths[b]) {
        memset(out, 0, sizeof(uint16_t) * QSA_NUM_Q_HEADS * QSA_HEAD_DIM);
        continue;
      }
      const uint16_t* in = indexQk + row * QSA_ROW_WIDTH;
      for (int h = 0; h < QSA_NUM_Q_HEADS; ++h) {
        float x[QSA_HEAD_DIM];
        for (int d = 0; d < QSA_HEAD_DIM; ++d)
          x[d] = qsa_oracle_t_to_f32(dtype, in[h * QSA_HEAD_DIM + d]);
        qsa_oracle_norm_rope(dtype, x, wQ, eps, cosSin + (int64_t)t * 64,
                             out + h * QSA_HEAD_DIM);
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ K1b */

/*
 * Validity of block (b, g) (launchQsaIndexKCompress): complete and fully inside the
 * provided rows.  The page's formula is 4g+3 < ctx_b and 4g >= pastLen; its words
 * also say "fully inside the provided rows", read here as the extra condition
 * 4g+3-pastLen < seqLen (a no-op whenever ctx_b - pastLen <= seqLen holds).
 */
int qsa_oracle_block_valid(int32_t g, int32_t ctx, int32_t seqLen, int32_t pastLen) {
  int64_t first = (int64_t)QSA_COMPRESS_RATIO * g;
  int64_t last = first + (QSA_COMPRESS_RATIO - 1);
  return last < ctx && first >= pastLen && last - pastLen < seqLen;
}

/*
 * launchQsaIndexKCompress: for g in [blockBegin, blockEnd) write kbar[b][g][:]
 * (row stride numBlocks).  Valid blocks: fixed-order mean of indexQk rows
 * 4g+j-pastLen (j = 0..3), columns [512, 640); cast; norm with wK; rope at
 * position 4g; cast.  Invalid blocks are exact zeros; rows outside the range are
 * not touched.
 */
int qsa_oracle_k_compress(int dtype, uint16_t* kbar, const uint16_t* indexQk,
                          const float* cosSin, const int32_t* contextLengths,
                          const uint16_t* wK, float eps, int32_t B, int32_t S,
                          int32_t numBlocks, int32_t blockBegin, int32_t blockEnd,
                          int32_t pastLen) {
  if (blockBegin < 0 || blockEnd > numBlocks || blockBegin > blockEnd || pastLen < 0) return -3;
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t g = blockBegin; g < blockEnd; ++g) {
      uint16_t* out = kbar + ((int64_t)b * numBlocks + g) * QSA_HEAD_DIM;
      if (!qsa_oracle_block_valid(g, contextLengths[b], S, pastLen)) {
        memset(out, 0, sizeof(uint16_t) * QSA_HEAD_DIM);
        continue;
      }
      const uint16_t* k[QSA_COMPRESS_RATIO];
      for (int j = 0; j < QSA_COMPRESS_RATIO; ++j) {
        int64_t row = (int64_t)b * S + ((int64_t)QSA_COMPRESS_RATIO * g + j - pastLen);
        k[j] = indexQk + row * QSA_ROW_WIDTH + QSA_K_COL;
      }
      uint16_t m[QSA_HEAD_DIM];
      qsa_oracle_block_mean(dtype, k[0], k[1], k[2], k[3], m);
      float x[QSA_HEAD_DIM];
      for (int d = 0; d < QSA_HEAD_DIM; ++d) x[d] = qsa_oracle_t_to_f32(dtype, m[d]);
      qsa_oracle_norm_rope(dtype, x, wK, eps,
                           cosSin + (int64_t)QSA_COMPRESS_RATIO * g * 64, out);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------- K2 */

/*
 * One query row of launchQsaIndexScores.  q is that row's [4, 128] normed heads,
 * kb the sequence's kbar [numBlocks, 128], t the row's position, ctx its sequence's
 * context length.  out[g], g < numBlocks:
 *   padded row (ctx <= 0 or t >= ctx):  -FLT_MAX everywhere, q and kbar unread
 *   g >= (t + 1) / 4:                   -FLT_MAX
 *   otherwise: (1/sqrt(128)) * sum_{h ascending} max(0, sum_d q[h][d] * kb[g][d])
 */
void qsa_oracle_scores_row(int dtype, float* out, const uint16_t* q, const uint16_t* kb,
                           int32_t t, int32_t ctx, int32_t numBlocks) {
  if (ctx <= 0 || t >= ctx) {
    for (int32_t g = 0; g < numBlocks; ++g) out[g] = -FLT_MAX;
    return;
  }
  const float scale = 1.0f / sqrtf(128.0f);
  int32_t nVis = (t + 1) / QSA_COMPRESS_RATIO;
  float qf[QSA_NUM_Q_HEADS][QSA_HEAD_DIM];
  for (int h = 0; h < QSA_NUM_Q_HEADS; ++h)
    for (int d = 0; d < QSA_HEAD_DIM; ++d)
      qf[h][d] = qsa_oracle_t_to_f32(dtype, q[h * QSA_HEAD_DIM + d]);
  for (int32_t g = 0; g < numBlocks; ++g) {
    if (g >= nVis) { out[g] = -FLT_MAX; continue; }
    const uint16_t* k = kb + (int64_t)g * QSA_HEAD_DIM;
    float kf[QSA_HEAD_DIM];
    for (int d = 0; d < QSA_HEAD_DIM; ++d) kf[d] = qsa_oracle_t_to_f32(dtype, k[d]);
    float sum = 0.0f;
    for (int h = 0; h < QSA_NUM_Q_HEADS; ++h) {
      float dot = 0.0f;
      for (int d = 0; d < QSA_HEAD_DIM; ++d) {
        float p = qf[h][d] * kf[d];
        dot = dot + p;
      }
      float rel = fmaxf(0.0f, dot);
      sum = sum + rel;
    }
    out[g] = scale * sum;
  }
}

/*
 * launchQsaIndexScores over global rows r = b*S + t in [rowStart, rowStart+numRows);
 * logits is chunk-local [numRows, numBlocks].
 */
int qsa_oracle_scores(int dtype, float* logits, const uint16_t* qNormed, const uint16_t* kbar,
                      const int32_t* contextLengths, int32_t B, int32_t S, int32_t numBlocks,
                      int32_t rowStart, int32_t numRows) {
  if (rowStart < 0 || numRows < 0 || (int64_t)rowStart + numRows > (int64_t)B * S) return -3;
  for (int32_t i = 0; i < numRows; ++i) {
    int64_t r = (int64_t)rowStart + i;
    int32_t b = (int32_t)(r / S);
    int32_t t = (int32_t)(r - (int64_t)b * S);
    qsa_oracle_scores_row(dtype, logits + (int64_t)i * numBlocks,
                          qNormed + r * (QSA_NUM_Q_HEADS * QSA_HEAD_DIM),
                          kbar + (int64_t)b * numBlocks * QSA_HEAD_DIM,
                          t, contextLengths[b], numBlocks);
  }
  return 0;
}

/* --------------------------------------------------------- prefill selection */

#define QSA_TOPK_BLOCKS 512
#define QSA_INDEX_WIDTH (QSA_TOPK_BLOCKS * QSA_COMPRESS_RATIO + QSA_COMPRESS_RATIO - 1) /* 2051 */

/* Order-preserving map of binary32 bit patterns to unsigned integers
 * (launchQsaTopKExpandDecode): u = bits >= 0 ? bits | 0x80000000 : ~bits. */
uint32_t qsa_oracle_orderable(float f) {
  uint32_t b = f32_bits(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

/* launchQsaIndexIdsFill: ids[r * numBlocks + c] = c. */
void qsa_oracle_ids_fill(int32_t* ids, int32_t numRows, int32_t numBlocks) {
  for (int64_t r = 0; r < numRows; ++r)
    for (int32_t c = 0; c < numBlocks; ++c) ids[r * numBlocks + c] = c;
}

/* Stable merge sort of ids by key, descending (equal keys keep their input order). */
static void stable_sort_desc(uint32_t* key, int32_t* id, uint32_t* tk, int32_t* ti, int32_t n) {
  for (int32_t width = 1; width < n; width *= 2) {
    for (int32_t lo = 0; lo < n; lo += 2 * width) {
      int32_t mid = lo + width < n ? lo + width : n;
      int32_t hi = lo + 2 * width < n ? lo + 2 * width : n;
      int32_t a = lo, b = mid, o = lo;
      while (a < mid && b < hi) {
        if (key[b] > key[a]) { tk[o] = key[b]; ti[o++] = id[b++]; }   /* only strictly larger jumps ahead */
        else { tk[o] = key[a]; ti[o++] = id[a++]; }
      }
      while (a < mid) { tk[o] = key[a]; ti[o++] = id[a++]; }
      while (b < hi) { tk[o] = key[b]; ti[o++] = id[b++]; }
    }
    memcpy(key, tk, sizeof(uint32_t) * (size_t)n);
    memcpy(id, ti, sizeof(int32_t) * (size_t)n);
  }
}

/*
 * launchQsaIndexExpand for one row: top kSel = min(512, nVis) block ids (given in
 * sortedIds order) -> token ids 4*id + j, then the causal tail 4*nVis + j for
 * j < (t+1) % 4, then -1 to width 2051.  nVis = (t+1)/4.  Padded rows (ctx <= 0 or
 * t >= ctx) are all -1 and sortedIds is not read.
 */
void qsa_oracle_expand_row(int32_t* out, const int32_t* sortedIds, int32_t t, int32_t ctx) {
  for (int32_t i = 0; i < QSA_INDEX_WIDTH; ++i) out[i] = -1;
  if (ctx <= 0 || t >= ctx) return;
  int32_t nVis = (t + 1) / QSA_COMPRESS_RATIO;
  int32_t kSel = nVis < QSA_TOPK_BLOCKS ? nVis : QSA_TOPK_BLOCKS;
  int32_t tail = (t + 1) % QSA_COMPRESS_RATIO;
  for (int32_t i = 0; i < kSel; ++i)
    for (int32_t j = 0; j < QSA_COMPRESS_RATIO; ++j) out[QSA_COMPRESS_RATIO * i + j] = sortedIds[i] * QSA_COMPRESS_RATIO + j;
  for (int32_t j = 0; j < tail; ++j) out[QSA_COMPRESS_RATIO * kSel + j] = QSA_COMPRESS_RATIO * nVis + j;
}

/*
 * The prefill selection for one row, as the page's pipeline computes it: ids
 * 0..numBlocks-1, a stable descending sort of the row's FP32 logits (compared by
 * the order-preserving map, so ties keep ascending ids), then the expand.  Only
 * the first nVis keys can be selected; the rest are the masked -FLT_MAX cells,
 * which sort last, so sorting the visible prefix gives the same first kSel ids.
 * scratch: 4 * numBlocks 32-bit words.
 */
void qsa_oracle_select_expand_row(int32_t* out, const float* logits_row, int32_t numBlocks,
                                  int32_t t, int32_t ctx, uint32_t* scratch) {
  if (ctx <= 0 || t >= ctx) {
    for (int32_t i = 0; i < QSA_INDEX_WIDTH; ++i) out[i] = -1;
    return;
  }
  int32_t n = numBlocks;
  uint32_t* key = scratch;
  int32_t* id = (int32_t*)(scratch + n);
  uint32_t* tk = scratch + 2 * (int64_t)n;
  int32_t* ti = (int32_t*)(scratch + 3 * (int64_t)n);
  for (int32_t g = 0; g < n; ++g) { key[g] = qsa_oracle_orderable(logits_row[g]); id[g] = g; }
  stable_sort_desc(key, id, tk, ti, n);
  qsa_oracle_expand_row(out, id, t, ctx);
}

/* Rows [rowStart, rowStart + numRows): logits chunk-local [numRows, numBlocks];
 * outIdx global [B*S, 2051] (rows of the chunk written). */
int qsa_oracle_select_expand(int32_t* outIdx, const float* logits, const int32_t* contextLengths,
                             int32_t B, int32_t S, int32_t numBlocks, int32_t rowStart,
                             int32_t numRows, uint32_t* scratch) {
  if (rowStart < 0 || numRows < 0 || (int64_t)rowStart + numRows > (int64_t)B * S) return -3;
  for (int32_t i = 0; i < numRows; ++i) {
    int64_t r = (int64_t)rowStart + i;
    int32_t b = (int32_t)(r / S);
    int32_t t = (int32_t)(r - (int64_t)b * S);
    qsa_oracle_select_expand_row(outIdx + r * QSA_INDEX_WIDTH, logits + (int64_t)i * numBlocks,
                                 numBlocks, t, contextLengths[b], scratch);
  }
  return 0;
}

/* ------------------------------------------------- paged pool (decode state) */

/*
 * QsaIndexerPoolState: pool [2*numPages, 128, numKVHeads, poolHeadDim] T; element
 * (page, row, head, col) at ((page*128 + row)*numKVHeads + head)*poolHeadDim + col.
 * pageTable [B, 2, maxPagesPerSeq]: plane 0 = K pages, plane 1 = V pages (ids already
 * offset by +numPages).  Token t's raw index-K tail: K page pageTable[b][0][t >> 7],
 * row t & 127, head 0, columns [headSize, headSize + 128).  Block g's kbar: V page
 * pageTable[b][1][(4g) >> 7], row (4g) & 127, head 0, same columns.  Entries equal to
 * -1 (unused) -- and slots past maxPagesPerSeq or ids outside the pool -- mean
 * "nothing persistable here" and are never dereferenced.
 */
typedef struct {
  uint16_t* pool;
  const int32_t* pageTable;
  int32_t maxPagesPerSeq;
  int32_t numPages;
  int32_t numKVHeads;
  int32_t poolHeadDim;
  int32_t headSize;
} qsa_oracle_pool_t;

#define QSA_PAGE_TOKENS 128

static uint16_t* pool_tail(const qsa_oracle_pool_t* ps, int32_t b, int32_t plane, int32_t token) {
  if (token < 0) return 0;
  int32_t slot = token / QSA_PAGE_TOKENS;
  if (slot >= ps->maxPagesPerSeq) return 0;
  int32_t page = ps->pageTable[((int64_t)b * 2 + plane) * ps->maxPagesPerSeq + slot];
  if (page < 0 || page >= 2 * ps->numPages) return 0;
  int64_t row = token % QSA_PAGE_TOKENS;
  int64_t off = (((int64_t)page * QSA_PAGE_TOKENS + row) * ps->numKVHeads + 0) * ps->poolHeadDim + ps->headSize;
  return ps->pool + off;
}

/* launchQsaIndexKCompressPaged: launchQsaIndexKCompress, and each VALID block's kbar
 * row is also copied to the V-tail of token 4g when that page slot is usable. */
int qsa_oracle_k_compress_paged(int dtype, uint16_t* kbar, const uint16_t* indexQk, const float* cosSin,
                                const int32_t* contextLengths, const uint16_t* wK, float eps,
                                const qsa_oracle_pool_t* ps, int32_t B, int32_t S, int32_t numBlocks,
                                int32_t blockBegin, int32_t blockEnd, int32_t pastLen) {
  int rc = qsa_oracle_k_compress(dtype, kbar, indexQk, cosSin, contextLengths, wK, eps, B, S, numBlocks,
                                 blockBegin, blockEnd, pastLen);
  if (rc) return rc;
  for (int32_t b = 0; b < B; ++b)
    for (int32_t g = blockBegin; g < blockEnd; ++g) {
      if (!qsa_oracle_block_valid(g, contextLengths[b], S, pastLen)) continue;
      uint16_t* dst = pool_tail(ps, b, 1, QSA_COMPRESS_RATIO * g);
      if (dst) memcpy(dst, kbar + ((int64_t)b * numBlocks + g) * QSA_HEAD_DIM, 2 * QSA_HEAD_DIM);
    }
  return 0;
}

/* launchQsaRawKTailWritePrefill: tokens t in [ctx - ctx % 4, ctx) copy their raw
 * index-K (indexQk columns [512, 640)) bit for bit to their K-tails. */
int qsa_oracle_raw_k_tail_write_prefill(const uint16_t* indexQk, const int32_t* contextLengths,
                                        const qsa_oracle_pool_t* ps, int32_t B, int32_t S) {
  for (int32_t b = 0; b < B; ++b) {
    int32_t c = contextLengths[b];
    if (c <= 0) continue;
    for (int32_t t = c - c % QSA_COMPRESS_RATIO; t < c && t < S; ++t) {
      uint16_t* dst = pool_tail(ps, b, 0, t);
      if (dst) memcpy(dst, indexQk + ((int64_t)b * S + t) * QSA_ROW_WIDTH + QSA_K_COL, 2 * QSA_HEAD_DIM);
    }
  }
  return 0;
}

/*
 * launchQsaIndexerPreDecode, per sequence b with one new token (indexQk [B, 640]) and
 * TOTAL length ctx = contextLengths[b], pos = ctx - 1:
 *   ctx <= 0: qNormed[b] = exact zeros, nothing else.
 *   q-prep of the new row at rope position pos (launchQsaIndexQPrep numerics).
 *   ctx % 4 != 0: the row's raw index-K goes bit for bit to the K-tail of pos.
 *   ctx % 4 == 0: block g = ctx/4 - 1 is complete: tokens 4g..4g+2 come from their
 *   K-tails, token 4g+3 from the new row; launchQsaIndexKCompress numerics; the kbar
 *   row goes to the V-tail of 4g.  If a needed page slot is unusable, the block is
 *   not written.
 */
int qsa_oracle_pre_decode(int dtype, uint16_t* qNormed, const uint16_t* indexQk, const float* cosSin,
                          const int32_t* contextLengths, const uint16_t* wQ, const uint16_t* wK, float eps,
                          const qsa_oracle_pool_t* ps, int32_t B) {
  for (int32_t b = 0; b < B; ++b) {
    int32_t c = contextLengths[b];
    uint16_t* q = qNormed + (int64_t)b * QSA_NUM_Q_HEADS * QSA_HEAD_DIM;
    const uint16_t* in = indexQk + (int64_t)b * QSA_ROW_WIDTH;
    if (c <= 0) {
      memset(q, 0, sizeof(uint16_t) * QSA_NUM_Q_HEADS * QSA_HEAD_DIM);
      continue;
    }
    int32_t pos = c - 1;
    for (int h = 0; h < QSA_NUM_Q_HEADS; ++h) {
      float x[QSA_HEAD_DIM];
      for (int d = 0; d < QSA_HEAD_DIM; ++d) x[d] = qsa_oracle_t_to_f32(dtype, in[h * QSA_HEAD_DIM + d]);
      qsa_oracle_norm_rope(dtype, x, wQ, eps, cosSin + (int64_t)pos * 64, q + h * QSA_HEAD_DIM);
    }
    if (c % QSA_COMPRESS_RATIO != 0) {
      uint16_t* dst = pool_tail(ps, b, 0, pos);
      if (dst) memcpy(dst, in + QSA_K_COL, 2 * QSA_HEAD_DIM);
      continue;
    }
    int32_t g = c / QSA_COMPRESS_RATIO - 1;
    const uint16_t* k[QSA_COMPRESS_RATIO];
    int ok = 1;
    for (int j = 0; j < QSA_COMPRESS_RATIO - 1; ++j) {
      k[j] = pool_tail(ps, b, 0, QSA_COMPRESS_RATIO * g + j);
      if (!k[j]) ok = 0;
    }
    k[QSA_COMPRESS_RATIO - 1] = in + QSA_K_COL;
    uint16_t* dst = pool_tail(ps, b, 1, QSA_COMPRESS_RATIO * g);
    if (!ok || !dst) continue;
    uint16_t m[QSA_HEAD_DIM];
    qsa_oracle_block_mean(dtype, k[0], k[1], k[2], k[3], m);
    float x[QSA_HEAD_DIM];
    for (int d = 0; d < QSA_HEAD_DIM; ++d) x[d] = qsa_oracle_t_to_f32(dtype, m[d]);
    qsa_oracle_norm_rope(dtype, x, wK, eps, cosSin + (int64_t)QSA_COMPRESS_RATIO * g * 64, dst);
  }
  return 0;
}

/*
 * launchQsaIndexScoresDecode: logits[b][g] for g < nVis = ctx/4 only, K2 numerics
 * with kbar gathered from the V-tail of token 4g; a block whose page slot is
 * unusable scores -FLT_MAX (reading: "nothing persistable here").  Entries at
 * g >= nVis are not written.
 */
int qsa_oracle_scores_decode(int dtype, float* logits, const uint16_t* qNormed, const int32_t* contextLengths,
                             const qsa_oracle_pool_t* ps, int32_t B, int32_t maxBlocks) {
  const float scale = 1.0f / sqrtf(128.0f);
  for (int32_t b = 0; b < B; ++b) {
    int32_t c = contextLengths[b];
    int32_t nVis = c > 0 ? c / QSA_COMPRESS_RATIO : 0;
    if (nVis > maxBlocks) nVis = maxBlocks;
    const uint16_t* q = qNormed + (int64_t)b * QSA_NUM_Q_HEADS * QSA_HEAD_DIM;
    float qf[QSA_NUM_Q_HEADS][QSA_HEAD_DIM];
    for (int h = 0; h < QSA_NUM_Q_HEADS; ++h)
      for (int d = 0; d < QSA_HEAD_DIM; ++d) qf[h][d] = qsa_oracle_t_to_f32(dtype, q[h * QSA_HEAD_DIM + d]);
    for (int32_t g = 0; g < nVis; ++g) {
      const uint16_t* k = pool_tail(ps, b, 1, QSA_COMPRESS_RATIO * g);
      float* out = logits + (int64_t)b * maxBlocks + g;
      if (!k) { *out = -FLT_MAX; continue; }
      float sum = 0.0f;
      for (int h = 0; h < QSA_NUM_Q_HEADS; ++h) {
        float dot = 0.0f;
        for (int d = 0; d < QSA_HEAD_DIM; ++d) {
          float p = qf[h][d] * qsa_oracle_t_to_f32(dtype, k[d]);
          dot = dot + p;
        }
        float rel = fmaxf(0.0f, dot);
        sum = sum + rel;
      }
      *out = scale * sum;
    }
  }
  return 0;
}

/*
 * launchQsaTopKExpandDecode, per sequence b (ctx = contextLengths[b], nVis = ctx/4,
 * kSel = min(512, nVis), tail = ctx % 4): splitCounters[b*numKVHeads ..) zeroed if
 * given; the selected set is the first kSel blocks of the stable descending sort of
 * logits[b][0..nVis) (keys above the kSel-th largest, ties in ascending id), emitted
 * in ascending block order; out[b][4i + j] = sel[i]*4 + j, then tokens 4*nVis + j for
 * j < tail, then -1 to width 2051.  scratch: 4 * maxBlocks words.
 */
int qsa_oracle_topk_expand_decode(int32_t* outIdx, const float* logits, const int32_t* contextLengths,
                                  int32_t* splitCounters, int32_t numKVHeads, int32_t B, int32_t maxBlocks,
                                  uint32_t* scratch) {
  for (int32_t b = 0; b < B; ++b) {
    if (splitCounters)
      for (int32_t h = 0; h < numKVHeads; ++h) splitCounters[(int64_t)b * numKVHeads + h] = 0;
    int32_t* out = outIdx + (int64_t)b * QSA_INDEX_WIDTH;
    for (int32_t i = 0; i < QSA_INDEX_WIDTH; ++i) out[i] = -1;
    int32_t c = contextLengths[b];
    if (c <= 0) continue;
    int32_t nVis = c / QSA_COMPRESS_RATIO;
    if (nVis > maxBlocks) nVis = maxBlocks;
    if (nVis < 0) nVis = 0;
    int32_t kSel = nVis < QSA_TOPK_BLOCKS ? nVis : QSA_TOPK_BLOCKS;
    int32_t tail = c % QSA_COMPRESS_RATIO;
    uint32_t* key = scratch;
    int32_t* id = (int32_t*)(scratch + maxBlocks);
    uint32_t* tk = scratch + 2 * (int64_t)maxBlocks;
    int32_t* ti = (int32_t*)(scratch + 3 * (int64_t)maxBlocks);
    for (int32_t g = 0; g < nVis; ++g) { key[g] = qsa_oracle_orderable(logits[(int64_t)b * maxBlocks + g]); id[g] = g; }
    stable_sort_desc(key, id, tk, ti, nVis);
    /* ascending block order of the selected set: mark, then scan */
    uint8_t* mark = (uint8_t*)tk;
    memset(mark, 0, (size_t)nVis);
    for (int32_t i = 0; i < kSel; ++i) mark[id[i]] = 1;
    int32_t n = 0;
    for (int32_t g = 0; g < nVis; ++g)
      if (mark[g])
        for (int32_t j = 0; j < QSA_COMPRESS_RATIO; ++j) out[n++] = g * QSA_COMPRESS_RATIO + j;
    for (int32_t j = 0; j < tail; ++j) out[n++] = QSA_COMPRESS_RATIO * nVis + j;
  }
  return 0;
}
