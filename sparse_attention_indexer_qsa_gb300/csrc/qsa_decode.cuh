// Device routines of the decode step ("Qsa Indexer Kernels": launchQsaIndexerPreDecode,
// launchQsaIndexScoresDecode), shared by the separate decode kernels (k_decode.cu) and
// the fused decode step (k_decode_step.cu), so both compute the same bits.
#pragma once

#include <cfloat>

#include "qsa_common.cuh"
#include "qsa_launch.h"

namespace qsa {
namespace dec {

__device__ __forceinline__ void copy_tail(uint16_t* dst, const uint16_t* src, int lane) {
  if (lane < 16) st_v4(dst + 8 * lane, ld_stream_v4(src + 8 * lane));  // 256 bytes, 16 B per lane
}

// One warp: the new row's 4 q heads at rope position pos (K1a numerics); lane (h, j)
// gets the T bits of dims chunk_a(j) and chunk_b(j) of head h.  c <= 0: zeros.  The
// loads (q_heads_load, which reads nothing when c <= 0) may be issued before g1q is
// staged; q_heads_finish needs g1q.
struct QHeadsIn {
  uint4 ra, rb;
  RopeCS cs;
};
__device__ __forceinline__ QHeadsIn q_heads_load(const uint16_t* row, const float* cos_sin, int32_t c, int lane) {
  const int h = lane >> 3, j = lane & 7;
  QHeadsIn in{};
  if (c > 0) {  // warp-uniform
    in.ra = ld_stream_v4(row + h * kHeadDim + chunk_a(j));
    in.rb = ld_stream_v4(row + h * kHeadDim + chunk_b(j));
    if (j < 4) in.cs = load_rope(cos_sin + static_cast<int64_t>(c - 1) * kCsWidth, j);
  }
  return in;
}
template <class T>
__device__ __forceinline__ void q_heads_finish(const QHeadsIn& in, int32_t c, const float* g1q, float eps, int lane,
                                               uint4& oa, uint4& ob) {
  oa = make_uint4(0u, 0u, 0u, 0u);
  ob = oa;
  if (c > 0) {  // warp-uniform
    float a[8], bv[8];
    unpack8<T>(in.ra, a);
    unpack8<T>(in.rb, bv);
    norm_rope_group<T>(a, bv, g1q, eps, in.cs, lane & 7, oa, ob);
  }
}
template <class T>
__device__ __forceinline__ void q_heads(const uint16_t* row, const float* cos_sin, int32_t c, const float* g1q,
                                        float eps, int lane, uint4& oa, uint4& ob) {
  q_heads_finish<T>(q_heads_load(row, cos_sin, c, lane), c, g1q, eps, lane, oa, ob);
}

// One warp, c % 4 == 0: block g = c/4 - 1 compressed from the K-tails of 4g..4g+2 and
// the new row's raw K (K1b numerics).  compress_load issues every load (the page
// entries, the K rows, the rope row: none needs g1k, so they may be in flight while
// g1k is staged); compress_finish forms the block.  ok: every page slot involved is
// usable; then lanes of group 0 (lane < 8) hold the kbar bits of dims chunk_a(lane) and
// chunk_b(lane), and vtail is the block's V-tail.
struct CompressIn {
  uint4 ka[kRatio], kb[kRatio];
  RopeCS cs;
  uint16_t* vtail;
  bool ok;
};
__device__ __forceinline__ CompressIn compress_load(const PoolDev& pool, int32_t b, int32_t c, const uint16_t* row,
                                                    const float* cos_sin, int lane) {
  const int j = lane & 7;
  const int32_t g = c / kRatio - 1;
  CompressIn in{};
  const uint16_t* k0 = pool_tail(pool, b, 0, kRatio * g);
  const uint16_t* k1 = pool_tail(pool, b, 0, kRatio * g + 1);
  const uint16_t* k2 = pool_tail(pool, b, 0, kRatio * g + 2);
  in.vtail = pool_tail(pool, b, 1, kRatio * g);
  in.ok = k0 != nullptr && k1 != nullptr && k2 != nullptr && in.vtail != nullptr;  // warp-uniform
  if (in.ok) {
    const uint16_t* src[kRatio] = {k0, k1, k2, row + kKCol};
#pragma unroll
    for (int q = 0; q < kRatio; ++q) {
      in.ka[q] = ld_cached_v4(src[q] + chunk_a(j));
      in.kb[q] = ld_cached_v4(src[q] + chunk_b(j));
    }
    if (j < 4) in.cs = load_rope(cos_sin + static_cast<int64_t>(kRatio) * g * kCsWidth, j);
  }
  return in;
}
template <class T>
__device__ __forceinline__ void compress_finish(const CompressIn& in, const float* g1k, float eps, int lane,
                                                uint4& oa, uint4& ob) {
  float a[8], bv[8];
  if (in.ok) {
    float fa[kRatio][8], fb[kRatio][8];
#pragma unroll
    for (int q = 0; q < kRatio; ++q) {
      unpack8<T>(in.ka[q], fa[q]);
      unpack8<T>(in.kb[q], fb[q]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float s = __fadd_rn(__fadd_rn(__fadd_rn(fa[0][e], fa[1][e]), fa[2][e]), fa[3][e]);
      a[e] = T::round_trip(__fmul_rn(s, 0.25f));
      s = __fadd_rn(__fadd_rn(__fadd_rn(fb[0][e], fb[1][e]), fb[2][e]), fb[3][e]);
      bv[e] = T::round_trip(__fmul_rn(s, 0.25f));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) { a[e] = 0.0f; bv[e] = 0.0f; }
  }
  norm_rope_group<T>(a, bv, g1k, eps, in.cs, lane & 7, oa, ob);  // every lane takes part in the shuffles
}
template <class T>
__device__ __forceinline__ bool compress_block(const PoolDev& pool, int32_t b, int32_t c, const uint16_t* row,
                                               const float* cos_sin, const float* g1k, float eps, int lane,
                                               uint4& oa, uint4& ob, uint16_t** vtail) {
  const CompressIn in = compress_load(pool, b, c, row, cos_sin, lane);
  compress_finish<T>(in, g1k, eps, lane, oa, ob);
  *vtail = in.vtail;
  return in.ok;
}

constexpr int kDecThreads = 256;                              // threads of the one-launch decode step
constexpr int kDecBlocksPerCta = 128;                         // the unit a CTA's run is made of
constexpr int kPageWindow = 128;                              // V pages a run may span
constexpr int kDecRunMax = kPageWindow * (128 / kRatio);      // blocks a run may hold (4096)
constexpr int kScoresCtasPerSm = 2;                           // resident CTAs the run length assumes

// Blocks per CTA (a multiple of kDecBlocksPerCta, at most kDecRunMax) so that a grid of
// (batch, ceilDiv(max_blocks, run)) CTAs is about one wave of ctas_per_sm CTAs per SM.
inline int32_t decode_run_blocks(int sms, int ctas_per_sm, int32_t batch, int32_t max_blocks) {
  const int32_t units = (max_blocks + kDecBlocksPerCta - 1) / kDecBlocksPerCta;
  int32_t want_y = sms * ctas_per_sm / (batch > 0 ? batch : 1);
  if (want_y < 1) want_y = 1;
  int32_t per = (units + want_y - 1) / want_y;
  if (per < 1) per = 1;
  if (per > kDecRunMax / kDecBlocksPerCta) per = kDecRunMax / kDecBlocksPerCta;
  return per * kDecBlocksPerCta;
}

// The V page of each 128-token slot that blocks [g_begin, g_end) of sequence b touch
// (g_begin a multiple of 32, g_end - g_begin <= kDecRunMax), into pages[0, ..): the
// pool page, or -1 where pool_tail gives no address (slot past maxPagesPerSeq, -1 or
// outside the pool).  The caller synchronises before reading them.  Callers pass the
// whole run (not clipped to the sequence's valid prefix), so that the page-table loads
// need not wait for the context length; entries past the prefix are never used.
__device__ __forceinline__ void stage_vpages(int32_t* pages, const PoolDev& pool, int32_t b, int32_t g_begin,
                                             int32_t g_end, int first = threadIdx.x, int stride = blockDim.x) {
  if (g_end <= g_begin) return;
  const int32_t s0 = (kRatio * g_begin) >> 7;
  const int32_t n = ((kRatio * (g_end - 1)) >> 7) - s0 + 1;
  for (int i = first; i < n; i += stride) {
    const int32_t slot = s0 + i;
    int32_t page = -1;
    if (slot < pool.max_pages) {
      page = __ldg(pool.table + (static_cast<int64_t>(b) * 2 + 1) * pool.max_pages + slot);
      if (page < 0 || page >= 2 * pool.num_pages) page = -1;
    }
    pages[i] = page;
  }
}

}  // namespace dec
}  // namespace qsa
