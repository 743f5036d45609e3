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
// gets the T bits of dims chunk_a(j) and chunk_b(j) of head h.  c <= 0: zeros.
template <class T>
__device__ __forceinline__ void q_heads(const uint16_t* row, const float* cos_sin, int32_t c, const float* g1q,
                                        float eps, int lane, uint4& oa, uint4& ob) {
  const int h = lane >> 3, j = lane & 7;
  const int ca = chunk_a(j), cb = chunk_b(j);
  oa = make_uint4(0u, 0u, 0u, 0u);
  ob = oa;
  if (c > 0) {  // warp-uniform
    const int32_t pos = c - 1;
    float a[8], bv[8];
    unpack8<T>(ld_stream_v4(row + h * kHeadDim + ca), a);
    unpack8<T>(ld_stream_v4(row + h * kHeadDim + cb), bv);
    RopeCS cs{};
    if (j < 4) cs = load_rope(cos_sin + static_cast<int64_t>(pos) * kCsWidth, j);
    norm_rope_group<T>(a, bv, g1q, eps, cs, j, oa, ob);
  }
}

// One warp, c % 4 == 0: block g = c/4 - 1 compressed from the K-tails of 4g..4g+2 and
// the new row's raw K (K1b numerics).  Returns whether every page slot involved is
// usable; then lanes of group 0 (lane < 8) hold the kbar bits of dims chunk_a(lane)
// and chunk_b(lane), and *vtail is the block's V-tail.
template <class T>
__device__ __forceinline__ bool compress_block(const PoolDev& pool, int32_t b, int32_t c, const uint16_t* row,
                                               const float* cos_sin, const float* g1k, float eps, int lane,
                                               uint4& oa, uint4& ob, uint16_t** vtail) {
  const int j = lane & 7;
  const int ca = chunk_a(j), cb = chunk_b(j);
  const int32_t g = c / kRatio - 1;
  const uint16_t* k0 = pool_tail(pool, b, 0, kRatio * g);
  const uint16_t* k1 = pool_tail(pool, b, 0, kRatio * g + 1);
  const uint16_t* k2 = pool_tail(pool, b, 0, kRatio * g + 2);
  *vtail = pool_tail(pool, b, 1, kRatio * g);
  const bool ok = k0 != nullptr && k1 != nullptr && k2 != nullptr && *vtail != nullptr;  // warp-uniform
  float a[8], bv[8];
  RopeCS cs{};
  if (ok) {
    const uint16_t* src[kRatio] = {k0, k1, k2, row + kKCol};
    float fa[kRatio][8], fb[kRatio][8];
#pragma unroll
    for (int q = 0; q < kRatio; ++q) {
      unpack8<T>(ld_cached_v4(src[q] + ca), fa[q]);
      unpack8<T>(ld_cached_v4(src[q] + cb), fb[q]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float s = __fadd_rn(__fadd_rn(__fadd_rn(fa[0][e], fa[1][e]), fa[2][e]), fa[3][e]);
      a[e] = T::round_trip(__fmul_rn(s, 0.25f));
      s = __fadd_rn(__fadd_rn(__fadd_rn(fb[0][e], fb[1][e]), fb[2][e]), fb[3][e]);
      bv[e] = T::round_trip(__fmul_rn(s, 0.25f));
    }
    if (j < 4) cs = load_rope(cos_sin + static_cast<int64_t>(kRatio) * g * kCsWidth, j);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) { a[e] = 0.0f; bv[e] = 0.0f; }
  }
  norm_rope_group<T>(a, bv, g1k, eps, cs, j, oa, ob);  // every lane takes part in the shuffles
  return ok;
}

// Paged scores.  A 16-lane half-warp scores one block: lane ch holds dims [8ch, 8ch+8)
// of the 4 q heads (qf) and 16 bytes of the block's kbar (raw), forms 4 partial dots,
// and the half-warp reduces them (a reduce-scatter over lane bits 3 and 2, then bits 1
// and 0), so that lanes 0/4/8/12 hold heads 0/1/2/3.  Returns, on lane ch == 0, the sum
// of relu of the heads in ascending order (before the scale).  Every lane of the warp
// must call it.
template <class T>
__device__ __forceinline__ float score_block(const float (&qf)[kNumQHeads][8], uint4 raw, int ch) {
  const unsigned half = threadIdx.x & 16;
  const bool keep_hi = (ch & 8) != 0, keep_odd = (ch & 4) != 0;
  float kf[8];
  unpack8<T>(raw, kf);
  float d[kNumQHeads];
#pragma unroll
  for (int h = 0; h < kNumQHeads; ++h) {
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(qf[h][e], kf[e], acc);
    d[h] = acc;
  }
  // lane bit 3: keep heads {2,3} or {0,1}; send the other pair to the partner
  const float s0 = keep_hi ? d[0] : d[2], s1 = keep_hi ? d[1] : d[3];
  const float r0 = __shfl_xor_sync(0xffffffffu, s0, 8), r1 = __shfl_xor_sync(0xffffffffu, s1, 8);
  const float e0 = (keep_hi ? d[2] : d[0]) + r0, e1 = (keep_hi ? d[3] : d[1]) + r1;
  // lane bit 2: keep the pair's second or first head
  const float r2 = __shfl_xor_sync(0xffffffffu, keep_odd ? e0 : e1, 4);
  float f = (keep_odd ? e1 : e0) + r2;
  f += __shfl_xor_sync(0xffffffffu, f, 2);
  f += __shfl_xor_sync(0xffffffffu, f, 1);
  const float rel = fmaxf(0.0f, f);  // head ((ch >> 3) & 1) * 2 + ((ch >> 2) & 1)
  const float h1 = __shfl_sync(0xffffffffu, rel, half | 4);
  const float h2 = __shfl_sync(0xffffffffu, rel, half | 8);
  const float h3 = __shfl_sync(0xffffffffu, rel, half | 12);
  return __fadd_rn(__fadd_rn(__fadd_rn(rel, h1), h2), h3);
}

constexpr int kDecThreads = 256;
constexpr int kDecUnroll = 4;   // blocks a half-warp has in flight in one round
constexpr int kDecRounds = 2;
constexpr int kDecBlocksPerCta = (kDecThreads / 16) * kDecUnroll * kDecRounds;

// One round of a half-warp: blocks g0 + 16*u, u < kDecUnroll; lane ch's 16 bytes of each
// block's V-tail (zeros where the block is past g_end or its page slot is unusable).
struct Round {
  uint4 raw[kDecUnroll];
  bool ok[kDecUnroll];
};

__device__ __forceinline__ void load_round(Round& r, const PoolDev& pool, int32_t b, int32_t g0, int32_t g_end,
                                           int ch) {
#pragma unroll
  for (int u = 0; u < kDecUnroll; ++u) {
    const int32_t g = g0 + 16 * u;
    const uint16_t* k = g < g_end ? pool_tail(pool, b, 1, kRatio * g) : nullptr;
    r.ok[u] = k != nullptr;
    r.raw[u] = r.ok[u] ? ld_stream_v4(k + 8 * ch) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Scores one loaded round into the logits row `out`; block `own` (>= 0) takes its kbar
// from `own_kbar` (shared memory) instead of the pool.  Every lane of the warp calls it.
template <class T>
__device__ __forceinline__ void score_round(float* out, const float (&qf)[kNumQHeads][8], Round& r, int32_t g0,
                                            int32_t g_end, float scale, int32_t own, const uint16_t* own_kbar,
                                            int ch) {
#pragma unroll
  for (int u = 0; u < kDecUnroll; ++u) {
    const int32_t g = g0 + 16 * u;
    if (g == own) {
      r.ok[u] = true;
      r.raw[u] = *reinterpret_cast<const uint4*>(own_kbar + 8 * ch);
    }
    const float sum = score_block<T>(qf, r.raw[u], ch);
    if (ch == 0 && g < g_end) out[g] = r.ok[u] ? __fmul_rn(sum, scale) : -FLT_MAX;
  }
}

// The paged scores of blocks [g_begin, g_end) (g_end - g_begin <= kDecBlocksPerCta) of
// sequence b by a CTA of kDecThreads threads; logits row `out`.  qf holds this lane's 8
// dims (8 * (lane % 16) ..) of the 4 q heads.  All rounds' loads are issued first.
template <class T>
__device__ __forceinline__ void score_range(float* out, const float (&qf)[kNumQHeads][8], const PoolDev& pool,
                                            int32_t b, int32_t g_begin, int32_t g_end, float scale, int32_t own,
                                            const uint16_t* own_kbar) {
  const int ch = threadIdx.x & 15, hw = threadIdx.x >> 4;
  Round r[kDecRounds];
#pragma unroll
  for (int k = 0; k < kDecRounds; ++k) load_round(r[k], pool, b, g_begin + 16 * kDecUnroll * k + hw, g_end, ch);
#pragma unroll
  for (int k = 0; k < kDecRounds; ++k)
    score_round<T>(out, qf, r[k], g_begin + 16 * kDecUnroll * k + hw, g_end, scale, own, own_kbar, ch);
}

}  // namespace dec
}  // namespace qsa
