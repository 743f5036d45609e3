// Device helpers shared by the K1a (q-prep) and K1b (K-compress) kernels.
//
// Layout facts ("Qsa Indexer Kernels", launchQsaIndexQPrep / launchQsaIndexKCompress):
//   indexQk row = 640 T: q heads 0..3 x 128 dims (columns 0..511), raw k x 128 (512..639)
//   qNormed row = 4 x 128 T, kbar row = 128 T, cosSin row = 64 FP32 (cos 0..31, sin 32..63)
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace qsa {

constexpr int kHeadDim = 128;
constexpr int kNumQHeads = 4;
constexpr int kRowWidth = 640;
constexpr int kKCol = 512;
constexpr int kRatio = 4;
constexpr int kCsWidth = 64;

// ---------------------------------------------------------------- element types

struct Bf16 {
  static constexpr bool kIsBf16 = true;
  static __device__ __forceinline__ float one(uint16_t u) { return __uint_as_float(static_cast<uint32_t>(u) << 16); }
  static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
  static __device__ __forceinline__ uint32_t pack(float a, float b) {  // a -> low half
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ float round_trip(float f) {  // cast to T, re-load
    return __bfloat162float(__float2bfloat16_rn(f));
  }
};

struct F16 {
  static constexpr bool kIsBf16 = false;
  static __device__ __forceinline__ float one(uint16_t u) { return __half2float(__ushort_as_half(u)); }
  static __device__ __forceinline__ float lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
  }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  }
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ float round_trip(float f) {
    return __half2float(__float2half_rn(f));
  }
};

template <class T>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = T::lo(v.x); f[1] = T::hi(v.x);
  f[2] = T::lo(v.y); f[3] = T::hi(v.y);
  f[4] = T::lo(v.z); f[5] = T::hi(v.z);
  f[6] = T::lo(v.w); f[7] = T::hi(v.w);
}

template <class T>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  v.x = T::pack(f[0], f[1]);
  v.y = T::pack(f[2], f[3]);
  v.z = T::pack(f[4], f[5]);
  v.w = T::pack(f[6], f[7]);
  return v;
}

// ------------------------------------------------------------- 16-byte memory I/O

// Streamed, read-once input (indexQk): non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Re-used read-only input (cos/sin rows, gammas): non-coherent cached path.
__device__ __forceinline__ float4 ld_cached_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_cached_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ------------------------------------------------------ 8-lane vector ownership
//
// An aligned group of 8 lanes owns one 128-dim vector.  Lane j (0..7) holds two
// 8-dim chunks, chosen so that every rope pair (i, i+32), i < 32, sits in one lane:
//   j < 4 : chunk A = dims [8j, 8j+8),       chunk B = dims [32+8j, 40+8j)   (rotated)
//   j >= 4: chunk A = dims [64+8(j-4), ...),  chunk B = dims [96+8(j-4), ...) (pass-through)
__device__ __forceinline__ int chunk_a(int j) { return j < 4 ? 8 * j : 64 + 8 * (j - 4); }
__device__ __forceinline__ int chunk_b(int j) { return j < 4 ? 32 + 8 * j : 96 + 8 * (j - 4); }

// (1 + w) for all 128 dims into shared memory, once per CTA (w is the raw
// checkpoint gamma [128] in T).  Call before the CTA's first __syncthreads().
template <class T>
__device__ __forceinline__ void stage_gamma(const uint16_t* w, float* g1, int first = threadIdx.x,
                                            int stride = blockDim.x) {
  for (int d = first; d < kHeadDim; d += stride) g1[d] = __fadd_rn(1.0f, T::one(w[d]));
}

// The lane's cos/sin values for rope position row `cs` (only lanes j < 4 rotate).
struct RopeCS {
  float4 c0, c1, s0, s1;
};

__device__ __forceinline__ RopeCS load_rope(const float* cs, int j) {
  RopeCS r;
  const float* p = cs + 8 * (j & 3);
  r.c0 = ld_cached_f4(p);
  r.c1 = ld_cached_f4(p + 4);
  r.s0 = ld_cached_f4(p + 32);
  r.s1 = ld_cached_f4(p + 36);
  return r;
}

// Gemma-style RMS norm with (1 + w) and partial neox rope, then one cast to T
// ("Qsa Indexer Kernels", launchQsaIndexQPrep "Exact numerics"; the same numerics
// are used verbatim by launchQsaIndexKCompress on the block mean):
//   meanSq = sum x^2 / 128 (lane sum, then an xor tree over the 8 lanes; every
//   lane ends with the same bits), r = rsqrtf(meanSq + eps), y = (x * r) * (1 + w),
//   rotated pair (y_i*c - y_{i+32}*s, y_{i+32}*c + y_i*s), dims >= 64 unrotated.
// Every lane of the warp must call this (it shuffles with a full mask).
template <class T>
__device__ __forceinline__ void norm_rope_group(const float (&a)[8], const float (&b)[8],
                                                const float* g1, float eps, const RopeCS& cs, int j,
                                                uint4& out_a, uint4& out_b) {
  float s = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) s = fmaf(a[e], a[e], s);
#pragma unroll
  for (int e = 0; e < 8; ++e) s = fmaf(b[e], b[e], s);
  s += __shfl_xor_sync(0xffffffffu, s, 4);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  const float mean_sq = __fmul_rn(s, 1.0f / 128.0f);  // exact power-of-two scaling
  const float r = rsqrtf(__fadd_rn(mean_sq, eps));
  const float4* ga4 = reinterpret_cast<const float4*>(g1 + chunk_a(j));
  const float4* gb4 = reinterpret_cast<const float4*>(g1 + chunk_b(j));
  // every chunk starts on a bank that is a multiple of 8: lanes j >= 4 read each chunk's
  // second half first, so a 16-byte load's eight lanes of a group cover 32 banks
  const int h0 = j >= 4 ? 1 : 0;
  const float4 pa = ga4[h0], qa = ga4[h0 ^ 1], pb = gb4[h0], qb = gb4[h0 ^ 1];
  const float4 ga0 = h0 ? qa : pa, ga1 = h0 ? pa : qa, gb0 = h0 ? qb : pb, gb1 = h0 ? pb : qb;
  const float ga[8] = {ga0.x, ga0.y, ga0.z, ga0.w, ga1.x, ga1.y, ga1.z, ga1.w};
  const float gb[8] = {gb0.x, gb0.y, gb0.z, gb0.w, gb1.x, gb1.y, gb1.z, gb1.w};
  float ya[8], yb[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ya[e] = __fmul_rn(__fmul_rn(a[e], r), ga[e]);
    yb[e] = __fmul_rn(__fmul_rn(b[e], r), gb[e]);
  }
  if (j < 4) {
    const float c[8] = {cs.c0.x, cs.c0.y, cs.c0.z, cs.c0.w, cs.c1.x, cs.c1.y, cs.c1.z, cs.c1.w};
    const float sn[8] = {cs.s0.x, cs.s0.y, cs.s0.z, cs.s0.w, cs.s1.x, cs.s1.y, cs.s1.z, cs.s1.w};
    float oa[8], ob[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      oa[e] = __fsub_rn(__fmul_rn(ya[e], c[e]), __fmul_rn(yb[e], sn[e]));
      ob[e] = __fadd_rn(__fmul_rn(yb[e], c[e]), __fmul_rn(ya[e], sn[e]));
    }
    out_a = pack8<T>(oa);
    out_b = pack8<T>(ob);
  } else {
    out_a = pack8<T>(ya);
    out_b = pack8<T>(yb);
  }
}

}  // namespace qsa
