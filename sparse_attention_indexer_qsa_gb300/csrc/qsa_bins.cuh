// First-pass threshold bins of the top-512 selection, shared by the fused scoring +
// selection kernel and the scoring kernel's per-row hints.
//
// A visible logit's order-preserving key (bits >= 0 ? bits | 2^31 : ~bits) falls in
// one of 256 bins, monotone in the key: bin 0 holds -0 and anything ordered below
// +0, bin 1 exactly +0 (a whole tie class: a logit is +0 whenever every head's dot
// is negative), bins 2..255 the positive keys on a log scale, 64 bins an octave
// (key >> 17) from `base`, clamped at both ends.  Bins 3..254 are exact prefix ranges
// of 2^17 keys; bins 2 and 255 are the clamped ends.  Where the bins sit decides
// only how many keys share the threshold bin, never which keys are selected.
#pragma once

#include <cstdint>

namespace qsa {
namespace bins {

constexpr int kBins = 256;
constexpr int kBaseMin = 0x3FFE;   // keeps bin 2 = (+0, first log bin] a proper range
constexpr int kBaseMax = 0x7F00;   // keeps (base + 255) << 17 inside 32 bits
constexpr int kLogShift = 17;      // 64 bins an octave: 6 mantissa bits
// bins centred a little below key(1.0f) >> 17: thresholds of unit-RMS q and kbar rows
// fall in [0.35, 5.3)
constexpr int kDefaultBase = static_cast<int>(0xBF800000u >> kLogShift) - 100;

__device__ __forceinline__ uint32_t bin_of(uint32_t key, int32_t base) {
  const int32_t d = static_cast<int32_t>(key >> kLogShift) - base;
  const uint32_t b = static_cast<uint32_t>(min(max(d, 2), 255));
  return key <= 0x80000000u ? key >> 31 : b;
}

__device__ __forceinline__ void bin_range(uint32_t b, int32_t base, uint32_t& lo, uint32_t& hi) {
  const uint32_t ub = static_cast<uint32_t>(base);
  if (b == 0u) {
    lo = 0u;
    hi = 0x7FFFFFFFu;
  } else if (b == 1u) {
    lo = hi = 0x80000000u;
  } else if (b == 2u) {
    lo = 0x80000001u;
    hi = ((ub + 3u) << kLogShift) - 1u;
  } else if (b == 255u) {
    lo = (ub + 255u) << kLogShift;
    hi = 0xFFFFFFFFu;
  } else {
    lo = (ub + b) << kLogShift;
    hi = ((ub + b + 1u) << kLogShift) - 1u;
  }
}

// The next base from where a unit's thresholds fell: `d` is base + bin for an exact bin,
// an octave beyond the clamped ends for bins 2 and 255.
__device__ __forceinline__ int32_t threshold_digit(uint32_t b, int32_t base) {
  return b == 2u ? base + 2 - 64 : (b == 255u ? base + 255 + 64 : base + static_cast<int32_t>(b));
}

__device__ __forceinline__ int32_t next_base(uint32_t sum, uint32_t n, int32_t base) {
  if (n == 0u) return base;
  const int32_t avg = static_cast<int32_t>(sum / n);
  return min(max(avg - 128, kBaseMin), kBaseMax);
}

// One warp finds, in a row's 256 bins (packed u16 pairs: bin 2i in the low half of
// word i), the bin holding the rem-th largest key, the count above it and its own
// count; every lane gets the result.
struct Found {
  uint32_t bin, above, count;
};

__device__ __forceinline__ Found find_bin(const uint32_t* hist_row, uint32_t want, int lane) {
  const uint4 v = reinterpret_cast<const uint4*>(hist_row)[31 - lane];
  // this lane's 8 bins, highest first: bins 8*(31-lane) + 7 .. + 0
  const uint32_t b8[8] = {v.w >> 16, v.w & 0xFFFFu, v.z >> 16, v.z & 0xFFFFu,
                          v.y >> 16, v.y & 0xFFFFu, v.x >> 16, v.x & 0xFFFFu};
  uint32_t mine = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) mine += b8[j];
  uint32_t incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += x;
  }
  const uint32_t excl = incl - mine;
  const bool hit = excl < want && want <= incl;
  Found f{0u, 0u, 0u};
  if (hit) {
    uint32_t c = excl;
    bool done = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!done) {
        if (c + b8[j] >= want) {
          f = Found{8u * static_cast<uint32_t>(31 - lane) + 7u - static_cast<uint32_t>(j), c, b8[j]};
          done = true;
        } else {
          c += b8[j];
        }
      }
    }
  }
  const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
  f.bin = __shfl_sync(0xffffffffu, f.bin, src);
  f.above = __shfl_sync(0xffffffffu, f.above, src);
  f.count = __shfl_sync(0xffffffffu, f.count, src);
  return f;
}

}  // namespace bins
}  // namespace qsa
