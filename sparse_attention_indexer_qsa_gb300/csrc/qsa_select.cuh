// Device routines of the top-512 block selection ("Qsa Indexer Kernels": the prefill
// selection between launchQsaIndexIdsFill and launchQsaIndexExpand, and
// launchQsaTopKExpandDecode), shared by the selection kernels (k34_select.cu) and the
// fused decode step (k_decode_step.cu).
#pragma once

#include <cstdint>

namespace qsa {
namespace sel {

constexpr int kTopK = 512;
constexpr int kRatio = 4;
constexpr int kWidth = kTopK * kRatio + kRatio - 1;  // 2051

// bits >= 0 ? bits | 2^31 : ~bits, as b ^ (sign-fill | 2^31): two instructions, no select
__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t b = __float_as_uint(f);
  return b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
}


// ---------------------------------------------------------------------------
// topk: one CTA of T threads per row.
//
//  1. histogram of the first digit (digit1) over the visible blocks (coalesced; or the
//     counts a caller's kernel made, checked to total the row); warp 0 finds the bin b1
//     holding the kSel-th largest key, the count above it and c1, its own count.  For
//     rows of at most 32*T*MW blocks the pass also stores each key's digit >> 2 as one
//     byte in shared memory (the codes);
//  2. one ordered pass: thread k owns the 32*MW contiguous blocks from 32*MW*k and
//     records, as bit masks, which lie above b1 (selected) and in b1 (candidates), from
//     the keys in registers, from the codes (reloading only the keys that share b1's
//     code), or from the row; candidates are listed (their keys, or their block ids),
//     each thread's in ascending order;
//  3. unless b1 is filled exactly, the threshold key T inside b1, and how many keys
//     equal to T are still to be taken, are resolved by 8-bit radix passes: over
//     the listed candidates by warp 0 alone (up to kWarpCap of them), otherwise by
//     the whole CTA over the row;
//  4. candidates above T become selected and ties are taken in ascending block
//     order; one block scan of packed (selected, tied) counts gives each thread the
//     position of its first winner; winners are written in ascending order and the
//     row is expanded.
// Keys are read from global memory.  Small CTAs (64 threads, 8.2 KB of shared memory
// with the codes, 24 a SM) keep many rows in flight: the warp-0 steps between the
// passes are serial and would otherwise leave the SM idle.
#ifndef QSA_SEL_D1_BITS
#define QSA_SEL_D1_BITS 10
#endif
#ifndef QSA_SEL_WARPS_PER_SM
#define QSA_SEL_WARPS_PER_SM 48
#endif
constexpr int kD1 = QSA_SEL_D1_BITS;
constexpr int kBins1 = 1 << kD1;
constexpr int kShift1 = 32 - kD1;

// The first digit of a key: a monotone map of the u32 keys onto at most kBins1 bins,
// each an exact prefix range of keys.  QSA_SEL_FINE_DIGIT = 0: the top kD1 key bits.
// QSA_SEL_FINE_DIGIT = 1: keys whose sign-and-exponent field e = key >> 23 lies below
// kFineLo or from kFineHi on take one bin an exponent (2^23 keys); the positive values
// of the octaves around 1.0 take finer bins (1024 bins: 64 an octave over [2^-4, 2^4),
// key >> 17), so that the bin of the 512th key of a row of relu-summed logits holds
// tens of keys instead of hundreds.  Which keys are selected does not depend on the map.
#ifndef QSA_SEL_FINE_DIGIT
#define QSA_SEL_FINE_DIGIT 1
#endif
// 2048 bins: 128 bins an octave over [2^-6, 2^6); 1024 bins: 64 an octave over [2^-4, 2^4)
constexpr int kFineShift = kD1 >= 11 ? 16 : 17;                  // fine bins: key >> kFineShift
constexpr uint32_t kFineOctaves = kD1 >= 11 ? 6u : 4u;           // on each side of 1.0
constexpr uint32_t kFineLo = 256u + 127u - kFineOctaves;         // e of +2^-kFineOctaves
constexpr uint32_t kFineHi = 256u + 127u + kFineOctaves;
constexpr uint32_t kFineBins = (kFineHi - kFineLo) << (23 - kFineShift);
static_assert(kFineLo + kFineBins + (511u - kFineHi) < static_cast<uint32_t>(kBins1) || !QSA_SEL_FINE_DIGIT,
              "the fine first digit does not fit the bins");

// The three pieces (e below kFineLo, the fine bins, e - kFineHi + kFineLo + kFineBins from
// kFineHi on) as min(max(e, fine), high): below kFineLo the fine term is the smaller (it
// falls 2^(23 - kFineShift) a step of e, e by one), inside the fine range it is the larger,
// and from kFineHi on the high term is below it.  Six integer operations, no selects.
__device__ __forceinline__ uint32_t digit1(uint32_t key) {
#if QSA_SEL_FINE_DIGIT
  const int32_t e = static_cast<int32_t>(key >> 23);
  const int32_t fine = static_cast<int32_t>(key >> kFineShift) -
                       static_cast<int32_t>((kFineLo << (23 - kFineShift)) - kFineLo);
  const int32_t high = e - static_cast<int32_t>(kFineHi - kFineLo - kFineBins);
  return static_cast<uint32_t>(min(max(e, fine), high));
#else
  return key >> kShift1;
#endif
}

// the key range [lo, lo + 2^top - 1] of first-digit bin b
__device__ __forceinline__ void digit1_range(uint32_t b, uint32_t& lo, int& top) {
#if QSA_SEL_FINE_DIGIT
  if (b < kFineLo) {
    lo = b << 23;
    top = 23;
  } else if (b < kFineLo + kFineBins) {
    lo = (b - kFineLo + (kFineLo << (23 - kFineShift))) << kFineShift;
    top = kFineShift;
  } else {
    lo = (b - kFineLo - kFineBins + kFineHi) << 23;
    top = 23;
  }
#else
  lo = b << kShift1;
  top = kShift1;
#endif
}
constexpr int kSuper = kBins1 / 128;   // 128-bin super-bins for the two-level search
constexpr int kCpl = 16;               // listed candidates a lane of warp 0 may hold
constexpr int kWarpCap = 32 * kCpl;
constexpr int kMaxBlocks = 65536;
static_assert(kWarpCap <= kBins1, "the candidate list reuses the histogram's storage");

// Shared state of one row's selection.  After the threshold search the first-digit
// histogram is dead, and its storage holds the later steps' data: the candidate list
// (words [0, kWarpCap)), the radix counts (words [kHist2Word, +256)), the candidates'
// classes (bytes from word kClsWord) and, last, the winners (words [0, kTopK)).  Each
// reuse is separated from the previous use by CTA barriers.
constexpr int kHist2Word = kBins1 >= 2048 ? 1024 : kWarpCap;
constexpr int kClsWord = kBins1 >= 2048 ? 1536 : kHist2Word + 256;
static_assert(kWarpCap <= kHist2Word && kTopK <= kHist2Word && kHist2Word + 256 <= kClsWord &&
                  kClsWord + kWarpCap / 4 <= kBins1,
              "selection shared-memory layout");

template <int T>
struct SelShared {
  uint32_t hist1[kBins1];
  uint32_t warp_tot[T / 32];
  uint32_t thr_bin, thr_above, thr_count, ncand;
  int32_t rem;
  uint32_t recount;  // given first-digit counts that do not total the row's keys
  __device__ __forceinline__ uint32_t* hist2() { return hist1 + kHist2Word; }
  __device__ __forceinline__ uint8_t* cls() { return reinterpret_cast<uint8_t*>(hist1 + kClsWord); }
  __device__ __forceinline__ int32_t* win() { return reinterpret_cast<int32_t*>(hist1); }
};

// The visible keys of one row.
struct GlobalKeys {
  const float* p;
  bool vec;  // p is 16-byte aligned
  __device__ __forceinline__ float4 ld4(int32_t g) const { return __ldg(reinterpret_cast<const float4*>(p + g)); }
  __device__ __forceinline__ float ld1(int32_t g) const { return __ldg(p + g); }
};

// Keys written earlier in the same launch by other CTAs: loaded at L2 (ld.global.cg),
// never from a possibly stale L1 line.
struct L2Keys {
  const float* p;
  bool vec;  // p is 16-byte aligned
  __device__ __forceinline__ float4 ld4(int32_t g) const { return __ldcg(reinterpret_cast<const float4*>(p + g)); }
  __device__ __forceinline__ float ld1(int32_t g) const { return __ldcg(p + g); }
};

// exclusive scan of one value per thread over the CTA of T threads
template <int T>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += x;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint32_t base = 0;
#pragma unroll
  for (int w = 0; w < T / 32; ++w)
    if (w < warp) base += warp_tot[w];
  __syncthreads();  // warp_tot may be reused by the next scan
  return base + incl - v;
}

struct Threshold {
  uint32_t bin, above, count;
};

__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += x;
  }
  return v;
}

// The lane whose bins hold the k-th count (`hit`) walks its NB bins, highest first,
// from running count c; the result goes to every lane.
template <int NB>
__device__ __forceinline__ Threshold walk_and_share(const uint32_t (&bins)[NB], uint32_t top, uint32_t c,
                                                    uint32_t k, bool hit) {
  Threshold th{0u, 0u, 0u};
  if (hit) {
    bool done = false;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      if (!done) {
        if (c + bins[j] >= k) {
          th = Threshold{top - j, c, bins[j]};
          done = true;
        } else {
          c += bins[j];
        }
      }
    }
  }
  const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
  th.bin = __shfl_sync(0xffffffffu, th.bin, src);
  th.above = __shfl_sync(0xffffffffu, th.above, src);
  th.count = __shfl_sync(0xffffffffu, th.count, src);
  return th;
}

// One warp: walk the kBins1 bins from the highest down to where the running count
// reaches k (1 <= k <= total).  128-bin super-bins are summed first (a 16-byte load
// and a warp reduction each); the chosen one is searched 4 bins a lane.  *total: the sum
// of every bin.
__device__ __forceinline__ Threshold find_first_digit(const uint32_t* hist, uint32_t k, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  const uint4* h4 = reinterpret_cast<const uint4*>(hist);
  uint32_t ssum[kSuper];
  uint32_t all = 0u;
#pragma unroll
  for (int s = 0; s < kSuper; ++s) {
    const uint4 v = h4[s * 32 + lane];
    ssum[s] = __reduce_add_sync(0xffffffffu, v.x + v.y + v.z + v.w);
    all += ssum[s];
  }
  *total = all;
  uint32_t cum = 0;
  int sstar = 0;
  bool found = false;
#pragma unroll
  for (int s = kSuper - 1; s >= 0; --s) {
    if (!found) {
      if (cum + ssum[s] >= k) {
        sstar = s;
        found = true;
      } else {
        cum += ssum[s];
      }
    }
  }
  const uint4 v = h4[sstar * 32 + 31 - lane];  // lane 0 holds the super-bin's top 4 bins
  const uint32_t b4[4] = {v.w, v.z, v.y, v.x};
  const uint32_t mine = v.x + v.y + v.z + v.w;
  const uint32_t incl = cum + warp_inclusive_sum(mine, lane);
  const uint32_t excl = incl - mine;
  const uint32_t top = static_cast<uint32_t>(sstar) * 128u + 4u * static_cast<uint32_t>(31 - lane) + 3u;
  return walk_and_share(b4, top, excl, k, excl < k && k <= incl);
}

// One warp: the same over 256 bins, 8 a lane.
__device__ __forceinline__ Threshold find_digit256(const uint32_t* hist, uint32_t k) {
  const int lane = threadIdx.x & 31;
  const uint4* h4 = reinterpret_cast<const uint4*>(hist);
  const uint4 lo = h4[2 * (31 - lane)], hi = h4[2 * (31 - lane) + 1];
  const uint32_t b8[8] = {hi.w, hi.z, hi.y, hi.x, lo.w, lo.z, lo.y, lo.x};
  uint32_t mine = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) mine += b8[j];
  const uint32_t incl = warp_inclusive_sum(mine, lane);
  const uint32_t excl = incl - mine;
  return walk_and_share(b8, 8u * static_cast<uint32_t>(31 - lane) + 7u, excl, k, excl < k && k <= incl);
}

#ifndef QSA_SEL_P1_UNROLL
#define QSA_SEL_P1_UNROLL 1
#endif
constexpr int kP1Unroll = QSA_SEL_P1_UNROLL;
#ifndef QSA_SEL_GATHER
#define QSA_SEL_GATHER 4
#endif
constexpr int kGather = QSA_SEL_GATHER;  // candidate-key loads a lane keeps in flight

// f(key) for every visible block, T-strided (coalesced / conflict-free).
template <int T, class K, class F>
__device__ __forceinline__ void for_each_key(const K& keys, int32_t n, F&& f) {
  int32_t g = threadIdx.x;
  if (keys.vec) {
    const int32_t nv = n >> 2;
#pragma unroll kP1Unroll
    for (int32_t v = threadIdx.x; v < nv; v += T) {
      const float4 x = keys.ld4(4 * v);
      f(orderable(x.x));
      f(orderable(x.y));
      f(orderable(x.z));
      f(orderable(x.w));
    }
    g = 4 * nv + threadIdx.x;
  }
  for (; g < n; g += T) f(orderable(keys.ld1(g)));
}

// The selection of one visible row (n_vis > 512 keys): winners' block ids, ascending,
// in sh.win()[0, 512).  Ends with a CTA barrier.  kRegs (MW == 1 only): each thread loads
// its 32 contiguous keys once and keeps them in registers, so the ordered pass and the
// candidate resolution read no key from memory again.
template <int T, int MW, bool kRegs = false, class K>
__device__ __forceinline__ void select_row(const K& keys, int32_t n_vis, SelShared<T>& sh,
                                           uint32_t* ghist = nullptr, uint8_t* codes = nullptr) {
  static_assert(!kRegs || MW == 1, "keys in registers: one 32-key word a thread");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t k_sel = kTopK;
  // 32-key words a thread owns in this row: as few as the row needs, so that short rows
  // spread over every warp of the CTA (words past wpt stay empty)
  const int wpt = kRegs ? 1 : min(MW, static_cast<int>((n_vis + 32 * T - 1) / (32 * T)));
  const int32_t g0 = tid * (32 * wpt);

  // ---- 1. first-digit histogram and its threshold bin.  ghist (optional, 16-byte
  // aligned): the row's kBins1 first-digit counts, added by the kernels that wrote the
  // keys and made visible to this CTA; they are copied (loads issued before the keys')
  // and ghist is left zeroed for the next row that counts into it.
  constexpr int kHq = (kBins1 / 4 + T - 1) / T;  // 16-byte pieces of ghist a thread copies
  uint4 gh[kHq];
  if (ghist != nullptr) {
#pragma unroll
    for (int q = 0; q < kHq; ++q)
      if (tid + q * T < kBins1 / 4) gh[q] = __ldcg(reinterpret_cast<const uint4*>(ghist) + tid + q * T);
  }
  uint32_t kr[kRegs ? 32 : 1];  // kRegs: keys of blocks g0 .. g0 + 31 (those >= n_vis unused)
  if constexpr (kRegs) {
    if (keys.vec && g0 + 32 <= n_vis) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float4 x = keys.ld4(g0 + 4 * e);
        kr[4 * e] = orderable(x.x);
        kr[4 * e + 1] = orderable(x.y);
        kr[4 * e + 2] = orderable(x.z);
        kr[4 * e + 3] = orderable(x.w);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) kr[e] = g0 + e < n_vis ? orderable(keys.ld1(g0 + e)) : 0u;
    }
  }
#pragma unroll
  for (int q = 0; q < kHq; ++q) {
    const int k = tid + q * T;
    if (k < kBins1 / 4) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (ghist != nullptr) {
        v = gh[q];
        __stcg(reinterpret_cast<uint4*>(ghist) + k, make_uint4(0u, 0u, 0u, 0u));
      }
      reinterpret_cast<uint4*>(sh.hist1)[k] = v;
    }
  }
  if (tid == 0) sh.ncand = 0;
  __syncthreads();
  // the row's own first-digit counts (when ghist gives none, or gives counts that do not
  // total the row's keys: then the search below finds recount set, and the CTA counts here)
  auto count_keys = [&]() {
    if constexpr (kRegs) {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (g0 + e < n_vis) atomicAdd(&sh.hist1[digit1(kr[e])], 1u);
    } else if (codes != nullptr) {
      // codes (n_vis <= 32 * T * MW bytes, 16-byte aligned): each key's first digit >> 2,
      // so that the ordered pass reads one byte a key instead of the row.  Key l of a
      // 32-key block has its code at byte l >> 3 of the block's word l & 7: the ordered
      // pass compares a word's four codes at once, and one shift a word puts their flags
      // at bits l of the block's masks
      int32_t g = tid;
      if (keys.vec) {
        const int32_t nv = n_vis >> 2;
        for (int32_t v = tid; v < nv; v += T) {
          const float4 x = keys.ld4(4 * v);
          const uint32_t d0 = digit1(orderable(x.x)), d1 = digit1(orderable(x.y));
          const uint32_t d2 = digit1(orderable(x.z)), d3 = digit1(orderable(x.w));
          atomicAdd(&sh.hist1[d0], 1u);
          atomicAdd(&sh.hist1[d1], 1u);
          atomicAdd(&sh.hist1[d2], 1u);
          atomicAdd(&sh.hist1[d3], 1u);
          // keys 4v + j: byte ((v & 7) >> 1) of word 4 (v & 1) + j of their 32-key block
          uint8_t* cp = codes + 32 * (v >> 3) + 16 * (v & 1) + ((v & 7) >> 1);
          cp[0] = static_cast<uint8_t>(d0 >> 2);
          cp[4] = static_cast<uint8_t>(d1 >> 2);
          cp[8] = static_cast<uint8_t>(d2 >> 2);
          cp[12] = static_cast<uint8_t>(d3 >> 2);
        }
        g = 4 * nv + tid;
      }
      for (; g < n_vis; g += T) {
        const uint32_t d = digit1(orderable(keys.ld1(g)));
        atomicAdd(&sh.hist1[d], 1u);
        codes[32 * (g >> 5) + 4 * (g & 7) + ((g >> 3) & 3)] = static_cast<uint8_t>(d >> 2);
      }
    } else {
      for_each_key<T>(keys, n_vis, [&](uint32_t key) { atomicAdd(&sh.hist1[digit1(key)], 1u); });
    }
  };
  auto search = [&]() {
    if (warp == 0) {
      uint32_t total;
      const Threshold th = find_first_digit(sh.hist1, static_cast<uint32_t>(k_sel), &total);
      if (lane == 0) {
        sh.thr_bin = th.bin;
        sh.thr_above = th.above;
        sh.thr_count = th.count;
        sh.recount = total != static_cast<uint32_t>(n_vis) ? 1u : 0u;
      }
    }
    __syncthreads();
  };
  if (ghist == nullptr) {
    count_keys();
    __syncthreads();
  }
  search();
  if (ghist != nullptr && sh.recount != 0u) {  // CTA-uniform
    for (int k = tid; k < kBins1 / 4; k += T) reinterpret_cast<uint4*>(sh.hist1)[k] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    count_keys();
    __syncthreads();
    search();
  }
  const uint32_t b1 = sh.thr_bin;
  const uint32_t c1 = sh.thr_count;
  int32_t rem = k_sel - static_cast<int32_t>(sh.thr_above);
  const bool exact1 = c1 == static_cast<uint32_t>(rem);
  const bool listed = !exact1 && c1 <= static_cast<uint32_t>(kWarpCap);
  uint32_t lo1;
  int top1;
  digit1_range(b1, lo1, top1);
  const uint32_t hi1 = lo1 | ((1u << top1) - 1u);

  // ---- 2. ordered pass over this thread's contiguous blocks (keys in registers:
  // branch-free bit masks, key in [lo1, hi1] as one unsigned compare, the word's keys
  // past n_vis masked off)
  const uint32_t span1 = hi1 - lo1;
  uint32_t gtm[MW], cm[MW];
#pragma unroll
  for (int w = 0; w < MW; ++w) {
    gtm[w] = 0u;
    cm[w] = 0u;
    const int32_t gb = g0 + 32 * w;
    if (w >= wpt) {
      // not this row's word
    } else if constexpr (kRegs) {
      uint32_t gt = 0u, in = 0u;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        gt |= static_cast<uint32_t>(kr[e] > hi1) << e;
        in |= static_cast<uint32_t>(kr[e] - lo1 <= span1) << e;
      }
      const int32_t nk = n_vis - gb;  // keys of this word that exist
      const uint32_t valid = nk >= 32 ? 0xFFFFFFFFu : (nk > 0 ? (1u << nk) - 1u : 0u);
      gtm[w] = gt & valid;
      cm[w] = in & valid;
    } else if (codes != nullptr) {
      // keys whose code is above b1's are selected, below it out; the few that share b1's
      // code (four first-digit bins) are compared exactly, their keys reloaded.  Four
      // codes a word at once: x > cb is the carry out of each byte of x + (255 - cb)
      // (bit 7 of the byte sum of the low seven bits, then the majority of the three
      // bit-7 inputs), x == cb a zero byte of x ^ cb (exact: (t & 0x7F) + 0x7F sets bit 7
      // unless t's low bits are zero); byte b's flag of word q lands at bit 8b + q
      const uint32_t cb = b1 >> 2;
      const int32_t nk = n_vis - gb;
      const uint32_t valid = nk >= 32 ? 0xFFFFFFFFu : (nk > 0 ? (1u << nk) - 1u : 0u);
      uint32_t gt = 0u, amb = 0u;
      const uint4* c16 = reinterpret_cast<const uint4*>(codes + gb);
      const uint32_t c4 = cb * 0x01010101u, nc4 = ~c4, ncl = nc4 & 0x7F7F7F7Fu;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 c = c16[h];
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const uint32_t x = cw[qq];
          const uint32_t s = (x & 0x7F7F7F7Fu) + ncl;  // bit 7 of a byte: carry into bit 7 of x + ~cb
          const uint32_t g = ((x & nc4) | (x & s) | (nc4 & s)) & 0x80808080u;  // carry out: x > cb
          const uint32_t t = x ^ c4;
          const uint32_t y = (t & 0x7F7F7F7Fu) + 0x7F7F7F7Fu;
          const uint32_t e = ~(y | t) & 0x80808080u;  // t's zero bytes: x == cb
          gt |= g >> (7 - (4 * h + qq));
          amb |= e >> (7 - (4 * h + qq));
        }
      }
      gt &= valid;
      amb &= valid;
      uint32_t in = 0u;
      while (amb != 0u) {  // up to four reloads in flight
        int e4[4];
        float x4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          e4[u] = amb != 0u ? __ffs(amb) - 1 : -1;
          amb &= amb - 1u;
          x4[u] = e4[u] >= 0 ? keys.ld1(gb + e4[u]) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (e4[u] >= 0) {
            const uint32_t key = orderable(x4[u]);
            gt |= static_cast<uint32_t>(key > hi1) << e4[u];
            in |= static_cast<uint32_t>(key - lo1 <= span1) << e4[u];
          }
        }
      }
      gtm[w] = gt;
      cm[w] = in;
    } else if (keys.vec && gb + 32 <= n_vis) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float4 x = keys.ld4(gb + 4 * e);
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t key = orderable(xs[j]);
          const uint32_t bit = 1u << (4 * e + j);
          if (key > hi1) gtm[w] |= bit;
          if (key >= lo1 && key <= hi1) cm[w] |= bit;
        }
      }
    } else if (gb < n_vis) {
      const int32_t n = n_vis - gb;  // ragged: fewer than 32, or unaligned
#pragma unroll 4
      for (int e = 0; e < 32; ++e) {
        if (e < n) {
          const uint32_t key = orderable(keys.ld1(gb + e));
          if (key > hi1) gtm[w] |= 1u << e;
          if (key >= lo1 && key <= hi1) cm[w] |= 1u << e;
        }
      }
    }
  }
  uint32_t my_cand = 0, cbase = 0;
  if (listed) {
#pragma unroll
    for (int w = 0; w < MW; ++w) my_cand += __popc(cm[w]);
    if (my_cand) {
      cbase = atomicAdd(&sh.ncand, my_cand);
      uint32_t j = cbase;
      if constexpr (kRegs) {  // the keys themselves, in ascending block order
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if ((cm[0] >> e) & 1u) sh.hist1[j++] = kr[e];
      } else if (codes != nullptr) {  // the keys themselves, reloaded (L1 since the ordered pass)
#pragma unroll
        for (int w = 0; w < MW; ++w) {
          uint32_t m = cm[w];
          while (m) {
            sh.hist1[j++] = orderable(keys.ld1(g0 + 32 * w + __ffs(m) - 1));
            m &= m - 1u;
          }
        }
      } else {  // block ids; warp 0 loads their keys
#pragma unroll
        for (int w = 0; w < MW; ++w) {
          uint32_t m = cm[w];
          while (m) {
            sh.hist1[j++] = static_cast<uint32_t>(g0 + 32 * w + __ffs(m) - 1);
            m &= m - 1u;
          }
        }
      }
    }
  }
  __syncthreads();

  // ---- 3. resolve the threshold inside bin b1
  if (listed) {
    if (warp == 0) {
      const uint32_t nc = c1;
      const int nq = static_cast<int>((nc + 31u) >> 5);
      if (!kRegs && codes == nullptr) {
        // candidates' keys, in place of their block ids: kGather loads in flight a lane
        // before their stores, so the L2 round trips overlap
        for (int q0 = 0; q0 < nq; q0 += kGather) {
          float x[kGather];
#pragma unroll
          for (int u = 0; u < kGather; ++u) {
            const uint32_t j = lane + 32u * (q0 + u);
            x[u] = q0 + u < nq && j < nc ? keys.ld1(static_cast<int32_t>(sh.hist1[j])) : 0.0f;
          }
#pragma unroll
          for (int u = 0; u < kGather; ++u) {
            const uint32_t j = lane + 32u * (q0 + u);
            if (q0 + u < nq && j < nc) sh.hist1[j] = orderable(x[u]);
          }
        }
        __syncwarp();
      }
      uint32_t prefix = lo1, mask = ~((1u << top1) - 1u);
      int32_t rm = rem;
#pragma unroll 1
      for (int top = top1; top > 0;) {
        const int width = min(8, top);
        const int shift = top - width;
        const uint32_t dmask = (1u << width) - 1u;
        reinterpret_cast<uint4*>(sh.hist2())[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(sh.hist2())[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
        for (int q = 0; q < nq; ++q) {
          const uint32_t j = lane + 32u * q;
          if (j < nc) {
            const uint32_t key = sh.hist1[j];
            if ((key & mask) == prefix) atomicAdd(&sh.hist2()[(key >> shift) & dmask], 1u);
          }
        }
        __syncwarp();
        const Threshold th = find_digit256(sh.hist2(), static_cast<uint32_t>(rm));
        rm -= static_cast<int32_t>(th.above);
        prefix |= th.bin << shift;
        mask |= dmask << shift;
        top = shift;
        if (th.count == static_cast<uint32_t>(rm)) break;
        __syncwarp();  // every lane has read hist2 before it is cleared
      }
      const uint32_t lo = prefix, hi = prefix | ~mask;
      for (int q = 0; q < nq; ++q) {
        const uint32_t j = lane + 32u * q;
        if (j < nc) {
          const uint32_t key = sh.hist1[j];
          sh.cls()[j] = key > hi ? 2 : (key >= lo ? 1 : 0);
        }
      }
      if (lane == 0) sh.rem = rm;
    }
    __syncthreads();
    rem = sh.rem;
    if (my_cand) {  // this thread's candidates sit at [cbase, cbase + my_cand), ascending
      uint32_t j = cbase;
#pragma unroll
      for (int w = 0; w < MW; ++w) {
        uint32_t m = cm[w];
        while (m) {
          const uint32_t bit = m & (0u - m);
          m &= m - 1u;
          const uint8_t k = sh.cls()[j++];
          if (k == 2) gtm[w] |= bit;
          if (k != 1) cm[w] &= ~bit;
        }
      }
    }
  } else if (!exact1) {  // more candidates than warp 0 holds: passes over the row
    uint32_t prefix = lo1, mask = ~((1u << top1) - 1u);
#pragma unroll 1
    for (int top = top1; top > 0;) {
      const int width = min(8, top);
      const int shift = top - width;
      const uint32_t dmask = (1u << width) - 1u;
      for (int k = tid; k < 256; k += T) sh.hist2()[k] = 0u;
      __syncthreads();
      if constexpr (kRegs) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (g0 + e < n_vis && (kr[e] & mask) == prefix) atomicAdd(&sh.hist2()[(kr[e] >> shift) & dmask], 1u);
      } else {
        for_each_key<T>(keys, n_vis, [&](uint32_t key) {
          if ((key & mask) == prefix) atomicAdd(&sh.hist2()[(key >> shift) & dmask], 1u);
        });
      }
      __syncthreads();
      if (warp == 0) {
        const Threshold th = find_digit256(sh.hist2(), static_cast<uint32_t>(rem));
        if (lane == 0) {
          sh.thr_bin = th.bin;
          sh.thr_above = th.above;
          sh.thr_count = th.count;
        }
      }
      __syncthreads();
      rem -= static_cast<int32_t>(sh.thr_above);
      prefix |= sh.thr_bin << shift;
      mask |= dmask << shift;
      top = shift;
      if (sh.thr_count == static_cast<uint32_t>(rem)) break;
    }
    const uint32_t lo = prefix, hi = prefix | ~mask;
    if constexpr (kRegs) {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        if ((cm[0] >> e) & 1u) {
          if (kr[e] > hi) gtm[0] |= 1u << e;
          if (kr[e] > hi || kr[e] < lo) cm[0] &= ~(1u << e);
        }
      }
    } else {
#pragma unroll
      for (int w = 0; w < MW; ++w) {
        uint32_t m = cm[w];
        while (m) {
          const int bit = __ffs(m) - 1;
          m &= m - 1u;
          const uint32_t key = orderable(keys.ld1(g0 + 32 * w + bit));
          if (key > hi) gtm[w] |= 1u << bit;
          if (key > hi || key < lo) cm[w] &= ~(1u << bit);
        }
      }
    }
  }

  // ---- 4. positions: selected count in bits [0, 10), tied count above
  uint32_t ngt = 0, ntie = 0;
#pragma unroll
  for (int w = 0; w < MW; ++w) {
    ngt += __popc(gtm[w]);
    ntie += __popc(cm[w]);
  }
  const uint32_t ex = block_exclusive_scan<T>(ngt | (ntie << 10), sh.warp_tot);
  const uint32_t rem_u = static_cast<uint32_t>(rem);
  const uint32_t tie_before = ex >> 10;
  uint32_t pos = (ex & 1023u) + min(tie_before, rem_u);
  uint32_t take = tie_before >= rem_u ? 0u : min(rem_u - tie_before, ntie);
#pragma unroll
  for (int w = 0; w < MW; ++w) {
    uint32_t tm = cm[w];
    uint32_t keep = 0u;
    const uint32_t n = __popc(tm);
    if (take >= n) {
      keep = tm;
      take -= n;
    } else {
      while (take) {
        keep |= tm & (0u - tm);
        tm &= tm - 1u;
        --take;
      }
    }
    uint32_t wm = gtm[w] | keep;
    while (wm) {
      sh.win()[pos++] = g0 + 32 * w + __ffs(wm) - 1;
      wm &= wm - 1u;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void st_s32x4(int32_t* p, int32_t a, int32_t b, int32_t c, int32_t d) {
  asm volatile("st.global.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// A selected row's 2051 token ids: win[p] expands to out[4p + j] = 4*win[p] + j
// (16-byte stores from the row's first aligned address on), then the causal tail
// tokens 4*nVis + j for j < tail, then -1.
template <int T>
__device__ __forceinline__ void write_selected(int32_t* out, const int32_t* win, int32_t tail, int32_t n_vis) {
  // every 16-byte-aligned group of four ids with one vector store; the few ids before the
  // row's first aligned address and after its last are written one by one
  const int k0 = static_cast<int>((4u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(out) >> 2) & 3u)) & 3u);
  const int nchunks = (kRatio * kTopK - k0) / 4;
  for (int c = threadIdx.x; c < nchunks; c += T) {
    const int i = k0 + 4 * c;
    int32_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = win[(i + j) >> 2] * kRatio + ((i + j) & 3);
    st_s32x4(out + i, v[0], v[1], v[2], v[3]);
  }
  const int tail_lo = k0 + 4 * nchunks;  // ids [tail_lo, 4 * kTopK): at most 3
  const int t = threadIdx.x;
  if (t < k0) out[t] = win[t >> 2] * kRatio + (t & 3);
  if (t >= k0 && t < k0 + (kRatio * kTopK - tail_lo)) {
    const int i = tail_lo + (t - k0);
    out[i] = win[i >> 2] * kRatio + (i & 3);
  }
  if (t < kRatio - 1) out[kRatio * kTopK + t] = t < tail ? kRatio * n_vis + t : -1;
}

// Rows whose selection needs no logits: padded rows (all -1) and rows with at most
// 512 visible blocks (every block, ascending, then the tail).
template <int T>
__device__ __forceinline__ void write_unselected(int32_t* out, bool padded, int32_t n_vis, int32_t tail) {
  const int32_t n_all = padded ? 0 : kRatio * n_vis + tail;  // token ids 0 .. n_all-1
  for (int k = threadIdx.x; k < kWidth; k += T) out[k] = k < n_all ? k : -1;
}

}  // namespace sel
}  // namespace qsa
