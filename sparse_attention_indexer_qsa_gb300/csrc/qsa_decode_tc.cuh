// Paged decode scores on the tensor cores ("Qsa Indexer Kernels":
// launchQsaIndexScoresDecode), shared by the paged-scores kernel (k_decode.cu) and
// the fused decode step (k_decode_step.cu), so both compute the same bits.
//
// A CTA scores a run of blocks [g_run, g_end) of one sequence b in tiles of 128
// blocks.  The tile's kbar rows (each block's V-tail, 256 bytes) are the MMA's A
// operand: one TMA box per pool page and K half brings 32 blocks (the page's 32
// V-tails, 6 KB apart in the pool) in 128-byte-swizzled K-major layout.  The B
// operand is the sequence's 4 q heads, written once per CTA, padded with zero rows
// to N = 16.  One thread issues 8 tcgen05.mma (M = 128, N = 16, K = 16) per tile
// into one of two TMEM accumulators; four epilogue warps (one per TMEM lane quarter)
// read the 4 head dots of their 32 blocks, take relu, the ascending head sum and the
// scale, and store one coalesced 128-byte row segment each.  The dots are formed as
// in the prefill scoring kernel: the same operand layouts, the same MMA shape along
// K and the same K order.
//
// Roles (warps of the CTA): 0 TMA producer (lane 0; engine_start issues the first
// tiles' copies before the CTA's setup barrier, engine_run the rest), 1 MMA issuer
// (lane 0), 2-5 epilogue.  Warp 1 allocates and frees TMEM.  Every mbarrier wait is bounded; a wait
// that runs out sets a fault bit and the CTA's abort flag, after which the CTA waits
// (bounded) for its own copies and MMAs and returns; that launch's logits are undefined.
#pragma once

#include <cfloat>

#include "qsa_common.cuh"
#include "qsa_launch.h"
#include "qsa_select.cuh"
#include "tc_ptx.cuh"

namespace qsa {
namespace dtc {

constexpr int kTile = 128;                          // blocks a tile (MMA M)
constexpr int kN = 16;                              // MMA N: 4 q heads + 12 zero rows
constexpr int kPagesPerTile = kTile / 32;           // 128-token pages (32 blocks) a tile
constexpr int kStages = 3;
constexpr int kAccStages = 2;
constexpr uint32_t kTmemCols = 32;                  // kAccStages accumulators of kN columns
constexpr uint32_t kAHalf = kTile * 128;            // one 64-element K half of a tile (16 KB)
constexpr uint32_t kABytes = 2 * kAHalf;
constexpr uint32_t kPageBox = 32 * 128;             // one TMA box: 32 rows x 128 bytes
constexpr uint32_t kBHalf = kN * 128;
constexpr uint32_t kBBytes = 2 * kBHalf;
constexpr int kEngineWarps = 6;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
enum : uint32_t { kFaultProducer = 1u, kFaultMma = 2u, kFaultEpilogue = 4u, kFaultDrain = 8u };

constexpr int kBarFull = 0;
constexpr int kBarEmpty = kBarFull + kStages;
constexpr int kBarAccFull = kBarEmpty + kStages;
constexpr int kBarAccEmpty = kBarAccFull + kAccStages;
constexpr int kBarDrain = kBarAccEmpty + kAccStages;
constexpr int kNumBars = kBarDrain + 1;

// Shared memory of the engine (1024-byte aligned base): the stages' A tiles, the B
// operand, barriers, the TMEM address and the abort flag.
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffBar = kOffB + kBBytes;
constexpr uint32_t kOffTmem = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmem + 4;
constexpr uint32_t kEngineBytes = kOffAbort + 4;
static_assert(kOffA % 1024 == 0 && kOffB % 1024 == 0 && kOffBar % 8 == 0, "engine smem misaligned");

struct Engine {
  uint32_t base;              // shared address of the engine region (1024-byte aligned)
  uint8_t* ptr;               // the same region, generic
  uint32_t* fault;            // device fault word of the calling kernel's module
  __device__ __forceinline__ uint32_t bar(int i) const { return base + kOffBar + 8u * static_cast<uint32_t>(i); }
  __device__ __forceinline__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(ptr + kOffAbort);
  }
};

// Wait for the phase of `bar` with the given parity for at most `limit_ns`; on time-out
// set `code` in the fault word and the CTA's abort flag.  Returns false (without
// waiting further) once the abort flag is set by any thread of the CTA.
__device__ __forceinline__ bool wait_bounded_raw(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                 uint32_t* fault, uint32_t code, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t start = ptx::global_timer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::global_timer_ns() - start > limit_ns) {
      atomicOr(fault, code);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bounded(const Engine& en, uint32_t bar, uint32_t parity, uint32_t code) {
  return wait_bounded_raw(bar, parity, en.abort_flag(), en.fault, code, kWaitLimitNs);
}

__device__ __forceinline__ void drain_wait(const Engine& en, uint32_t bar, uint32_t parity) {
  const uint64_t start = ptx::global_timer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::global_timer_ns() - start > kDrainLimitNs) {
      atomicOr(en.fault, kFaultDrain);
      return;
    }
  }
}

// Byte offset, inside the B operand, of the 16-byte chunk holding dims [8c, 8c + 8) of
// row n (128-byte swizzle, K-major, 8-row atoms of 1024 bytes, K halves 2 KB apart).
__device__ __forceinline__ uint32_t b_chunk_offset(int n, int c) {
  const int half = c >> 3, cc = c & 7;
  return static_cast<uint32_t>(half) * kBHalf + static_cast<uint32_t>(n >> 3) * 1024u +
         static_cast<uint32_t>(n & 7) * 128u + static_cast<uint32_t>((cc ^ (n & 7)) * 16);
}

// Zero rows 4..15 of the B operand (every thread of the CTA may call it; threads
// stride by nthreads).
__device__ __forceinline__ void zero_b_padding(const Engine& en, int tid, int nthreads) {
  for (int i = tid; i < (kN - kNumQHeads) * 16; i += nthreads) {
    const int n = kNumQHeads + i / 16, c = i % 16;
    *reinterpret_cast<uint4*>(en.ptr + kOffB + b_chunk_offset(n, c)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Store the 16 bytes of q dims [8c, 8c + 8) of head h into the B operand.
__device__ __forceinline__ void put_q_chunk(const Engine& en, int h, int c, const uint4& v) {
  *reinterpret_cast<uint4*>(en.ptr + kOffB + b_chunk_offset(h, c)) = v;
}

// Whether page j of tile t holds a block of [g_run, g_end) with a usable page slot.
__device__ __forceinline__ bool page_active(const int32_t* pages, int32_t g_run, int32_t g_end, int t, int j) {
  return g_run + kTile * t + 32 * j < g_end && pages[kPagesPerTile * t + j] >= 0;
}

__device__ __forceinline__ int run_tiles(int32_t g_run, int32_t g_end) {
  return g_end > g_run ? (g_end - g_run + kTile - 1) / kTile : 0;
}

// Tiles whose copies engine_start issues before the CTA's setup barrier: at most one
// per stage, and none from tile `limit` on.
__device__ __forceinline__ int pre_tiles(int nt, int limit) { return min(min(nt, kStages), limit); }

// The copies of tile t into stage s, completing on its full barrier (producer thread).
__device__ __forceinline__ void issue_tile(const Engine& en, const CUtensorMap* map, const int32_t* pages,
                                           int32_t head_size, int32_t g_run, int32_t g_end, int t, int s) {
  uint32_t bytes = 0;
#pragma unroll
  for (int j = 0; j < kPagesPerTile; ++j)
    if (page_active(pages, g_run, g_end, t, j)) bytes += 2 * kPageBox;
  ptx::mbar_arrive_expect_tx(en.bar(kBarFull + s), bytes);
  const uint32_t dst = en.base + kOffA + static_cast<uint32_t>(s) * kABytes;
#pragma unroll
  for (int j = 0; j < kPagesPerTile; ++j) {
    if (!page_active(pages, g_run, g_end, t, j)) continue;
    const int32_t row = pages[kPagesPerTile * t + j] * 32;  // the page's first block
    ptx::tma_load_3d(dst + j * kPageBox, map, en.bar(kBarFull + s), head_size, 0, row);
    ptx::tma_load_3d(dst + kAHalf + j * kPageBox, map, en.bar(kBarFull + s), head_size + 64, 0, row);
  }
}

// Warp 0, before the CTA's setup barrier (after it staged `pages` and a __syncwarp):
// lane 0 initialises the barriers and issues the copies of the first
// pre_tiles(nt, limit) tiles, so that they are in flight while the other warps prepare.
__device__ __forceinline__ void engine_start(const Engine& en, const CUtensorMap* map, const int32_t* pages,
                                             int32_t head_size, int32_t g_run, int32_t g_end, int limit) {
  if ((threadIdx.x & 31) != 0) return;
  for (int s = 0; s < kStages; ++s) {
    ptx::mbar_init(en.bar(kBarFull + s), 1);
    ptx::mbar_init(en.bar(kBarEmpty + s), 1);
  }
  for (int s = 0; s < kAccStages; ++s) {
    ptx::mbar_init(en.bar(kBarAccFull + s), 1);
    ptx::mbar_init(en.bar(kBarAccEmpty + s), 4);
  }
  ptx::mbar_init(en.bar(kBarDrain), 1);
  *en.abort_flag() = 0;
  ptx::fence_barrier_init();
  ptx::prefetch_tensormap(map);
  const int np = pre_tiles(run_tiles(g_run, g_end), limit);
  for (int t = 0; t < np; ++t) issue_tile(en, map, pages, head_size, g_run, g_end, t, t);
}

// One warp, after the CTA barrier that follows engine_start, before engine_setup: once
// the copies of tile t (one engine_start issued) have landed, lanes 0-7 overwrite the A
// operand row of the tile's block rr (0 <= rr < kTile) with the 128 T values whose
// chunks at element offsets ca and cb they hold (chunk_a / chunk_b of the lane), in the
// 128-byte-swizzled layout the copies wrote, and fence them for the MMAs.  Returns false
// if the wait ran out (the abort flag is then set).
__device__ __forceinline__ bool patch_a_row(const Engine& en, int t, int rr, int lane, int ca, int cb, uint4 va,
                                            uint4 vb) {
  const int s = t % kStages;
  if (!wait_bounded(en, en.bar(kBarFull + s), (t / kStages) & 1, kFaultEpilogue)) return false;
  if (lane < 8) {
    const int r = rr & 31;  // row of the 32-row page box, which starts 1024-byte aligned
    const uint32_t box = kOffA + static_cast<uint32_t>(s) * kABytes + static_cast<uint32_t>(rr >> 5) * kPageBox +
                         static_cast<uint32_t>(r) * 128u;
    const int e2[2] = {ca, cb};
    const uint4 v2[2] = {va, vb};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t half = static_cast<uint32_t>(e2[k] >> 6), c = static_cast<uint32_t>((e2[k] & 63) >> 3);
      *reinterpret_cast<uint4*>(en.ptr + box + half * kAHalf + ((c ^ static_cast<uint32_t>(r & 7)) << 4)) = v2[k];
    }
  }
  ptx::fence_proxy_async_shared();
  return true;
}

// TMEM; every thread of the CTA calls it after engine_start (contains __syncthreads).
// The caller has written the B operand (and fenced it for the async proxy) before.
__device__ __forceinline__ uint32_t engine_setup(const Engine& en) {
  if ((threadIdx.x >> 5) == 1) {
    __syncwarp();
    ptx::tmem_alloc(en.base + kOffTmem, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return *reinterpret_cast<volatile uint32_t*>(en.ptr + kOffTmem);
}

// Frees TMEM; every thread of the CTA calls it after its role (contains __syncthreads).
__device__ __forceinline__ void engine_teardown(uint32_t tmem) {
  ptx::tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// The roles over the run's tiles, after engine_setup.  pages: stage_vpages of the run
// (visible to every thread); out: the sequence's logits row; pool map: 3-D
// {poolHeadDim, 4 x numKVHeads, 2 x numPages x 32} over the pool, box {64, 1, 32},
// 128-byte swizzle; limit: the one given to engine_start; hist (optional): the row's
// first-digit histogram of the selection (sel::digit1 bins), to which every logit the
// run writes adds one.  Warps 6+ (if any) return at once.
template <bool kBf16>
__device__ __forceinline__ void engine_run(const Engine& en, uint32_t tmem, const CUtensorMap* map,
                                           const int32_t* pages, int32_t head_size, int32_t g_run, int32_t g_end,
                                           float* out, float scale, int limit, uint32_t* hist = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = run_tiles(g_run, g_end);
  if (warp == 0) {
    if (lane != 0) return;
    // ------------------------------------------- producer (after engine_start's tiles)
    int t = pre_tiles(nt, limit);
    for (; t < nt; ++t) {
      const int s = t % kStages;
      if (!wait_bounded(en, en.bar(kBarEmpty + s), ((t / kStages) & 1) ^ 1, kFaultProducer)) break;
      issue_tile(en, map, pages, head_size, g_run, g_end, t, s);
    }
    if (*en.abort_flag()) {  // the last copy issued into each stage lands before the CTA exits
      for (int s = 0; s < kStages; ++s)
        if (t > s) {
          const int n = ((t - 1 - s) / kStages) * kStages + s;
          drain_wait(en, en.bar(kBarFull + s), (n / kStages) & 1);
        }
    }
  } else if (warp == 1) {
    if (lane != 0) return;
    // -------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = ptx::idesc_f16(kBf16, kTile, kN);
    const uint32_t b_addr = en.base + kOffB;
    int t = 0;
    for (; t < nt; ++t) {
      const int s = t % kStages, a = t % kAccStages;
      if (!wait_bounded(en, en.bar(kBarFull + s), (t / kStages) & 1, kFaultMma) ||
          !wait_bounded(en, en.bar(kBarAccEmpty + a), ((t / kAccStages) & 1) ^ 1, kFaultMma))
        break;
      ptx::tc_fence_after();
      const uint32_t a_addr = en.base + kOffA + static_cast<uint32_t>(s) * kABytes;
      const uint32_t d = tmem + static_cast<uint32_t>(a) * kN;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = static_cast<uint32_t>(kk & 3) * 32u;
        const uint64_t adesc = ptx::smem_desc_sw128(a_addr + (kk >> 2) * kAHalf + koff);
        const uint64_t bdesc = ptx::smem_desc_sw128(b_addr + (kk >> 2) * kBHalf + koff);
        ptx::mma_f16(d, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
      }
      ptx::mma_commit(en.bar(kBarEmpty + s));
      ptx::mma_commit(en.bar(kBarAccFull + a));
    }
    if (t > 0) {  // every MMA (and the arrivals committed after it) completes before TMEM is freed
      ptx::mma_commit(en.bar(kBarDrain));
      drain_wait(en, en.bar(kBarDrain), 0);
    }
  } else if (warp < kEngineWarps) {
    // ---------------------------------------------------------------- epilogue
    const int sp = warp & 3;  // TMEM lane quarter: blocks 32 sp .. 32 sp + 31 of a tile
    for (int t = 0; t < nt; ++t) {
      const int a = t % kAccStages;
      const int32_t g = g_run + kTile * t + 32 * sp + lane;
      if (!wait_bounded(en, en.bar(kBarAccFull + a), (t / kAccStages) & 1, kFaultEpilogue)) break;
      ptx::tc_fence_after();
      uint32_t r[4];
      ptx::tmem_ld_32x32b_x4(tmem + (static_cast<uint32_t>(32 * sp) << 16) + static_cast<uint32_t>(a) * kN, r);
      ptx::tmem_ld_wait4(r);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(en.bar(kBarAccEmpty + a));
      if (g < g_end) {  // the block's page was staged
        const bool usable = pages[kPagesPerTile * t + sp] >= 0;
        float v = __fadd_rn(fmaxf(0.0f, __uint_as_float(r[0])), fmaxf(0.0f, __uint_as_float(r[1])));
        v = __fadd_rn(v, fmaxf(0.0f, __uint_as_float(r[2])));
        v = __fadd_rn(v, fmaxf(0.0f, __uint_as_float(r[3])));
        const float logit = usable ? __fmul_rn(v, scale) : -FLT_MAX;
        out[g] = logit;
        if (hist != nullptr) atomicAdd(hist + sel::digit1(sel::orderable(logit)), 1u);
      }
    }
  }
}

}  // namespace dtc
}  // namespace qsa
