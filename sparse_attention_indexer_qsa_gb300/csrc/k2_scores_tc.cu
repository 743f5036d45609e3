// K2: causal block-relevance logits on the tcgen05 tensor cores
// ("Qsa Indexer Kernels", launchQsaIndexScores):
//   logits[r][g] = (1/sqrtf(128)) * sum_{h ascending} max(0, q[r][h] . kbar[b][g])
// for g < (t+1)/4 on rows with t < contextLengths[b]; -FLT_MAX elsewhere.
//
// GEMM mapping (roles chosen so the epilogue needs no shuffles and stores coalesce):
//   A (M = 128)  = 128 kbar blocks g of one sequence, K-major, 128 dims
//   B (N = 256)  = 64 tokens x 4 heads of qNormed ([.., 4, 128] rows are exactly
//                  the K-major B rows), so TMEM lane = block g, column = 4*token + head
//   D            = FP32 in TMEM, two 256-column accumulators (all 512 columns)
// An epilogue thread owns one block g (one TMEM lane): it reads 4 heads of a token
// from 4 consecutive columns, applies relu per head, sums them in ascending h, scales
// and masks, and the 32 lanes of a warp write 32 consecutive logits (128 bytes).
//
// Persistent CTA per SM, warp-specialised, with work units taken dynamically in
// address order from a device-wide counter (statically assigned persistent CTAs
// drift apart and spread the live write front over DRAM, which costs ~15% of HBM
// write bandwidth on GB300):
//   warp 0     scheduler + TMA producer (q tile once per unit, kbar tiles per MMA g-tile)
//   warp 1     TMEM allocator + single-thread MMA issuer
//   warps 2+   epilogue (kEpiWarps: two or four per TMEM sub-partition, each a token slice)
// A work unit is (sequence b, 64-token tile, every n_groups-th g-tile of 128 blocks).
// Tiles whose blocks are all masked for every stored row skip the MMA and only store
// -FLT_MAX.  Rows outside the chunk or the sequence are computed but never stored;
// TMA reads past the end of a sequence's q or kbar rows return zeros.
//
// Every mbarrier wait is bounded (about two seconds of %globaltimer).  A wait that
// runs out sets a bit in the device fault word and a CTA-wide abort flag; the CTA
// then waits (bounded) for its own TMA copies and MMAs in flight, frees TMEM and exits.
#include <cfloat>
#include <mutex>

#include <cudaTypedefs.h>

#include "qsa_launch.h"
#include "tc_ptx.cuh"

namespace qsa {

__device__ uint32_t g_fault_flags;

// Work-unit scheduler state of the scoring kernel: kSchedSlots independent
// {next unit, CTAs finished} counter pairs.  Each launch takes the next slot of its
// device (so up to kSchedSlots launches may execute concurrently), CTAs fetch work
// units from it in address order, and the last CTA to finish puts the slot back to
// zero for its next user.  Zero-initialised at module load; never allocated.
constexpr int kSchedSlots = 64;
__device__ __align__(256) uint32_t g_k2_sched[kSchedSlots * 2];

namespace k2 {

constexpr int kTokTile = 64;                  // tokens per tile
constexpr int kN = kTokTile * 4;              // MMA N: token x head rows
constexpr int kGTile = 128;                   // MMA M: kbar blocks per tile
#ifndef QSA_K2_GTILES_PER_UNIT
#define QSA_K2_GTILES_PER_UNIT 8
#endif
constexpr int kGTilesPerUnit = QSA_K2_GTILES_PER_UNIT;
constexpr int kQStages = 2;
constexpr int kKStages = 3;
constexpr int kAccStages = 2;
#ifndef QSA_K2_EPI_WARPS
#define QSA_K2_EPI_WARPS 8
#endif
constexpr int kEpiWarps = QSA_K2_EPI_WARPS;         // 8 or 16
static_assert(kEpiWarps == 8 || kEpiWarps == 16, "epilogue warps: two or four per TMEM sub-partition");
constexpr int kTokPerWarp = kTokTile / (kEpiWarps / 4);  // tokens of a tile per epilogue warp
constexpr int kLdPerWarp = kTokPerWarp / 8;              // 32-column TMEM loads (8 tokens each)
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kQHalfBytes = kN * 64 * 2;       // one 64-element K half of the q tile
constexpr uint32_t kQBytes = 2 * kQHalfBytes;
constexpr uint32_t kKHalfBytes = kGTile * 64 * 2;
constexpr uint32_t kKBytes = 2 * kKHalfBytes;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQStages * kQBytes;
constexpr uint32_t kOffBar = kOffK + kKStages * kKBytes;
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = kBarQFull + kQStages;
constexpr int kBarKFull = kBarQEmpty + kQStages;
constexpr int kBarKEmpty = kBarKFull + kKStages;
constexpr int kBarAccFull = kBarKEmpty + kKStages;
constexpr int kBarAccEmpty = kBarAccFull + kAccStages;
constexpr int kSchedStages = 4;                 // work units published ahead by the producer
constexpr int kBarSchedFull = kBarAccEmpty + kAccStages;
constexpr int kBarSchedEmpty = kBarSchedFull + kSchedStages;
constexpr int kBarDrain = kBarSchedEmpty + kSchedStages;
constexpr int kNumBars = kBarDrain + 1;
constexpr uint32_t kUnitBytes = 48;             // sizeof(Unit), checked below
constexpr uint32_t kOffRing = (kOffBar + kNumBars * 8 + 15u) & ~15u;  // 16-byte aligned entries
constexpr uint32_t kOffTmemSlot = kOffRing + kSchedStages * kUnitBytes;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1024
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
static_assert(kOffRing % 16 == 0 && kOffBar % 8 == 0 && kOffQ % 1024 == 0 && kOffK % 1024 == 0,
              "shared-memory regions misaligned");

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
enum : uint32_t {
  kFaultProducer = 1u,
  kFaultMma = 2u,
  kFaultEpilogue = 4u,
  kFaultDrain = 8u,
};

struct Params {
  uint32_t* sched;          // this launch's scheduler slot: {next unit, CTAs finished}
  float* logits;
  const int32_t* ctx;
  int32_t batch, seq_len, num_blocks, row_start, num_rows;
  int32_t tiles_per_batch;  // ceilDiv(seq_len, 64)
  int32_t tile_lo;          // first global token tile (b * tiles_per_batch + i) of the chunk
  int32_t n_gtiles;         // ceilDiv(num_blocks, 128)
  int32_t n_groups;         // g-tile groups a token tile is split into (unit_groups)
  int32_t units;
  uint32_t idesc;
  float scale;
  int32_t vec_fill;         // logits rows are 16-byte aligned: fully masked sub-tiles use v4 stores
};

// A work unit is (sequence b, 64-token tile at t0, g-tile group grp).  Group grp owns
// the interleaved g-tiles gt(i) = grp + n_groups * i, so every group of a token tile
// gets an even share of the (causal, prefix-shaped) MMA tiles and the persistent
// CTAs stay balanced.
struct alignas(16) Unit {
  int32_t b, t0, grp;       // b < 0: no more work
  int32_t n_tiles;   // g-tiles of this unit: i in [0, n_tiles)
  int32_t n_mma;     // the first n_mma of them need the MMA; the rest are fully masked
  int32_t t_lo, t_hi;                    // stored rows [t_lo, t_hi)
  int32_t t_vis_hi;                      // rows below this (and >= t_lo) are unpadded
  int64_t row_base;                      // chunk-local row of (b, t = 0)
};

__device__ __forceinline__ Unit unit_info(const Params& p, int32_t u) {
  Unit x;
  const int32_t tq = u / p.n_groups;
  x.grp = u - tq * p.n_groups;
  const int32_t tile = p.tile_lo + tq;
  x.b = tile / p.tiles_per_batch;
  x.t0 = (tile - x.b * p.tiles_per_batch) * kTokTile;
  x.n_tiles = (p.n_gtiles - x.grp + p.n_groups - 1) / p.n_groups;
  const int64_t bs = static_cast<int64_t>(x.b) * p.seq_len;
  const int64_t c_lo = static_cast<int64_t>(p.row_start) - bs;
  const int64_t c_hi = static_cast<int64_t>(p.row_start) + p.num_rows - bs;
  x.t_lo = static_cast<int32_t>(max(static_cast<int64_t>(x.t0), max(c_lo, int64_t{0})));
  x.t_hi = static_cast<int32_t>(min(static_cast<int64_t>(x.t0 + kTokTile),
                                    min(c_hi, static_cast<int64_t>(p.seq_len))));
  const int32_t ctx = max(__ldg(p.ctx + x.b), 0);
  x.t_vis_hi = min(x.t_hi, ctx);
  // The last unpadded row t_vis_hi - 1 sees blocks g < t_vis_hi / 4, so g-tiles
  // gt < lim need the MMA; visibility only shrinks with g, so within the unit they
  // are the prefix i < n_mma.
  x.n_mma = 0;
  if (x.t_vis_hi > x.t_lo) {
    const int32_t lim = (x.t_vis_hi / 4 + kGTile - 1) / kGTile;
    x.n_mma = max(0, min(x.n_tiles, (lim - x.grp + p.n_groups - 1) / p.n_groups));
  }
  x.row_base = bs - p.row_start;
  return x;
}

static_assert(sizeof(Unit) == kUnitBytes, "scheduler ring entry size");

__device__ __forceinline__ int32_t unit_gtile(const Params& p, const Unit& x, int32_t i) {
  return x.grp + p.n_groups * i;
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint32_t fault_code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t start = ptx::global_timer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::global_timer_ns() - start > kWaitLimitNs) {
      atomicOr(&g_fault_flags, fault_code);
      *abort_flag = 1;
      return false;
    }
  }
}

// Used only while draining after an abort: ignores the abort flag, shorter limit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t start = ptx::global_timer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::global_timer_ns() - start > kDrainLimitNs) {
      atomicOr(&g_fault_flags, kFaultDrain);
      return;
    }
  }
}

// Logits are written once and never re-read by this kernel.  Policy 1 marks them
// evict-first in L2 (st.global.cs) so q and kbar tiles stay resident.
#ifndef QSA_K2_STORE_POLICY
#define QSA_K2_STORE_POLICY 1
#endif
__device__ __forceinline__ void st_f32x4_neg_max(float* p) {
  const float v = -FLT_MAX;
#if QSA_K2_STORE_POLICY == 1
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%1,%1,%1};" :: "l"(p), "f"(v) : "memory");
#else
  asm volatile("st.global.v4.f32 [%0], {%1,%1,%1,%1};" :: "l"(p), "f"(v) : "memory");
#endif
}

__device__ __forceinline__ void st_f32(float* p, float v) {
#if QSA_K2_STORE_POLICY == 1
  asm volatile("st.global.cs.f32 [%0], %1;" :: "l"(p), "f"(v) : "memory");
#else
  asm volatile("st.global.f32 [%0], %1;" :: "l"(p), "f"(v) : "memory");
#endif
}

// relu per head, ascending-h sum, scale after the sum ("Qsa Indexer Kernels",
// launchQsaIndexScores): r holds 8 tokens x 4 heads of one block g.
__device__ __forceinline__ float head_sum(const uint32_t (&r)[32], int k) {
  float v = __fadd_rn(fmaxf(0.0f, __uint_as_float(r[4 * k + 0])), fmaxf(0.0f, __uint_as_float(r[4 * k + 1])));
  v = __fadd_rn(v, fmaxf(0.0f, __uint_as_float(r[4 * k + 2])));
  return __fadd_rn(v, fmaxf(0.0f, __uint_as_float(r[4 * k + 3])));
}

// Two rounded binary32 operations per instruction (add.rn.f32x2 / mul.rn.f32x2):
// lane-wise identical to the scalar forms.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t c;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(c) : "l"(a), "l"(b));
  return c;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t c;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(c) : "l"(a), "l"(b));
  return c;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ float relu_bits(uint32_t x) { return fmaxf(0.0f, __uint_as_float(x)); }

// 8 consecutive token rows, all stored and all visible.  Tokens k and k+1 share the
// packed adds: per token the sum is still ((h0 + h1) + h2) + h3, then times scale.
__device__ __forceinline__ void store8_visible(float* out, const uint32_t (&r)[32], int64_t nb, float scale) {
  const uint64_t sc = pack2(scale, scale);
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    uint64_t v = add2(pack2(relu_bits(r[4 * k + 0]), relu_bits(r[4 * k + 4])),
                      pack2(relu_bits(r[4 * k + 1]), relu_bits(r[4 * k + 5])));
    v = add2(v, pack2(relu_bits(r[4 * k + 2]), relu_bits(r[4 * k + 6])));
    v = add2(v, pack2(relu_bits(r[4 * k + 3]), relu_bits(r[4 * k + 7])));
    v = mul2(v, sc);
    float lo, hi;
    unpack2(v, lo, hi);
    st_f32(out + k * nb, lo);
    st_f32(out + (k + 1) * nb, hi);
  }
}

// 8 consecutive token rows from t: store only rows of the chunk, mask per element
__device__ __forceinline__ void store8_checked(float* out, const uint32_t (&r)[32], int64_t nb, float scale,
                                               int32_t t, int32_t g, const Unit& x) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int32_t tk = t + k;
    if (tk >= x.t_lo && tk < x.t_hi) {
      const bool vis = tk < x.t_vis_hi && g < (tk + 1) / 4;
      st_f32(out + k * nb, vis ? __fmul_rn(head_sum(r, k), scale) : -FLT_MAX);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
k2_scores_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ CUtensorMap tmap_k, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + kOffBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base_ptr + kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + kOffAbort);
  Unit* ring = reinterpret_cast<Unit*>(base_ptr + kOffRing);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      ptx::mbar_init(bar(kBarQFull + s), 1);
      ptx::mbar_init(bar(kBarQEmpty + s), 1);
    }
    for (int s = 0; s < kKStages; ++s) {
      ptx::mbar_init(bar(kBarKFull + s), 1);
      ptx::mbar_init(bar(kBarKEmpty + s), 1);
    }
    for (int s = 0; s < kAccStages; ++s) {
      ptx::mbar_init(bar(kBarAccFull + s), 1);
      ptx::mbar_init(bar(kBarAccEmpty + s), kEpiWarps);
    }
    for (int s = 0; s < kSchedStages; ++s) {
      ptx::mbar_init(bar(kBarSchedFull + s), 1);
      ptx::mbar_init(bar(kBarSchedEmpty + s), 1 + kEpiWarps);
    }
    ptx::mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmap_q);
    ptx::prefetch_tensormap(&tmap_k);
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_alloc(base + kOffTmemSlot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The producer takes its first unit and prefetches that unit's q tile and first kbar
  // tiles into L2, so the copies after the wait find them there.  A prefetch reads nothing
  // into this CTA, and L2 keeps later writes of the previous kernel current, so it may run
  // before the wait; it needs no context length.
  uint32_t u_first = 0u;
  if (warp == 0 && lane == 0) {
    u_first = atomicAdd(p.sched, 1u);
    if (u_first < static_cast<uint32_t>(p.units)) {
      const int32_t tq = static_cast<int32_t>(u_first) / p.n_groups;
      const int32_t grp = static_cast<int32_t>(u_first) - tq * p.n_groups;
      const int32_t tile = p.tile_lo + tq;
      const int32_t b = tile / p.tiles_per_batch;
      const int32_t t0 = (tile - b * p.tiles_per_batch) * kTokTile;
      ptx::tma_prefetch_3d(&tmap_q, 0, 4 * t0, b);
      ptx::tma_prefetch_3d(&tmap_q, 64, 4 * t0, b);
      const int32_t n_tiles = (p.n_gtiles - grp + p.n_groups - 1) / p.n_groups;
      for (int i = 0; i < n_tiles && i < kKStages; ++i) {
        const int32_t gt = grp + p.n_groups * i;
        ptx::tma_prefetch_3d(&tmap_k, 0, gt * kGTile, b);
        ptx::tma_prefetch_3d(&tmap_k, 64, gt * kGTile, b);
      }
    }
  }
  // Everything above overlaps the previous kernel's tail when this launch is a
  // programmatic dependent; nothing below may read its inputs (q, kbar, ctx) or
  // overwrite the logits buffer before that kernel has completed.
  ptx::grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // Work units are taken in increasing order (increasing logits address) from a
      // device-wide counter, so the CTAs' write fronts advance together.
      int qcnt = 0, kcnt = 0, scnt = 0;
      bool first = true;
      while (true) {
        const uint32_t u = first ? u_first : atomicAdd(p.sched, 1u);
        first = false;
        Unit x;
        if (u < static_cast<uint32_t>(p.units)) {
          x = unit_info(p, static_cast<int32_t>(u));
        } else {
          x = Unit{};
          x.b = -1;
          // this CTA takes no more work: the next kernel may start launching
          ptx::launch_dependents();
        }
        const int ss = scnt % kSchedStages;
        if (!wait_bounded(bar(kBarSchedEmpty + ss), ((scnt / kSchedStages) & 1) ^ 1, abort_flag, kFaultProducer)) break;
        ring[ss] = x;
        ptx::mbar_arrive(bar(kBarSchedFull + ss));
        ++scnt;
        if (x.b < 0) break;
        if (x.n_mma == 0) continue;
        const int qs = qcnt % kQStages;
        if (!wait_bounded(bar(kBarQEmpty + qs), ((qcnt / kQStages) & 1) ^ 1, abort_flag, kFaultProducer)) break;
        ptx::mbar_arrive_expect_tx(bar(kBarQFull + qs), kQBytes);
        const uint32_t qdst = base + kOffQ + qs * kQBytes;
        ptx::tma_load_3d(qdst, &tmap_q, bar(kBarQFull + qs), 0, 4 * x.t0, x.b);
        ptx::tma_load_3d(qdst + kQHalfBytes, &tmap_q, bar(kBarQFull + qs), 64, 4 * x.t0, x.b);
        ++qcnt;
        bool ok = true;
        for (int i = 0; i < x.n_mma; ++i) {
          const int32_t gt = unit_gtile(p, x, i);
          const int ks = kcnt % kKStages;
          if (!wait_bounded(bar(kBarKEmpty + ks), ((kcnt / kKStages) & 1) ^ 1, abort_flag, kFaultProducer)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(bar(kBarKFull + ks), kKBytes);
          const uint32_t kdst = base + kOffK + ks * kKBytes;
          ptx::tma_load_3d(kdst, &tmap_k, bar(kBarKFull + ks), 0, gt * kGTile, x.b);
          ptx::tma_load_3d(kdst + kKHalfBytes, &tmap_k, bar(kBarKFull + ks), 64, gt * kGTile, x.b);
          ++kcnt;
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // wait for the last copy issued into each stage before the CTA can exit
        for (int s = 0; s < kQStages; ++s) {
          if (qcnt > s) {
            const int n = ((qcnt - 1 - s) / kQStages) * kQStages + s;
            drain_wait(bar(kBarQFull + s), (n / kQStages) & 1);
          }
        }
        for (int s = 0; s < kKStages; ++s) {
          if (kcnt > s) {
            const int n = ((kcnt - 1 - s) / kKStages) * kKStages + s;
            drain_wait(bar(kBarKFull + s), (n / kKStages) & 1);
          }
        }
      }
      // This CTA takes no more units; the last CTA to get here resets the slot.
      __threadfence();
      if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
        atomicExch(p.sched, 0u);
        atomicExch(p.sched + 1, 0u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int qcnt = 0, kcnt = 0, acnt = 0, scnt = 0;
      bool ok = true;
      while (ok) {
        const int ss = scnt % kSchedStages;
        if (!wait_bounded(bar(kBarSchedFull + ss), (scnt / kSchedStages) & 1, abort_flag, kFaultMma)) break;
        const Unit x = ring[ss];
        ptx::mbar_arrive(bar(kBarSchedEmpty + ss));
        ++scnt;
        if (x.b < 0) break;
        if (x.n_mma == 0) continue;
        const int qs = qcnt % kQStages;
        if (!wait_bounded(bar(kBarQFull + qs), (qcnt / kQStages) & 1, abort_flag, kFaultMma)) break;
        ptx::tc_fence_after();
        const uint32_t qaddr = base + kOffQ + qs * kQBytes;
        for (int i = 0; i < x.n_mma; ++i) {
          const int ks = kcnt % kKStages;
          const int as = acnt % kAccStages;
          if (!wait_bounded(bar(kBarKFull + ks), (kcnt / kKStages) & 1, abort_flag, kFaultMma) ||
              !wait_bounded(bar(kBarAccEmpty + as), ((acnt / kAccStages) & 1) ^ 1, abort_flag, kFaultMma)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t kaddr = base + kOffK + ks * kKBytes;
          const uint32_t d = tmem + static_cast<uint32_t>(as) * kAccCols;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = static_cast<uint32_t>(kk & 3) * 32u;
            const uint64_t adesc = ptx::smem_desc_sw128(kaddr + (kk >> 2) * kKHalfBytes + koff);
            const uint64_t bdesc = ptx::smem_desc_sw128(qaddr + (kk >> 2) * kQHalfBytes + koff);
            ptx::mma_f16(d, adesc, bdesc, p.idesc, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(bar(kBarKEmpty + ks));
          ptx::mma_commit(bar(kBarAccFull + as));
          ++kcnt;
          ++acnt;
        }
        if (!ok) break;
        ptx::mma_commit(bar(kBarQEmpty + qs));
        ++qcnt;
      }
      // every MMA (and the arrivals committed after it) completes before TMEM is freed
      ptx::mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  } else {
    // --------------------------------------------------------------- epilogue
    // Warp ew reads TMEM sub-partition sp = warp % 4 (blocks g0 + 32*sp + lane) for
    // the token slice [kTokPerWarp*grp, +kTokPerWarp) of the tile.  The common case, a
    // warp sub-tile entirely inside the chunk, the sequence's valid rows and the
    // visible triangle, takes a predicate-free path; edges take the checked path.
    const int ew = warp - 2;
    const int sp = warp & 3;
    const int grp = ew >> 2;
    const int64_t nb = p.num_blocks;
    const float scale = p.scale;
    int acnt = 0, scnt = 0;
    bool ok = true;
    while (ok) {
      const int ss = scnt % kSchedStages;
      if (!wait_bounded(bar(kBarSchedFull + ss), (scnt / kSchedStages) & 1, abort_flag, kFaultEpilogue)) break;
      const Unit x = ring[ss];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarSchedEmpty + ss));
      ++scnt;
      if (x.b < 0) break;
      const int32_t tb = x.t0 + kTokPerWarp * grp;  // first token of this warp's slice
      const bool rows_full = x.t_lo <= tb && tb + kTokPerWarp <= x.t_hi;
      for (int i = 0; i < x.n_tiles; ++i) {
        const int32_t gw = unit_gtile(p, x, i) * kGTile + 32 * sp;    // first block of this warp
        const int32_t g = gw + lane;
        const bool g_ok = g < p.num_blocks;
        const bool cols_full = gw + 32 <= p.num_blocks;
        float* out = p.logits + (x.row_base + tb) * nb + g;  // row of token tb
        if (i < x.n_mma) {
          const int as = acnt % kAccStages;
          if (!wait_bounded(bar(kBarAccFull + as), (acnt / kAccStages) & 1, abort_flag, kFaultEpilogue)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          // every (t, g) of the sub-tile visible: g <= gw+31 < (tb+1)/4 <= (t+1)/4, t < ctx
          const bool interior = rows_full && cols_full && tb + kTokPerWarp <= x.t_vis_hi &&
                                gw + 31 < (tb + 1) / 4;
          const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * sp) << 16) +
                                 static_cast<uint32_t>(as) * kAccCols + 4u * kTokPerWarp * grp;
          // 8 tokens per 32-column load; the next load is in flight while the
          // current 8 tokens are reduced and stored
          auto emit = [&](const uint32_t (&r)[32], int c) {
            if (interior) {
              store8_visible(out + 8 * c * nb, r, nb, scale);
            } else if (g_ok) {
              store8_checked(out + 8 * c * nb, r, nb, scale, tb + 8 * c, g, x);
            }
          };
          uint32_t ra[32], rb[32];
          ptx::tmem_ld_32x32b_x32(taddr, ra);
          ptx::tmem_ld_wait(ra);
#pragma unroll
          for (int c = 0; c < kLdPerWarp; c += 2) {
            ptx::tmem_ld_32x32b_x32(taddr + 32u * (c + 1), rb);
            emit(ra, c);
            ptx::tmem_ld_wait(rb);
            if (c + 2 < kLdPerWarp) ptx::tmem_ld_32x32b_x32(taddr + 32u * (c + 2), ra);
            emit(rb, c + 1);
            if (c + 2 < kLdPerWarp) ptx::tmem_ld_wait(ra);
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(kBarAccEmpty + as));
          ++acnt;
        } else if (rows_full && cols_full && p.vec_fill) {
          // lanes re-mapped for the fill: 4 rows x 128 bytes per store instruction
          float* o = out - lane + (lane >> 3) * nb + 4 * (lane & 7);
#pragma unroll
          for (int k = 0; k < kTokPerWarp; k += 4) st_f32x4_neg_max(o + k * nb);
        } else if (rows_full && cols_full) {
#pragma unroll 8
          for (int k = 0; k < kTokPerWarp; ++k) {
            st_f32(out, -FLT_MAX);
            out += nb;
          }
        } else if (g_ok) {
#pragma unroll 4
          for (int k = 0; k < kTokPerWarp; ++k) {
            const int32_t t = tb + k;
            if (t >= x.t_lo && t < x.t_hi) st_f32(out, -FLT_MAX);
            out += nb;
          }
        }
      }
    }
  }

  ptx::launch_dependents();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace k2

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn(cudaError_t* err) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                              cudaEnableDefault, &q);
    if (status == cudaSuccess && q != cudaDriverEntryPointSuccess) status = cudaErrorNotSupported;
    if (status == cudaSuccess) fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  *err = status;
  return fn;
}

// 3-D map over [dim2][dim1][128] two-byte elements, box {64, box1, 1}, 128-byte swizzle.
cudaError_t encode_rows(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map,
                        const void* ptr, uint64_t dim1, uint64_t dim2, uint32_t box1) {
  cuuint64_t dims[3] = {128, dim1, dim2};
  cuuint64_t strides[2] = {256, dim1 * 256};
  cuuint32_t box[3] = {64, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(ptr), dims, strides,
                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

std::mutex g_attr_mu;
bool g_attr_set[64] = {};
uint32_t* g_sched_base[64] = {};      // device address of g_k2_sched, per device
uint32_t g_launch_seq[64] = {};       // launches so far, per device (guarded by g_attr_mu)

}  // namespace

// Groups a token tile's g-tiles are split into, one work unit each (every n_groups-th
// g-tile).  kGTilesPerUnit g-tiles a unit by default; half as many when a launch would
// give each CTA fewer than kMinUnitsPerCta units, as row-chunked calls do: the last
// units of a launch run while other SMs idle, and smaller units shorten that tail
// (16 chunks of 8192 rows at B=8, S=16384: 0.495 -> 0.469 ms; one launch over every row
// keeps the larger units, 0.350 against 0.358 ms).  The logits do not depend on it.
constexpr int kMinUnitsPerCta = 16;
static int32_t unit_groups(int64_t tiles, int32_t n_gtiles, int num_sms) {
  using k2::kGTilesPerUnit;
  const int32_t full = (n_gtiles + kGTilesPerUnit - 1) / kGTilesPerUnit;
  if (kGTilesPerUnit < 2 || tiles * full >= static_cast<int64_t>(kMinUnitsPerCta) * num_sms) return full;
  constexpr int32_t half = kGTilesPerUnit / 2;
  return (n_gtiles + half - 1) / half;
}

cudaError_t launch_scores_tc(const LaunchScores& a) {
  using namespace k2;
  cudaError_t e;
  auto encode = get_encode_fn(&e);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  uint32_t slot = 0;
  uint32_t* sched_base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_attr_set[dev]) {
      e = cudaFuncSetAttribute(k2_scores_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBytes));
      if (e != cudaSuccess) return e;
      // the symbol's name is only a host-side stand-in: ask the runtime for the
      // device address, once per device, with that device current
      void* sched = nullptr;
      if ((e = cudaGetSymbolAddress(&sched, g_k2_sched)) != cudaSuccess) return e;
      g_sched_base[dev] = static_cast<uint32_t*>(sched);
      g_attr_set[dev] = true;
    }
    slot = g_launch_seq[dev]++ % kSchedSlots;
    sched_base = g_sched_base[dev];
  }
  CUtensorMap tq, tk;
  if ((e = encode_rows(encode, &tq, a.q_normed, 4ull * a.seq_len, a.batch, kN)) != cudaSuccess) return e;
  if ((e = encode_rows(encode, &tk, a.kbar, a.num_blocks, a.batch, kGTile)) != cudaSuccess) return e;

  Params p{};
  p.sched = sched_base + 2 * slot;
  p.logits = a.logits;
  p.ctx = a.context_lengths;
  p.batch = a.batch;
  p.seq_len = a.seq_len;
  p.num_blocks = a.num_blocks;
  p.row_start = a.row_start;
  p.num_rows = a.num_rows;
  p.tiles_per_batch = (a.seq_len + kTokTile - 1) / kTokTile;
  const int64_t first = a.row_start;
  const int64_t last = static_cast<int64_t>(a.row_start) + a.num_rows - 1;
  const int64_t b_first = first / a.seq_len, b_last = last / a.seq_len;
  const int64_t tile_lo = b_first * p.tiles_per_batch + (first - b_first * a.seq_len) / kTokTile;
  const int64_t tile_hi = b_last * p.tiles_per_batch + (last - b_last * a.seq_len) / kTokTile + 1;
  p.tile_lo = static_cast<int32_t>(tile_lo);
  p.n_gtiles = (a.num_blocks + kGTile - 1) / kGTile;
  p.n_groups = unit_groups(tile_hi - tile_lo, p.n_gtiles, a.num_sms);
  const int64_t units = (tile_hi - tile_lo) * p.n_groups;
  if (units > INT32_MAX) return cudaErrorInvalidValue;
  p.units = static_cast<int32_t>(units);
  p.idesc = ptx::idesc_f16(a.bf16, kGTile, kN);
  p.scale = a.scale;
  p.vec_fill = (a.num_blocks % 4 == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0) ? 1 : 0;
  const int grid = static_cast<int>(units < a.num_sms ? units : a.num_sms);
  // A programmatic dependent of the previous kernel in the stream: this launch's CTAs
  // may become resident, and set up, while that kernel drains; they wait for it to
  // complete before touching any input or output (griddepcontrol.wait above).
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k2_scores_tc_kernel, tq, tk, p);
}

// ---------------------------------------------------------------------------
// No-allocation variant (qsa_index_scores_no_alloc).  Same kernel and numerics as
// launch_scores_tc; the only difference is where the kernel's scratch lives: one
// fixed 256-byte static array shared by every call on a device, instead of the
// rotating per-launch slot table.  Its first two words are the scheduler's
// {next unit, CTAs finished} counter pair; each call zeroes them on its stream
// before the kernel runs, so calls that overlap on the GPU race on them.
constexpr int kNoAllocScratchWords = 64;  // 256 bytes
// The header states the no-alloc limit with 1024 blocks per work unit's g-tile group.
static_assert(k2::kGTile * k2::kGTilesPerUnit == 1024,
              "qsa_index_scores_no_alloc's documented work-unit count assumes 1024 blocks a group");
static __device__ __align__(256) uint32_t g_k2_noalloc_scratch[kNoAllocScratchWords];

namespace {
std::mutex g_noalloc_mu;
bool g_noalloc_ready[64] = {};
uint32_t* g_noalloc_ptr[64] = {};
}  // namespace

// Largest number of work units the 32-bit counter can hand out: every CTA
// overshoots it by one when the work runs out, so keep a CTA-count margin.
int64_t scores_no_alloc_max_units() { return static_cast<int64_t>(INT32_MAX) - 65536; }

int64_t scores_work_units(int32_t batch, int32_t seq_len, int32_t num_blocks, int32_t row_start,
                          int32_t num_rows) {
  using namespace k2;
  const int64_t tpb = (seq_len + kTokTile - 1) / kTokTile;
  const int64_t first = row_start;
  const int64_t last = static_cast<int64_t>(row_start) + num_rows - 1;
  const int64_t b_first = first / seq_len, b_last = last / seq_len;
  const int64_t tile_lo = b_first * tpb + (first - b_first * seq_len) / kTokTile;
  const int64_t tile_hi = b_last * tpb + (last - b_last * seq_len) / kTokTile + 1;
  const int64_t n_gtiles = (num_blocks + kGTile - 1) / kGTile;
  (void)batch;
  return (tile_hi - tile_lo) * ((n_gtiles + kGTilesPerUnit - 1) / kGTilesPerUnit);
}

cudaError_t launch_scores_tc_no_alloc(const LaunchScores& a) {
  using namespace k2;
  cudaError_t e;
  auto encode = get_encode_fn(&e);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  uint32_t* scratch = nullptr;
  {
    // one-time set-up per device, with that device current: kernel attribute and the
    // device address of the static scratch array (its name is a host-side stand-in)
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_noalloc_ready[dev]) {
      e = cudaFuncSetAttribute(k2_scores_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBytes));
      if (e != cudaSuccess) return e;
      void* ptr = nullptr;
      if ((e = cudaGetSymbolAddress(&ptr, g_k2_noalloc_scratch)) != cudaSuccess) return e;
      g_noalloc_ptr[dev] = static_cast<uint32_t*>(ptr);
      g_noalloc_ready[dev] = true;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // the counter pair must start at zero: clear it in stream order (no allocation)
  if ((e = cudaMemsetAsync(scratch, 0, 2 * sizeof(uint32_t), a.stream)) != cudaSuccess) return e;

  CUtensorMap tq, tk;
  if ((e = encode_rows(encode, &tq, a.q_normed, 4ull * a.seq_len, a.batch, kN)) != cudaSuccess) return e;
  if ((e = encode_rows(encode, &tk, a.kbar, a.num_blocks, a.batch, kGTile)) != cudaSuccess) return e;
  Params p{};
  p.sched = scratch;
  p.logits = a.logits;
  p.ctx = a.context_lengths;
  p.batch = a.batch;
  p.seq_len = a.seq_len;
  p.num_blocks = a.num_blocks;
  p.row_start = a.row_start;
  p.num_rows = a.num_rows;
  p.tiles_per_batch = (a.seq_len + kTokTile - 1) / kTokTile;
  const int64_t first = a.row_start;
  const int64_t b_first = first / a.seq_len;
  p.tile_lo = static_cast<int32_t>(b_first * p.tiles_per_batch + (first - b_first * a.seq_len) / kTokTile);
  p.n_gtiles = (a.num_blocks + kGTile - 1) / kGTile;
  p.n_groups = (p.n_gtiles + kGTilesPerUnit - 1) / kGTilesPerUnit;
  const int64_t units = scores_work_units(a.batch, a.seq_len, a.num_blocks, a.row_start, a.num_rows);
  if (units > scores_no_alloc_max_units()) return cudaErrorInvalidValue;
  p.units = static_cast<int32_t>(units);
  p.idesc = ptx::idesc_f16(a.bf16, kGTile, kN);
  p.scale = a.scale;
  p.vec_fill = (a.num_blocks % 4 == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0) ? 1 : 0;
  const int grid = static_cast<int>(units < a.num_sms ? units : a.num_sms);
  k2_scores_tc_kernel<<<grid, kThreads, kSmemBytes, a.stream>>>(tq, tk, p);
  return cudaGetLastError();
}

cudaError_t read_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_fault_flags, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  if (clear && *flags != 0u) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_fault_flags, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
  }
  return e;
}

}  // namespace qsa
