// Prefill block scoring fused with the top-512 selection and expand
// ("Qsa Indexer Kernels": launchQsaIndexScores, then the selection between
// launchQsaIndexIdsFill and launchQsaIndexExpand), without writing the FP32 logits.
//
// The logits are those of K2 (the same tcgen05 tile: A = 128 kbar blocks, B = 64
// tokens x 4 heads, K = 128 in eight K = 16 steps, FP32 in TMEM, and the same
// epilogue arithmetic: relu per head, ascending-h sum, scale after the sum), so
// every logit is bit-identical to qsa_index_scores'.  The selected set is the one of
// qsa_index_topk_expand: on the order-preserving u32 keys of a row's visible logits,
// the 512 largest, keys equal to the 512th taken in ascending block order, emitted in
// ascending block order and expanded to 2051 token ids.
//
// A work unit is one 64-token tile of one sequence with every g-tile of 128 blocks.
// A CTA computes the unit's logits at least twice on the tensor cores and keeps
// per-row state in shared memory instead of the logits:
//   histogram pass  every visible key of a row selected by the pass is counted in a
//                   256-bin histogram of the row; one warp a row then finds the bin
//                   holding the row's 512th key.  The first pass bins keys on a
//                   log scale (64 bins an octave from a per-CTA base, +0 in a bin of
//                   its own, the ends clamped); later passes split the bin found into
//                   256 equal key ranges.
//   final pass      once every row's threshold bin is narrow (its keys fit a short
//                   list, all equal, or all taken), each key is classified: above the
//                   bin (a bit in the row's selected mask), inside it (listed with its
//                   block id, or a bit in a tie mask when the bin is one key), or below.
//   emission        one warp a row picks the bin's winners (largest keys first, equal
//                   keys by ascending block id), merges them into the selected mask,
//                   and writes the row's 2051 token ids.
// Typical rows need one histogram pass and the final pass; every extra pass narrows
// the bin by 8 bits, so no row needs more than five.  The bin base only decides how
// many passes a row needs, never which blocks are selected.
//
// Roles (one persistent CTA per SM, units taken from a device-wide counter, heaviest
// tiles first): warp 0 scheduler + TMA producer, warp 1 TMEM allocator + MMA issuer,
// warps 2..17 the epilogue (four per TMEM sub-partition, 16 tokens each).  Producer and
// MMA issuer learn after each histogram pass whether another one follows from a
// decision ring the epilogue fills.  Every mbarrier wait is bounded; a wait that runs
// out sets a fault bit, the CTA drains its own copies and MMAs, frees TMEM and exits.
#include <cfloat>
#include <mutex>

#include <cudaTypedefs.h>

#include "qsa_bins.cuh"
#include "qsa_launch.h"
#include "qsa_select.cuh"
#include "tc_ptx.cuh"

namespace qsa {

// Bits set by this kernel's bounded waits that ran out (read by read_fused_fault_flags).
__device__ uint32_t g_k2s_fault_flags;

// Scheduler counter pairs {next unit, CTAs finished}, one taken in turn per launch
// (up to kSchedSlots launches in flight per device); zero at module load, reset by
// the last CTA of each launch.
constexpr int kFusedSchedSlots = 64;
__device__ __align__(256) uint32_t g_k2s_sched[kFusedSchedSlots * 2];

namespace k2s {

constexpr int kTokTile = 64;
constexpr int kN = kTokTile * 4;
constexpr int kGTile = 128;
constexpr int kMaxBlocks = 4096;              // NB limit: a row's masks are 128 words
constexpr int kWords = kMaxBlocks / 32;
constexpr int kCap = 128;                      // candidates listed per row
constexpr int kKStages = 2;
constexpr int kAccStages = 2;
#ifndef QSA_FUSED_EPI_WARPS
#define QSA_FUSED_EPI_WARPS 16
#endif
constexpr int kEpiWarps = QSA_FUSED_EPI_WARPS;     // 8 or 16: two or four per TMEM sub-partition
static_assert(kEpiWarps == 8 || kEpiWarps == 16, "epilogue warps");
constexpr int kTokPerWarp = kTokTile / (kEpiWarps / 4);  // tokens of a tile per epilogue warp
constexpr int kLdPerWarp = kTokPerWarp / 8;              // 32-column TMEM loads (8 tokens each)
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kQHalfBytes = kN * 64 * 2;
constexpr uint32_t kQBytes = 2 * kQHalfBytes;
constexpr uint32_t kKHalfBytes = kGTile * 64 * 2;
constexpr uint32_t kKBytes = 2 * kKHalfBytes;
constexpr int kSchedStages = 4;
constexpr int kDecStages = 2;

// row modes
enum : uint32_t {
  kSkip = 0,     // not a row of this call
  kShort = 1,    // padded, or at most 512 visible blocks: no logits needed
  kActive = 2,   // threshold bin still to be narrowed by a histogram pass
  kTakeAll = 3,  // every key >= lo is selected
  kCand = 4,     // keys > hi selected; keys in [lo, hi] listed, rem of them win
  kTies = 5,     // lo == hi: keys > hi selected; the first rem keys equal to lo win
};

struct RowState {
  uint32_t lo, hi;   // key range that holds the row's 512th key
  int32_t rem;       // keys still to take inside [lo, hi]
  uint32_t cnt;      // candidates listed by the final pass
  uint32_t mode;
  uint32_t shift;    // refinement passes: bin = (key - lo) >> shift
  uint32_t level0;   // next histogram pass is the first (log-scale bins)
  int32_t n_vis;
};
static_assert(sizeof(RowState) == 32, "row state size");

// shared memory layout (offsets from the 1024-aligned base)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffA = kOffK + kKStages * kKBytes;          // per row: histogram, then selected mask
constexpr uint32_t kOffB = kOffA + kTokTile * kWords * 4;        // per row: candidates or tie mask
constexpr uint32_t kOffStage = kOffB + kTokTile * kWords * 4;    // per epilogue warp: 512 winners (u16)
constexpr uint32_t kOffRows = kOffStage + kEpiWarps * sel::kTopK * 2;
constexpr uint32_t kOffThr = kOffRows + kTokTile * sizeof(RowState);  // per epilogue warp: its tokens'
                                                                      // final-pass (sel_gt, in_lo) pairs
constexpr uint32_t kOffBar = kOffThr + kEpiWarps * kTokPerWarp * 8;
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 1;
constexpr int kBarKFull = 2;
constexpr int kBarKEmpty = kBarKFull + kKStages;
constexpr int kBarAccFull = kBarKEmpty + kKStages;
constexpr int kBarAccEmpty = kBarAccFull + kAccStages;
constexpr int kBarSchedFull = kBarAccEmpty + kAccStages;
constexpr int kBarSchedEmpty = kBarSchedFull + kSchedStages;
constexpr int kBarDecFull = kBarSchedEmpty + kSchedStages;
constexpr int kBarDecEmpty = kBarDecFull + kDecStages;
constexpr int kBarDrain = kBarDecEmpty + kDecStages;
constexpr int kNumBars = kBarDrain + 1;
constexpr uint32_t kUnitBytes = 32;
constexpr uint32_t kOffRing = (kOffBar + kNumBars * 8 + 15u) & ~15u;
constexpr uint32_t kOffDec = kOffRing + kSchedStages * kUnitBytes;
constexpr uint32_t kOffMisc = kOffDec + kDecStages * 4;   // tmem slot, abort, active, final, base, base sums
constexpr uint32_t kMiscWords = 8;
constexpr uint32_t kSmemBytes = kOffMisc + kMiscWords * 4 + 1024;
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
static_assert(kOffK % 1024 == 0 && kOffA % 16 == 0 && kOffBar % 8 == 0 && kOffRing % 16 == 0,
              "shared-memory regions misaligned");
static_assert(kCap <= kWords, "candidates share a row's 128-word region");

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
enum : uint32_t {
  kFaultProducer = 1u,
  kFaultMma = 2u,
  kFaultEpilogue = 4u,
  kFaultDrain = 8u,
};

constexpr int kBaseMin = bins::kBaseMin;
constexpr int kBaseMax = bins::kBaseMax;

struct Params {
  uint32_t* sched;
  int32_t* out_idx;          // [batch * seq_len, 2051], global rows
  const int32_t* ctx;
  int32_t batch, seq_len, num_blocks, row_start, num_rows;
  int32_t tiles_per_batch, tile_lo, units;
  uint32_t idesc;
  float scale;
  int32_t base0;             // first-pass bin base before any unit has adapted it
};

struct alignas(16) Unit {
  int32_t b, t0;            // b < 0: no more work
  int32_t t_lo, t_hi;       // stored rows [t_lo, t_hi)
  int32_t t_vis_hi;         // rows below this are unpadded
  int32_t n_gt;             // g-tiles the MMA covers (0: no row needs logits)
  int64_t row_base;         // global row of (b, t = 0)
};
static_assert(sizeof(Unit) == kUnitBytes, "scheduler ring entry size");

__device__ __forceinline__ Unit unit_info(const Params& p, int32_t u) {
  Unit x;
  const int32_t tile = p.tile_lo + (p.units - 1 - u);   // heaviest (latest) tiles first
  x.b = tile / p.tiles_per_batch;
  x.t0 = (tile - x.b * p.tiles_per_batch) * kTokTile;
  const int64_t bs = static_cast<int64_t>(x.b) * p.seq_len;
  const int64_t c_lo = static_cast<int64_t>(p.row_start) - bs;
  const int64_t c_hi = static_cast<int64_t>(p.row_start) + p.num_rows - bs;
  x.t_lo = static_cast<int32_t>(max(static_cast<int64_t>(x.t0), max(c_lo, int64_t{0})));
  x.t_hi = static_cast<int32_t>(min(static_cast<int64_t>(x.t0 + kTokTile), min(c_hi, static_cast<int64_t>(p.seq_len))));
  const int32_t ctx = max(__ldg(p.ctx + x.b), 0);
  x.t_vis_hi = min(x.t_hi, ctx);
  // the last unpadded stored row t_vis_hi - 1 sees t_vis_hi / 4 blocks
  const int32_t nv_max = x.t_vis_hi > x.t_lo ? min(x.t_vis_hi / 4, p.num_blocks) : 0;
  x.n_gt = nv_max > sel::kTopK ? (nv_max + kGTile - 1) / kGTile : 0;
  x.row_base = bs;
  return x;
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint32_t fault_code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t start = ptx::global_timer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::global_timer_ns() - start > kWaitLimitNs) {
      atomicOr(&g_k2s_fault_flags, fault_code);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t start = ptx::global_timer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::global_timer_ns() - start > kDrainLimitNs) {
      atomicOr(&g_k2s_fault_flags, kFaultDrain);
      return;
    }
  }
}

// The epilogue warps' own barrier (named barrier 1; warps 0 and 1 never take part).
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" :: "n"(kEpiThreads) : "memory");
}

// Two rounded binary32 operations per instruction (add.rn.f32x2, mul.rn.f32x2):
// lane-wise identical to the scalar forms, as in K2's epilogue.
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

// Keys of tokens k and k+1 of an 8-token TMEM load r (4 heads a token): per token
// ((h0 + h1) + h2) + h3 of the relus, then times scale, two tokens per instruction.
// The operations and their order are K2's, so every logit has K2's bits.
__device__ __forceinline__ void keys2(const uint32_t (&r)[32], int k, uint64_t sc, uint32_t& k0, uint32_t& k1) {
  uint64_t v = add2(pack2(relu_bits(r[4 * k + 0]), relu_bits(r[4 * k + 4])),
                    pack2(relu_bits(r[4 * k + 1]), relu_bits(r[4 * k + 5])));
  v = add2(v, pack2(relu_bits(r[4 * k + 2]), relu_bits(r[4 * k + 6])));
  v = add2(v, pack2(relu_bits(r[4 * k + 3]), relu_bits(r[4 * k + 7])));
  v = mul2(v, sc);
  float a, b;
  unpack2(v, a, b);
  k0 = sel::orderable(a);
  k1 = sel::orderable(b);
}

__device__ __forceinline__ uint32_t bin0_of(uint32_t key, int32_t base) { return bins::bin_of(key, base); }
__device__ __forceinline__ void bin0_range(uint32_t b, int32_t base, uint32_t& lo, uint32_t& hi) {
  bins::bin_range(b, base, lo, hi);
}

__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += x;
  }
  return v;
}

__device__ __forceinline__ void st_s32x4(int32_t* p, int32_t a, int32_t b, int32_t c, int32_t d) {
  asm volatile("st.global.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// A row's 2051 ids from its 512 winners (ascending): id 4p + j = 4*win[p] + j, then the
// causal tail, then -1; 16-byte stores from the row's first aligned address.
__device__ __forceinline__ void warp_write_selected(int32_t* out, const uint16_t* win, int32_t tail,
                                                    int32_t n_vis, int lane) {
  constexpr int kIds = sel::kRatio * sel::kTopK;
  const int k0 = static_cast<int>((4u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(out) >> 2) & 3u)) & 3u);
  const int nchunks = (kIds - k0) / 4;
  for (int c = lane; c < nchunks; c += 32) {
    const int i = k0 + 4 * c;
    // ids i .. i+3 come from winners i/4 and (i+3)/4 (the same one when the row is aligned)
    const int32_t wa = static_cast<int32_t>(win[i >> 2]) * sel::kRatio;
    const int32_t wb = static_cast<int32_t>(win[(i + 3) >> 2]) * sel::kRatio;
    int32_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = (((i + j) >> 2) == (i >> 2) ? wa : wb) + ((i + j) & 3);
    st_s32x4(out + i, v[0], v[1], v[2], v[3]);
  }
  const int tail_lo = k0 + 4 * nchunks;
  if (lane < k0) out[lane] = static_cast<int32_t>(win[lane >> 2]) * sel::kRatio + (lane & 3);
  if (lane >= k0 && lane < k0 + (kIds - tail_lo)) {
    const int i = tail_lo + (lane - k0);
    out[i] = static_cast<int32_t>(win[i >> 2]) * sel::kRatio + (i & 3);
  }
  if (lane < sel::kRatio - 1) out[kIds + lane] = lane < tail ? sel::kRatio * n_vis + lane : -1;
}

// A row that needs no logits: token ids 0 .. n_all-1, then -1 (n_all = 0 when padded).
__device__ __forceinline__ void warp_write_unselected(int32_t* out, int32_t n_all, int lane) {
  const int k0 = static_cast<int>((4u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(out) >> 2) & 3u)) & 3u);
  const int nchunks = (sel::kWidth - k0) / 4;
  for (int c = lane; c < nchunks; c += 32) {
    const int i = k0 + 4 * c;
    st_s32x4(out + i, i < n_all ? i : -1, i + 1 < n_all ? i + 1 : -1, i + 2 < n_all ? i + 2 : -1,
             i + 3 < n_all ? i + 3 : -1);
  }
  const int rest_lo = k0 + 4 * nchunks;
  if (lane < k0) out[lane] = lane < n_all ? lane : -1;
  if (lane >= k0 && lane < k0 + (sel::kWidth - rest_lo)) {
    const int i = rest_lo + (lane - k0);
    out[i] = i < n_all ? i : -1;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
k2_topk_fused_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + kOffBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  Unit* ring = reinterpret_cast<Unit*>(base_ptr + kOffRing);
  volatile uint32_t* dec = reinterpret_cast<volatile uint32_t*>(base_ptr + kOffDec);
  uint32_t* misc = reinterpret_cast<uint32_t*>(base_ptr + kOffMisc);
  volatile uint32_t* tmem_slot = misc + 0;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  uint32_t* n_active = misc + 2;         // rows still active after a search
  volatile uint32_t* final_next = misc + 3;
  int32_t* bin_base = reinterpret_cast<int32_t*>(misc + 4);
  uint32_t* base_sum = misc + 5;         // first-pass thresholds' key >> 17, summed
  uint32_t* base_n = misc + 6;
  uint32_t* reg_a = reinterpret_cast<uint32_t*>(base_ptr + kOffA);
  uint32_t* reg_b = reinterpret_cast<uint32_t*>(base_ptr + kOffB);
  RowState* rows = reinterpret_cast<RowState*>(base_ptr + kOffRows);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(kBarQFull), 1);
    ptx::mbar_init(bar(kBarQEmpty), 1);
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
    for (int s = 0; s < kDecStages; ++s) {
      ptx::mbar_init(bar(kBarDecFull + s), 1);
      ptx::mbar_init(bar(kBarDecEmpty + s), 2);
    }
    ptx::mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    *n_active = 0;
    *final_next = 0;
    *bin_base = p.base0;
    *base_sum = 0;
    *base_n = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmap_q);
    ptx::prefetch_tensormap(&tmap_k);
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_alloc(base + kOffMisc, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int qcnt = 0, kcnt = 0, scnt = 0, dcnt = 0;
      bool ok = true;
      while (ok) {
        const uint32_t u = atomicAdd(p.sched, 1u);
        Unit x;
        if (u < static_cast<uint32_t>(p.units)) {
          x = unit_info(p, static_cast<int32_t>(u));
        } else {
          x = Unit{};
          x.b = -1;
        }
        const int ss = scnt % kSchedStages;
        if (!wait_bounded(bar(kBarSchedEmpty + ss), ((scnt / kSchedStages) & 1) ^ 1, abort_flag, kFaultProducer)) break;
        ring[ss] = x;
        ptx::mbar_arrive(bar(kBarSchedFull + ss));
        ++scnt;
        if (x.b < 0) break;
        if (x.n_gt == 0) continue;
        if (!wait_bounded(bar(kBarQEmpty), (qcnt & 1) ^ 1, abort_flag, kFaultProducer)) break;
        ptx::mbar_arrive_expect_tx(bar(kBarQFull), kQBytes);
        ptx::tma_load_3d(base + kOffQ, &tmap_q, bar(kBarQFull), 0, 4 * x.t0, x.b);
        ptx::tma_load_3d(base + kOffQ + kQHalfBytes, &tmap_q, bar(kBarQFull), 64, 4 * x.t0, x.b);
        ++qcnt;
        for (int pass = 0; ok; ++pass) {
          for (int i = 0; i < x.n_gt; ++i) {
            const int ks = kcnt % kKStages;
            if (!wait_bounded(bar(kBarKEmpty + ks), ((kcnt / kKStages) & 1) ^ 1, abort_flag, kFaultProducer)) {
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx(bar(kBarKFull + ks), kKBytes);
            const uint32_t kdst = base + kOffK + ks * kKBytes;
            ptx::tma_load_3d(kdst, &tmap_k, bar(kBarKFull + ks), 0, i * kGTile, x.b);
            ptx::tma_load_3d(kdst + kKHalfBytes, &tmap_k, bar(kBarKFull + ks), 64, i * kGTile, x.b);
            ++kcnt;
          }
          if (!ok || pass == 0) continue;
          // after pass >= 1: was it the final pass?
          const int ds = dcnt % kDecStages;
          if (!wait_bounded(bar(kBarDecFull + ds), (dcnt / kDecStages) & 1, abort_flag, kFaultProducer)) {
            ok = false;
            break;
          }
          const uint32_t fin = dec[ds];
          ptx::mbar_arrive(bar(kBarDecEmpty + ds));
          ++dcnt;
          if (fin) break;
        }
      }
      if (*abort_flag) {
        if (qcnt > 0) drain_wait(bar(kBarQFull), (qcnt - 1) & 1);
        for (int s = 0; s < kKStages; ++s) {
          if (kcnt > s) {
            const int n = ((kcnt - 1 - s) / kKStages) * kKStages + s;
            drain_wait(bar(kBarKFull + s), (n / kKStages) & 1);
          }
        }
      }
      __threadfence();
      if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
        atomicExch(p.sched, 0u);
        atomicExch(p.sched + 1, 0u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int qcnt = 0, kcnt = 0, acnt = 0, scnt = 0, dcnt = 0;
      bool ok = true;
      while (ok) {
        const int ss = scnt % kSchedStages;
        if (!wait_bounded(bar(kBarSchedFull + ss), (scnt / kSchedStages) & 1, abort_flag, kFaultMma)) break;
        const Unit x = ring[ss];
        ptx::mbar_arrive(bar(kBarSchedEmpty + ss));
        ++scnt;
        if (x.b < 0) break;
        if (x.n_gt == 0) continue;
        if (!wait_bounded(bar(kBarQFull), qcnt & 1, abort_flag, kFaultMma)) break;
        ptx::tc_fence_after();
        const uint32_t qaddr = base + kOffQ;
        for (int pass = 0; ok; ++pass) {
          for (int i = 0; i < x.n_gt; ++i) {
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
          if (!ok || pass == 0) continue;
          const int ds = dcnt % kDecStages;
          if (!wait_bounded(bar(kBarDecFull + ds), (dcnt / kDecStages) & 1, abort_flag, kFaultMma)) {
            ok = false;
            break;
          }
          const uint32_t fin = dec[ds];
          ptx::mbar_arrive(bar(kBarDecEmpty + ds));
          ++dcnt;
          if (fin) break;
        }
        if (!ok) break;
        ptx::mma_commit(bar(kBarQEmpty));
        ++qcnt;
      }
      ptx::mma_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0);
    }
  } else {
    // --------------------------------------------------------------- epilogue
    const int ew = warp - 2;                      // 0 .. kEpiWarps-1
    const int sp = warp & 3;                      // TMEM sub-partition: blocks 32*sp + lane of a g-tile
    const int tok0 = kTokPerWarp * (ew >> 2);     // this warp's tokens [tok0, tok0 + kTokPerWarp) of the tile
    const int etid = threadIdx.x - 64;
    const uint64_t sc2 = pack2(p.scale, p.scale);
    uint16_t* stage = reinterpret_cast<uint16_t*>(base_ptr + kOffStage) + ew * sel::kTopK;
    uint2* thr_w = reinterpret_cast<uint2*>(base_ptr + kOffThr) + ew * kTokPerWarp;
    int acnt = 0, scnt = 0, dcnt = 0;
    bool ok = true;
    while (ok) {
      const int ss = scnt % kSchedStages;
      if (!wait_bounded(bar(kBarSchedFull + ss), (scnt / kSchedStages) & 1, abort_flag, kFaultEpilogue)) break;
      const Unit x = ring[ss];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarSchedEmpty + ss));
      ++scnt;
      if (x.b < 0) break;

      // ---- row states of this unit; first-pass histograms cleared
      if (etid < kTokTile) {
        const int32_t t = x.t0 + etid;
        RowState rs{};
        rs.lo = 0u;
        rs.hi = 0xFFFFFFFFu;
        rs.rem = sel::kTopK;
        rs.level0 = 1u;
        if (t < x.t_lo || t >= x.t_hi) {
          rs.mode = kSkip;
        } else {
          rs.n_vis = t < x.t_vis_hi ? min((t + 1) / sel::kRatio, p.num_blocks) : 0;
          rs.mode = rs.n_vis > sel::kTopK ? kActive : kShort;
        }
        rows[etid] = rs;
      }
      if (x.n_gt > 0) {
        // histograms (region A) and tie masks (region B) start at zero; A and B are adjacent
        uint4* a4 = reinterpret_cast<uint4*>(reg_a);
        for (int k = etid; k < 2 * kTokTile * kWords / 4; k += kEpiThreads) a4[k] = make_uint4(0u, 0u, 0u, 0u);
      }
      epi_sync();

      if (x.n_gt > 0) {
        const int32_t base0 = *bin_base;
        bool final_pass = false;
        for (int pass = 0; ok; ++pass) {
          // this warp's tokens: lane j (< kTokPerWarp) holds token tok0 + j's row state
          const RowState my = rows[tok0 + (lane % kTokPerWarp)];
          const bool mine = lane < kTokPerWarp;
          const uint32_t act = __ballot_sync(0xffffffffu, mine && (final_pass ? my.mode >= kTakeAll : my.mode == kActive));
          const uint32_t ties = __ballot_sync(0xffffffffu, mine && my.mode == kTies);
          const uint32_t cands = __ballot_sync(0xffffffffu, mine && my.mode == kCand);
          const bool lvl0 = my.level0 != 0u;         // the same for every active row of a pass
          const uint32_t lvl0_any = __ballot_sync(0xffffffffu, mine && my.mode == kActive && lvl0);
          // final pass: key > sel_gt selects; in_lo <= key <= sel_gt is the threshold bin
          // (take-all rows: in_lo = sel_gt + 1, an empty bin)
          const uint32_t my_sel_gt = my.mode == kTakeAll ? my.lo - 1u : my.hi;
          // (a take-all row has lo > 0: all keys >= 0 taken would mean nVis = 512)
          const uint32_t my_in_lo = my.lo;
          // the final pass's bin test starts at key 1: key 0 (a NaN pattern, never a visible
          // logit's) marks the blocks a token does not see
          const uint32_t my_in_lo1 = max(my.lo, 1u);
          // the final pass reads each token's pair with one broadcast shared load
          if (final_pass) {
            if (mine) thr_w[lane] = make_uint2(my_sel_gt, my_in_lo1);
            __syncwarp();
          }
          for (int i = 0; i < x.n_gt; ++i) {
            const int as = acnt % kAccStages;
            if (!wait_bounded(bar(kBarAccFull + as), (acnt / kAccStages) & 1, abort_flag, kFaultEpilogue)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const int32_t g = i * kGTile + 32 * sp + lane;
            const int wi = i * 4 + sp;               // mask word of this warp's 32 blocks
            // token tok0 + 8c + k sees block g iff 4g + 3 <= t, i.e. dv - 8c <= k
            const int32_t dv = 4 * g + 3 - (x.t0 + tok0);
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * sp) << 16) +
                                   static_cast<uint32_t>(as) * kAccCols + 4u * static_cast<uint32_t>(tok0);
            if (act != 0u) {
              uint32_t ra[32], rb[32];
              ptx::tmem_ld_32x32b_x32(taddr, ra);
              ptx::tmem_ld_wait(ra);
#pragma unroll
              for (int c = 0; c < kLdPerWarp; ++c) {
                uint32_t (&r)[32] = (c & 1) ? rb : ra;
                uint32_t (&nx)[32] = (c & 1) ? ra : rb;
                if (c + 1 < kLdPerWarp) ptx::tmem_ld_32x32b_x32(taddr + 32u * (c + 1), nx);
                const uint32_t a8 = (act >> (8 * c)) & 0xFFu;
                const int32_t dvc = dv - 8 * c;
                if (a8 != 0u) {
                  if (final_pass) {
                    // per token: its selected-bit word (kept by lane j, stored once for the 8
                    // tokens) and, per lane, which tokens hold a key of their threshold bin
                    uint32_t wsel = 0u, cbits = 0u, key8[8];
#pragma unroll
                    for (int k = 0; k < 8; k += 2) keys2(r, k, sc2, key8[k], key8[k + 1]);
                    // on a diagonal g-tile, a block a token does not see gets key 0: never above a
                    // threshold, never inside a bin (the test starts at key 1)
                    if (!__all_sync(0xffffffffu, dvc <= 0)) {
#pragma unroll
                      for (int k = 0; k < 8; ++k) key8[k] = dvc <= k ? key8[k] : 0u;
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                      const int j = 8 * c + k;       // token of this warp's slice
                      const uint32_t key = key8[k];
                      const uint2 th = thr_w[j];     // (sel_gt, in_lo) of token j
                      const uint32_t ws = __ballot_sync(0xffffffffu, key > th.x);
                      wsel = lane == k ? ws : wsel;
                      cbits |= (key >= th.y && key <= th.x) ? 1u << k : 0u;
                    }
                    // a row that is not in its final pass never reads this word again
                    if (lane < 8) reg_a[(tok0 + 8 * c + lane) * kWords + wi] = wsel;
                    const uint32_t todo_c = __reduce_or_sync(0xffffffffu, cbits) & a8;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                      if (!((todo_c >> kk) & 1u)) continue;  // the same for every lane
                      const int j = 8 * c + kk;
                      const int tt = tok0 + j;
                      const bool in = (cbits >> kk) & 1u;
                      const uint32_t wc = __ballot_sync(0xffffffffu, in);
                      if ((ties >> j) & 1u) {
                        if (lane == 0) reg_b[tt * kWords + wi] = wc;
                      } else if ((cands >> j) & 1u) {
                        const uint32_t kv = key8[kk];
                        const uint32_t in_lo = __shfl_sync(0xffffffffu, my_in_lo, j);
                        uint32_t at = 0u;
                        if (lane == 0) at = atomicAdd(&rows[tt].cnt, static_cast<uint32_t>(__popc(wc)));
                        at = __shfl_sync(0xffffffffu, at, 0);
                        const uint32_t slot = at + static_cast<uint32_t>(__popc(wc & ((1u << lane) - 1u)));
                        if (in && slot < static_cast<uint32_t>(kCap))
                          reg_b[tt * kWords + slot] = ((kv - in_lo) << 12) | static_cast<uint32_t>(g);
                      }
                    }
                  } else if (lvl0_any != 0u) {
                    // tokens of the group that count this lane's block: active rows that see it
                    const uint32_t cm8 = a8 & (dvc <= 0 ? 0xFFu : (dvc > 7 ? 0u : (0xFFu << dvc) & 0xFFu));
#pragma unroll
                    for (int k = 0; k < 8; k += 2) {
                      uint32_t key[2];
                      keys2(r, k, sc2, key[0], key[1]);
#pragma unroll
                      for (int h = 0; h < 2; ++h) {
                        const int j = 8 * c + k + h;
                        const uint32_t b = bin0_of(key[h], base0);
                        // every lane adds: a key the row does not count adds 0 (no divergence);
                        // rows outside this pass never read their histogram again
                        const bool cnt = (cm8 >> (k + h)) & 1u;
                        atomicAdd(&reg_a[(tok0 + j) * kWords + (b >> 1)], cnt ? 1u << ((b & 1u) << 4) : 0u);
                      }
                    }
                  } else {
                    const uint32_t cm8 = a8 & (dvc <= 0 ? 0xFFu : (dvc > 7 ? 0u : (0xFFu << dvc) & 0xFFu));
#pragma unroll
                    for (int k = 0; k < 8; k += 2) {
                      uint32_t key[2];
                      keys2(r, k, sc2, key[0], key[1]);
#pragma unroll
                      for (int h = 0; h < 2; ++h) {
                        const int j = 8 * c + k + h;
                        const uint32_t lo = __shfl_sync(0xffffffffu, my.lo, j);
                        const uint32_t hi = __shfl_sync(0xffffffffu, my.hi, j);
                        const uint32_t sh = __shfl_sync(0xffffffffu, my.shift, j);
                        const bool cnt = ((cm8 >> (k + h)) & 1u) && key[h] >= lo && key[h] <= hi;
                        const uint32_t b = cnt ? (key[h] - lo) >> sh : 0u;
                        atomicAdd(&reg_a[(tok0 + j) * kWords + (b >> 1)], cnt ? 1u << ((b & 1u) << 4) : 0u);
                      }
                    }
                  }
                }
                if (c + 1 < kLdPerWarp) ptx::tmem_ld_wait(nx);
              }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarAccEmpty + as));
            ++acnt;
          }
          if (!ok) break;
          epi_sync();
          if (final_pass) break;

          // ---- threshold search: one warp a row, for the rows still active
          for (int tt = ew; tt < kTokTile; tt += kEpiWarps) {
            RowState rs = rows[tt];
            if (rs.mode != kActive) continue;
            const uint4 v = reinterpret_cast<const uint4*>(reg_a + tt * kWords)[31 - lane];
            // this lane's 8 bins, highest first: bins 8*(31-lane) + 7 .. + 0
            const uint32_t b8[8] = {v.w >> 16, v.w & 0xFFFFu, v.z >> 16, v.z & 0xFFFFu,
                                    v.y >> 16, v.y & 0xFFFFu, v.x >> 16, v.x & 0xFFFFu};
            uint32_t mine8 = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) mine8 += b8[j];
            const uint32_t incl = warp_inclusive_sum(mine8, lane);
            const uint32_t excl = incl - mine8;
            const uint32_t want = static_cast<uint32_t>(rs.rem);
            const bool hit = excl < want && want <= incl;
            uint32_t fb = 0u, fabove = 0u, fcount = 0u;
            if (hit) {
              uint32_t c = excl;
              bool done = false;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                if (!done) {
                  if (c + b8[j] >= want) {
                    fb = 8u * static_cast<uint32_t>(31 - lane) + 7u - static_cast<uint32_t>(j);
                    fabove = c;
                    fcount = b8[j];
                    done = true;
                  } else {
                    c += b8[j];
                  }
                }
              }
            }
            const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
            fb = __shfl_sync(0xffffffffu, fb, src);
            fabove = __shfl_sync(0xffffffffu, fabove, src);
            fcount = __shfl_sync(0xffffffffu, fcount, src);
            uint32_t nlo, nhi;
            if (rs.level0) {
              bin0_range(fb, base0, nlo, nhi);
            } else {
              nlo = rs.lo + (fb << rs.shift);
              const uint64_t top = static_cast<uint64_t>(nlo) + ((1ull << rs.shift) - 1ull);
              nhi = static_cast<uint32_t>(min(top, static_cast<uint64_t>(rs.hi)));
            }
            if (rs.level0 && lane == 0 && fb >= 2u) {
              // where this row's threshold fell, for the next unit's first-pass base
              const int32_t d = fb == 2u ? base0 + 2 - 64 : (fb == 255u ? base0 + 255 + 64 : base0 + static_cast<int32_t>(fb));
              atomicAdd(base_sum, static_cast<uint32_t>(d));
              atomicAdd(base_n, 1u);
            }
            rs.rem -= static_cast<int32_t>(fabove);
            rs.lo = nlo;
            rs.hi = nhi;
            rs.level0 = 0u;
            rs.cnt = 0u;
            if (fcount == static_cast<uint32_t>(rs.rem)) {
              rs.mode = kTakeAll;
            } else if (nlo == nhi) {
              rs.mode = kTies;
            } else if (fcount <= static_cast<uint32_t>(kCap) && nhi - nlo < (1u << 20)) {
              rs.mode = kCand;
            } else {
              rs.mode = kActive;
              rs.shift = static_cast<uint32_t>(max(0, (32 - __clz(static_cast<int>(nhi - nlo))) - 8));
              // the row's histogram for the next pass
              reinterpret_cast<uint4*>(reg_a + tt * kWords)[lane] = make_uint4(0u, 0u, 0u, 0u);
              if (lane == 0) atomicAdd(n_active, 1u);
            }
            __syncwarp();
            if (lane == 0) rows[tt] = rs;
          }
          epi_sync();
          if (etid == 0) {
            const bool fin = *n_active == 0u;
            *n_active = 0u;
            *final_next = fin ? 1u : 0u;
            if (pass == 0 && *base_n > 0u) {
              const int32_t avg = static_cast<int32_t>(*base_sum / *base_n);
              *bin_base = min(max(avg - 128, kBaseMin), kBaseMax);
            }
            if (pass == 0) {
              *base_sum = 0u;
              *base_n = 0u;
            }
            const int ds = dcnt % kDecStages;
            if (wait_bounded(bar(kBarDecEmpty + ds), ((dcnt / kDecStages) & 1) ^ 1, abort_flag, kFaultEpilogue)) {
              dec[ds] = fin ? 1u : 0u;
              ptx::mbar_arrive(bar(kBarDecFull + ds));
            }
          }
          ++dcnt;
          epi_sync();
          if (*abort_flag) {
            ok = false;
            break;
          }
          final_pass = *final_next != 0u;
        }
        if (!ok) break;
      }

      // ---- winners of each row's threshold bin, then the row's 2051 ids
      for (int tt = ew; tt < kTokTile; tt += kEpiWarps) {
        const RowState rs = rows[tt];
        if (rs.mode == kSkip) continue;
        const int32_t t = x.t0 + tt;
        int32_t* out = p.out_idx + (x.row_base + t) * static_cast<int64_t>(sel::kWidth);
        if (rs.mode == kShort) {
          // token ids 0 .. 4*nVis + tail - 1 of an unpadded row; nothing of a padded one
          warp_write_unselected(out, t < x.t_vis_hi ? rs.n_vis * sel::kRatio + (t + 1) % sel::kRatio : 0, lane);
          continue;
        }
        uint32_t* selm = reg_a + tt * kWords;
        const int nw = (rs.n_vis + 31) / 32;
        if (rs.mode == kCand) {
          // rem of the cnt listed keys: largest first, equal keys by ascending block id;
          // sort key = offset, then 4095 - block, so all listed sort keys differ
          const int n = static_cast<int>(min(rs.cnt, static_cast<uint32_t>(kCap)));
          const uint32_t need = static_cast<uint32_t>(rs.rem);
          if (n <= 32) {
            const bool valid = lane < n;
            const uint32_t e = valid ? reg_b[tt * kWords + lane] : 0u;
            const uint32_t s = (e & 0xFFFFF000u) | (0xFFFu - (e & 0xFFFu));
            uint32_t rank = 0u;
            for (int j = 0; j < n; ++j) rank += __shfl_sync(0xffffffffu, s, j) > s ? 1u : 0u;
            if (valid && rank < need) {
              const uint32_t gb = e & 0xFFFu;
              atomicOr(&selm[gb >> 5], 1u << (gb & 31u));
            }
          } else {
            uint32_t e[4], s[4];
            bool valid[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int idx = lane + 32 * j;
              valid[j] = idx < n;
              e[j] = valid[j] ? reg_b[tt * kWords + idx] : 0u;
              s[j] = (e[j] & 0xFFFFF000u) | (0xFFFu - (e[j] & 0xFFFu));
            }
            uint32_t thr = 0u;
#pragma unroll 1
            for (int bit = 31; bit >= 0; --bit) {
              const uint32_t cand = thr | (1u << bit);
              uint32_t c = 0u;
#pragma unroll
              for (int j = 0; j < 4; ++j) c += __popc(__ballot_sync(0xffffffffu, valid[j] && s[j] >= cand));
              if (c >= need) thr = cand;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (valid[j] && s[j] >= thr) {
                const uint32_t gb = e[j] & 0xFFFu;
                atomicOr(&selm[gb >> 5], 1u << (gb & 31u));
              }
            }
          }
          __syncwarp();
        } else if (rs.mode == kTies) {
          // the first rem keys equal to lo, in ascending block order
          uint32_t w4[4], c4 = 0u;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int wj = 4 * lane + j;
            w4[j] = wj < nw ? reg_b[tt * kWords + wj] : 0u;
            c4 += __popc(w4[j]);
          }
          const uint32_t incl = warp_inclusive_sum(c4, lane);
          uint32_t before = incl - c4;
          const uint32_t need = static_cast<uint32_t>(rs.rem);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int wj = 4 * lane + j;
            if (wj >= nw) break;
            uint32_t keep = 0u, m = w4[j];
            while (m != 0u && before < need) {
              const uint32_t bit = m & (0u - m);
              keep |= bit;
              m &= m - 1u;
              ++before;
            }
            selm[wj] |= keep;
          }
          __syncwarp();
        }
        // ascending winners into this warp's stage, then the ids
        uint32_t w4[4], c4 = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int wj = 4 * lane + j;
          w4[j] = wj < nw ? selm[wj] : 0u;
          c4 += __popc(w4[j]);
        }
        const uint32_t incl = warp_inclusive_sum(c4, lane);
        uint32_t pos = incl - c4;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t m = w4[j];
          while (m != 0u) {
            const int bit = __ffs(m) - 1;
            m &= m - 1u;
            if (pos < static_cast<uint32_t>(sel::kTopK)) stage[pos] = static_cast<uint16_t>(32 * (4 * lane + j) + bit);
            ++pos;
          }
        }
        __syncwarp();
        warp_write_selected(out, stage, (t + 1) % sel::kRatio, rs.n_vis, lane);
        __syncwarp();
      }
      epi_sync();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace k2s

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn(cudaError_t* err) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (status == cudaSuccess && q != cudaDriverEntryPointSuccess) status = cudaErrorNotSupported;
    if (status == cudaSuccess) fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  *err = status;
  return fn;
}

// 3-D map over [dim2][dim1][128] two-byte elements, box {64, box1, 1}, 128-byte swizzle.
cudaError_t encode_rows(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* ptr,
                        uint64_t dim1, uint64_t dim2, uint32_t box1) {
  cuuint64_t dims[3] = {128, dim1, dim2};
  cuuint64_t strides[2] = {256, dim1 * 256};
  cuuint32_t box[3] = {64, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

std::mutex g_mu;
bool g_ready[64] = {};
uint32_t* g_sched_base[64] = {};
uint32_t g_launch_seq[64] = {};

}  // namespace

int32_t scores_topk_max_blocks() { return k2s::kMaxBlocks; }

cudaError_t launch_scores_topk_fused(const LaunchScoresTopk& a) {
  using namespace k2s;
  cudaError_t e;
  auto encode = get_encode_fn(&e);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  uint32_t slot = 0;
  uint32_t* sched_base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_ready[dev]) {
      e = cudaFuncSetAttribute(k2_topk_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBytes));
      if (e != cudaSuccess) return e;
      void* sched = nullptr;
      if ((e = cudaGetSymbolAddress(&sched, g_k2s_sched)) != cudaSuccess) return e;
      g_sched_base[dev] = static_cast<uint32_t*>(sched);
      g_ready[dev] = true;
    }
    slot = g_launch_seq[dev]++ % kFusedSchedSlots;
    sched_base = g_sched_base[dev];
  }
  CUtensorMap tq, tk;
  if ((e = encode_rows(encode, &tq, a.q_normed, 4ull * a.seq_len, a.batch, kN)) != cudaSuccess) return e;
  if ((e = encode_rows(encode, &tk, a.kbar, a.num_blocks, a.batch, kGTile)) != cudaSuccess) return e;

  Params p{};
  p.sched = sched_base + 2 * slot;
  p.out_idx = a.out_idx;
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
  const int64_t units = tile_hi - tile_lo;
  if (units > INT32_MAX - 65536) return cudaErrorInvalidValue;
  p.units = static_cast<int32_t>(units);
  p.idesc = ptx::idesc_f16(a.bf16, kGTile, kN);
  p.scale = a.scale;
  // each CTA then adapts the base to the thresholds it has seen
  p.base0 = bins::kDefaultBase;
  const int grid = static_cast<int>(units < a.num_sms ? units : a.num_sms);
  k2_topk_fused_kernel<<<grid, kThreads, kSmemBytes, a.stream>>>(tq, tk, p);
  return cudaGetLastError();
}

cudaError_t read_fused_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_k2s_fault_flags, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  if (clear && *flags != 0u) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_k2s_fault_flags, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
  }
  return e;
}

}  // namespace qsa
