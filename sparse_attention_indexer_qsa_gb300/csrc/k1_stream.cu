// Fused K1a + prefill K1b in ONE pass over indexQk ("Qsa Indexer Kernels",
// launchQsaIndexQPrep and launchQsaIndexKCompress with blockBegin = 0,
// blockEnd = ceilDiv(S, 4), pastLen = 0, as the prefill pipeline calls them).
//
// One CTA (4 warps) per work unit of 16 consecutive token rows of one sequence
// (4 compressed blocks); six CTAs per SM keep units in flight, and the hardware
// hands out CTAs in address order (on GB300, persistent CTAs on a static schedule
// drift apart and stream noticeably slower).  Thread 0 copies the unit's valid rows
// (a prefix of the sequence, so contiguous) and their cos/sin rows into shared
// memory with bulk asynchronous copies (cp.async.bulk, completion counted on an
// mbarrier); the warps then run the same norm_rope_group device routine as the
// register-streaming kernels on data read from shared memory, so outputs are
// bit-identical to them.  Mode QK reads each 1280-byte row once, as one contiguous
// copy, where the two separate kernels read its 1024-byte q part and its 256-byte K
// slice; the bytes are the same, and the pass saves one launch and its ramp.
//
// Padding rows (t >= contextLengths[b]) and invalid blocks are written as exact
// zeros and are never copied.  The one mbarrier wait is bounded; a wait that runs
// out sets a bit in the fault word and the CTA writes nothing.
#include <cstdint>

#include "qsa_common.cuh"
#include "qsa_launch.h"
#include "tc_ptx.cuh"

namespace qsa {

__device__ uint32_t g_k1_fault_flags;

namespace k1s {

constexpr int kModeQ = 1;   // q heads only (qsa_index_q_prep): each row's 1024-byte q part staged
constexpr int kModeQK = 3;  // q heads and compressed k together (qsa_index_qk_prep): whole rows
#ifndef QSA_K1S_ROWS
#define QSA_K1S_ROWS 16
#endif
#ifndef QSA_K1S_CTAS
#define QSA_K1S_CTAS 7
#endif
constexpr int kRows = QSA_K1S_ROWS;       // token rows per unit (one CTA)
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kCtasPerSm = QSA_K1S_CTAS;
static_assert(kRows % (kRatio * 2) == 0 && kRows / kRatio <= 2 * 4, "blocks of a unit: two 8-lane groups a warp");
constexpr uint32_t kCsBytes = kCsWidth * 4;  // 256-byte cos/sin row

template <int MODE>
struct Layout {
  static_assert(MODE == kModeQK || MODE == kModeQ, "modes built: q, q and k");
  // whole 1280-byte indexQk rows, or their 1024-byte q parts
  static constexpr uint32_t kRowBytes = MODE == kModeQK ? kRowWidth * 2 : kNumQHeads * kHeadDim * 2;
  static constexpr uint32_t kRowsOff = 0;
  static constexpr uint32_t kCsOff = kRows * kRowBytes;
  static constexpr uint32_t kStageBytes = kCsOff + kRows * kCsBytes;
  static constexpr uint32_t kGammaOff = kStageBytes;                    // 2 x 128 floats
  static constexpr uint32_t kBarOff = kGammaOff + 2 * kHeadDim * 4;     // one mbarrier
  static constexpr uint32_t kSmemBytes = kBarOff + 16 + 128;            // + slack to align to 128
  static_assert(kStageBytes % 128 == 0, "stage alignment");
  static_assert(kCtasPerSm * kSmemBytes <= 232448, "shared memory for the intended occupancy");
};

struct Params {
  uint16_t* q_normed;
  uint16_t* kbar;                // mode QK only
  const uint16_t* index_qk;
  const float* cos_sin;
  const int32_t* ctx;
  const uint16_t* w_q;
  const uint16_t* w_k;           // mode QK only
  float eps;
  int32_t batch, seq_len, num_blocks;
  int32_t units_per_seq;         // ceilDiv(seq_len, kRows)
};

constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Bounded wait for this CTA's own copies; on time-out set a fault bit and report.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t start = ptx::global_timer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::global_timer_ns() - start > kWaitLimitNs) {
      atomicOr(&g_k1_fault_flags, 1u);
      return false;
    }
  }
  return true;
}

// bulk global -> shared copy; both addresses 16-byte aligned, size a multiple of 16
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ RopeCS lds_rope(uint32_t cs_row, int j) {
  RopeCS r;
  const uint32_t p = cs_row + 32u * (j & 3);
  uint4 c0 = lds_v4(p), c1 = lds_v4(p + 16), s0 = lds_v4(p + 128), s1 = lds_v4(p + 144);
  r.c0 = make_float4(__uint_as_float(c0.x), __uint_as_float(c0.y), __uint_as_float(c0.z), __uint_as_float(c0.w));
  r.c1 = make_float4(__uint_as_float(c1.x), __uint_as_float(c1.y), __uint_as_float(c1.z), __uint_as_float(c1.w));
  r.s0 = make_float4(__uint_as_float(s0.x), __uint_as_float(s0.y), __uint_as_float(s0.z), __uint_as_float(s0.w));
  r.s1 = make_float4(__uint_as_float(s1.x), __uint_as_float(s1.y), __uint_as_float(s1.z), __uint_as_float(s1.w));
  return r;
}

// Chunks chunk_a(j) and chunk_b(j) of a staged 128-dim vector (2-byte elements at `row`).
// Within one 16-byte load, lanes j < 4 and j >= 4 of a group would read their chunk A
// from the same banks (bytes 16j and 128 + 16(j - 4)); lanes j >= 4 load chunk B first,
// so each load's eight lanes of a group cover 32 distinct banks.
template <class T>
__device__ __forceinline__ void lds_pair(uint32_t row, int ca, int cb, int j, float (&a)[8], float (&b)[8]) {
  const bool swap = j >= 4;
  const uint4 first = lds_v4(row + 2 * (swap ? cb : ca));
  const uint4 second = lds_v4(row + 2 * (swap ? ca : cb));
  unpack8<T>(swap ? second : first, a);
  unpack8<T>(swap ? first : second, b);
}

// valid (copied) rows of unit u: the prefix [t0, t0 + nq)
__device__ __forceinline__ void unit_rows(const Params& p, int32_t u, int32_t& b, int32_t& t0, int32_t& nq) {
  b = u / p.units_per_seq;
  t0 = (u - b * p.units_per_seq) * kRows;
  const int32_t lim = min(max(__ldg(p.ctx + b), 0), p.seq_len);
  nq = min(max(lim - t0, 0), kRows);
}

template <class T, int MODE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k1_stream_kernel(const Params p) {
  using L = Layout<MODE>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  float* g1q = reinterpret_cast<float*>(base_ptr + L::kGammaOff);
  float* g1k = g1q + kHeadDim;
  const uint32_t bar = base + L::kBarOff;

  // A kernel launched after this one as a programmatic dependent (K2 scoring these rows)
  // may start launching once every CTA of this grid has started: its CTAs then take the
  // SMs this grid's last CTAs leave and set up there, and wait for this grid to complete
  // before they read its outputs.
  ptx::launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int32_t b, t0, nq;
  unit_rows(p, static_cast<int32_t>(blockIdx.x), b, t0, nq);
  const int64_t row0 = static_cast<int64_t>(b) * p.seq_len + t0;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_barrier_init();
    ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nq) * (L::kRowBytes + kCsBytes));
    if (nq > 0) {
      if (MODE == kModeQK) {  // the unit's valid rows are contiguous: one copy
        bulk_load(base + L::kRowsOff, p.index_qk + row0 * kRowWidth, nq * L::kRowBytes, bar);
      } else {  // each row's q part (1280-byte pitch, 16-byte aligned)
        for (int r = 0; r < nq; ++r)
          bulk_load(base + L::kRowsOff + r * L::kRowBytes, p.index_qk + (row0 + r) * kRowWidth, L::kRowBytes, bar);
      }
      bulk_load(base + L::kCsOff, p.cos_sin + static_cast<int64_t>(t0) * kCsWidth, nq * kCsBytes, bar);
    }
  }
  stage_gamma<T>(p.w_q, g1q);
  if (MODE == kModeQK) stage_gamma<T>(p.w_k, g1k);
  __syncthreads();
  const bool ok = wait_bounded(bar, 0);

  const int h = lane >> 3;
  const int j = lane & 7;
  const int ca = chunk_a(j);
  const int cb = chunk_b(j);
  if (ok) {
    // K1a: warp w owns rows w, w+4, w+8, ... of the unit
#pragma unroll 1
    for (int r = warp; r < kRows; r += kWarps) {
      if (t0 + r >= p.seq_len) break;  // warp-uniform
      uint16_t* dst = p.q_normed + (row0 + r) * (kNumQHeads * kHeadDim) + h * kHeadDim;
      uint4 oa = make_uint4(0u, 0u, 0u, 0u), ob = oa;
      if (r < nq) {  // warp-uniform
        const uint32_t row = base + L::kRowsOff + r * L::kRowBytes + h * (kHeadDim * 2);
        float a[8], bv[8];
        lds_pair<T>(row, ca, cb, j, a, bv);
        RopeCS cs{};
        if (j < 4) cs = lds_rope(base + L::kCsOff + r * kCsBytes, j);
        norm_rope_group<T>(a, bv, g1q, p.eps, cs, j, oa, ob);
      }
      st_v4(dst + ca, oa);
      st_v4(dst + cb, ob);
    }
    if (MODE == kModeQK) {
      // K1b: the 8-lane group h of warp w owns block jb = 2*w + h (h < 2, jb < kRows/4) of the unit
      const int jb = 2 * warp + (h & 1);
      const int32_t g = t0 / kRatio + jb;
      const bool mine = h < 2 && jb < kRows / kRatio;
      const bool exists = mine && kRatio * g < p.seq_len;        // g < ceilDiv(S, 4)
      const bool valid = exists && kRatio * jb + (kRatio - 1) < nq;  // its four rows were copied
      float a[8], bv[8];
      RopeCS cs{};
      if (valid) {
        float fa[kRatio][8], fb[kRatio][8];
#pragma unroll
        for (int q = 0; q < kRatio; ++q) {
          const uint32_t row = base + L::kRowsOff + (kRatio * jb + q) * L::kRowBytes + kKCol * 2;
          lds_pair<T>(row, ca, cb, j, fa[q], fb[q]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float sm = __fadd_rn(__fadd_rn(__fadd_rn(fa[0][e], fa[1][e]), fa[2][e]), fa[3][e]);
          a[e] = T::round_trip(__fmul_rn(sm, 0.25f));
          sm = __fadd_rn(__fadd_rn(__fadd_rn(fb[0][e], fb[1][e]), fb[2][e]), fb[3][e]);
          bv[e] = T::round_trip(__fmul_rn(sm, 0.25f));
        }
        if (j < 4) cs = lds_rope(base + L::kCsOff + (kRatio * jb) * kCsBytes, j);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) { a[e] = 0.0f; bv[e] = 0.0f; }
      }
      uint4 oa, ob;
      norm_rope_group<T>(a, bv, g1k, p.eps, cs, j, oa, ob);
      if (exists) {
        if (!valid) { oa = make_uint4(0u, 0u, 0u, 0u); ob = oa; }
        uint16_t* dst = p.kbar + (static_cast<int64_t>(b) * p.num_blocks + g) * kHeadDim;
        st_v4(dst + ca, oa);
        st_v4(dst + cb, ob);
      }
    }
  }
}

}  // namespace k1s

namespace {

template <class T, int MODE>
cudaError_t launch_mode(const k1s::Params& p, int num_sms, cudaStream_t stream) {
  using L = k1s::Layout<MODE>;
  auto kern = k1s::k1_stream_kernel<T, MODE>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {  // idempotent: a racing second set is harmless
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  (void)num_sms;
  const int units = p.batch * p.units_per_seq;
  kern<<<units, k1s::kThreads, L::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

k1s::Params make_params(void* q_normed, void* kbar, const void* index_qk, const float* cos_sin,
                        const int32_t* ctx, const void* w_q, const void* w_k, float eps, int32_t batch,
                        int32_t seq_len, int32_t num_blocks) {
  k1s::Params p{};
  p.q_normed = static_cast<uint16_t*>(q_normed);
  p.kbar = static_cast<uint16_t*>(kbar);
  p.index_qk = static_cast<const uint16_t*>(index_qk);
  p.cos_sin = cos_sin;
  p.ctx = ctx;
  p.w_q = static_cast<const uint16_t*>(w_q);
  p.w_k = static_cast<const uint16_t*>(w_k);
  p.eps = eps;
  p.batch = batch;
  p.seq_len = seq_len;
  p.num_blocks = num_blocks;
  p.units_per_seq = (seq_len + k1s::kRows - 1) / k1s::kRows;
  return p;
}

}  // namespace

cudaError_t launch_q_prep_staged(const LaunchQPrep& a) {
  const k1s::Params p = make_params(a.q_normed, nullptr, a.index_qk, a.cos_sin, a.context_lengths, a.w_q,
                                    nullptr, a.eps, a.batch, a.seq_len, 0);
  return a.bf16 ? launch_mode<Bf16, k1s::kModeQ>(p, a.num_sms, a.stream)
                : launch_mode<F16, k1s::kModeQ>(p, a.num_sms, a.stream);
}

cudaError_t launch_qk_prep(const LaunchQKPrep& a) {
  const k1s::Params p = make_params(a.q_normed, a.kbar, a.index_qk, a.cos_sin, a.context_lengths, a.w_q,
                                    a.w_k, a.eps, a.batch, a.seq_len, a.num_blocks);
  return a.bf16 ? launch_mode<Bf16, k1s::kModeQK>(p, a.num_sms, a.stream)
                : launch_mode<F16, k1s::kModeQK>(p, a.num_sms, a.stream);
}

cudaError_t read_k1_fault_flags(uint32_t* flags, bool clear, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(flags, g_k1_fault_flags, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
  if (clear && *flags != 0u) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_k1_fault_flags, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
  }
  return e;
}

}  // namespace qsa
