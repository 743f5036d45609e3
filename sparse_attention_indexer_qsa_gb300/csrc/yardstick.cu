// Plain streaming kernels with a kernel's byte pattern, for the bench's same-size
// bandwidth yardsticks (qsa_testing_stream_yardstick, qsa_testing_gather_yardstick;
// test-only).
//
// stream_yardstick:
// Unit u reads `rows` slices of `bytes` bytes at src + u*unit_pitch + r*row_pitch +
// offset (r < rows), XORs them 16 bytes at a time and writes `bytes` bytes at
// dst + u*bytes.  One 16-byte chunk per thread, every row's load of a chunk issued
// before any is used, one unit per bytes/16 consecutive threads, no persistence:
// the simplest kernel that moves the same bytes in the same pattern as K1b
// (4 x 256 B at a 1280 B pitch in, 256 B out per block) or K1a (1024 B in and out
// per row).
#include <cstdint>

#include "qsa_launch.h"

namespace qsa {

namespace {

constexpr int kYardThreads = 256;
constexpr int kYardMaxRows = 8;

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kYardThreads)
stream_yardstick_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src, int64_t units, int rows,
                        int64_t row_pitch, int64_t unit_pitch, int64_t offset, int bytes) {
  const int tpu = bytes / 16;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kYardThreads + threadIdx.x;
  const int64_t u = tid / tpu;
  if (u >= units) return;
  const int64_t c = (tid - u * tpu) * 16;
  const uint8_t* p = src + u * unit_pitch + offset + c;
  uint4 v[kYardMaxRows];
#pragma unroll
  for (int r = 0; r < kYardMaxRows; ++r)
    if (r < rows) v[r] = ld_nc_v4(p + r * row_pitch);
  uint4 x = v[0];
#pragma unroll
  for (int r = 1; r < kYardMaxRows; ++r) {
    if (r < rows) {
      x.x ^= v[r].x;
      x.y ^= v[r].y;
      x.z ^= v[r].z;
      x.w ^= v[r].w;
    }
  }
  *reinterpret_cast<uint4*>(dst + u * bytes + c) = x;
}

// gather_yardstick: unit u reads `bytes` bytes at src + u*unit_pitch + offset and writes
// the XOR of their 32-bit words, 4 bytes, at dst + 4u: the paged decode scoring's
// pattern (one 256-byte V-tail a block at the pool's block pitch in, one FP32 logit a
// block out).  A group of tpu = bytes/16 consecutive lanes takes kGatherUnits
// consecutive units, issues all their 16-byte loads before using any, and reduces each
// unit across its lanes with shuffles.
constexpr int kGatherUnits = 4;

__global__ void __launch_bounds__(kYardThreads)
gather_yardstick_kernel(uint32_t* __restrict__ dst, const uint8_t* __restrict__ src, int64_t units,
                        int64_t unit_pitch, int64_t offset, int tpu) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kYardThreads + threadIdx.x;
  const int64_t group = tid / tpu;
  const int c = static_cast<int>(tid - group * tpu);
  const int64_t u0 = group * kGatherUnits;
  uint4 v[kGatherUnits];
#pragma unroll
  for (int k = 0; k < kGatherUnits; ++k) {
    v[k] = make_uint4(0u, 0u, 0u, 0u);
    if (u0 + k < units) v[k] = ld_nc_v4(src + (u0 + k) * unit_pitch + offset + 16 * c);
  }
#pragma unroll
  for (int k = 0; k < kGatherUnits; ++k) {
    uint32_t x = v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    for (int o = tpu >> 1; o > 0; o >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, o);  // every lane takes part
    if (c == 0 && u0 + k < units) dst[u0 + k] = x;
  }
}

}  // namespace

int yardstick_max_rows() { return kYardMaxRows; }

cudaError_t launch_gather_yardstick(void* dst, const void* src, int64_t units, int64_t unit_pitch, int64_t offset,
                                    int bytes, cudaStream_t stream) {
  const int tpu = bytes / 16;  // a power of two in [1, 32]: a group never straddles a warp
  const int64_t groups = (units + kGatherUnits - 1) / kGatherUnits;
  const int64_t grid = (groups * tpu + kYardThreads - 1) / kYardThreads;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  gather_yardstick_kernel<<<static_cast<unsigned>(grid), kYardThreads, 0, stream>>>(
      static_cast<uint32_t*>(dst), static_cast<const uint8_t*>(src), units, unit_pitch, offset, tpu);
  return cudaGetLastError();
}

cudaError_t launch_stream_yardstick(void* dst, const void* src, int64_t units, int rows, int64_t row_pitch,
                                    int64_t unit_pitch, int64_t offset, int bytes, cudaStream_t stream) {
  const int64_t threads = units * (bytes / 16);
  const int64_t grid = (threads + kYardThreads - 1) / kYardThreads;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  stream_yardstick_kernel<<<static_cast<unsigned>(grid), kYardThreads, 0, stream>>>(
      static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), units, rows, row_pitch, unit_pitch, offset, bytes);
  return cudaGetLastError();
}

}  // namespace qsa
