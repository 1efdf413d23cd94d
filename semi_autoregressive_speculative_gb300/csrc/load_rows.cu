// dspark_load_verified_rows: copy into device memory, from page-locked host
// memory, the target rows that verify reads (rows 0..lens[r] of request r).
//
// The lengths come from the scheduler on the device, so the set of rows is
// only known there.  A copy engine would need them on the host first (a
// device-to-host read and a stream synchronisation) and one copy per request;
// instead the SMs read the mapped host memory directly, each CTA taking
// 32 KB pieces of the admitted rows.  The host link (far below HBM speed) is
// the bound, and the copy engines stay free for the bulk copies of the next
// round that run at the same time.
#include <cstdint>

#include "common.h"
#include "device.cuh"

namespace dspark {

constexpr int kLoadThreads = 256;
constexpr int kLoadVec = 8;                                  // float4 loads in flight per thread
constexpr int kLoadPiece4 = kLoadThreads * kLoadVec;         // float4 per piece (32 KB)

// Units are (row slot s = r * (gamma + 1) + j, piece c), grid-strided; a unit
// whose row lies past lens[r] is skipped.
__global__ void __launch_bounds__(kLoadThreads) k_load_rows(const float4* __restrict__ src,
                                                            const int32_t* __restrict__ lens, int gamma,
                                                            long long n4, long long n_pieces, long long units,
                                                            float4* __restrict__ dst, int32_t* status) {
  const int g1 = gamma + 1;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const long long s = u / n_pieces;
    const long long c = u - s * n_pieces;
    const int r = static_cast<int>(s / g1);
    const int j = static_cast<int>(s - static_cast<long long>(r) * g1);
    int len = __ldg(lens + r);
    if (len < 0 || len > gamma) {
      if (j == 0 && c == 0 && threadIdx.x == 0) report(status, DSPARK_STATUS_BAD_LENGTH);
      len = len < 0 ? 0 : gamma;
    }
    if (j > len) continue;
    const long long base = s * n4 + c * kLoadPiece4 + threadIdx.x;
    const long long end = (s + 1) * n4;
    float4 v[kLoadVec];
#pragma unroll
    for (int i = 0; i < kLoadVec; ++i) {
      const long long k = base + static_cast<long long>(i) * kLoadThreads;
      if (k < end) v[i] = __ldcs(src + k);
    }
#pragma unroll
    for (int i = 0; i < kLoadVec; ++i) {
      const long long k = base + static_cast<long long>(i) * kLoadThreads;
      if (k < end) dst[k] = v[i];
    }
  }
}

int launch_load_verified_rows(const float* T_host, const int32_t* lens, int R, int gamma, int V, float* T,
                              int32_t* status, cudaStream_t stream) {
  // The source must be page-locked host memory mapped into the device's
  // address space; anything else is refused before a launch.
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, T_host) != cudaSuccess) {
    (void)cudaGetLastError();
    return DSPARK_ERR_INVALID_ARG;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return DSPARK_ERR_INVALID_ARG;
  const float4* src = static_cast<const float4*>(attr.devicePointer);
  if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0) return DSPARK_ERR_INVALID_ARG;
  const long long n4 = V / 4;  // V % 8 == 0
  const long long n_pieces = (n4 + kLoadPiece4 - 1) / kLoadPiece4;
  const long long units = static_cast<long long>(R) * (gamma + 1) * n_pieces;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  const int grid = static_cast<int>(units < cap ? units : cap);
  k_load_rows<<<grid, kLoadThreads, 0, stream>>>(src, lens, gamma, n4, n_pieces, units,
                                                 reinterpret_cast<float4*>(T), status);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark
