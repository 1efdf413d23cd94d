// Confidence head and survival products:
//   c_{r,j} = sigma(w_h . h_{r,j} + w_e . W1[x_{r,j-1}])   ("DSpark" §3.1, eq. c_k)
//   a_{r,j} = prod_{i<=j} c_{r,i}, left to right in fp32   (§1.1, eq. a_j)
// With sequential temperature scaling (§3.2, STS) the logit of position j is
// divided by its fitted temperature t_j before the sigmoid.
// One CTA per request, one warp per position (strided); fp32 accumulation of
// the two dot products; the running product by one thread in position order.
#include <cmath>

#include "common.h"
#include "device.cuh"

namespace dspark {

constexpr int kConfWarps = 16;

__device__ __forceinline__ float dot_bf16_f32(const uint16_t* x, const float* w, int n, int lane) {
  float acc = 0.f;
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) && ((reinterpret_cast<uintptr_t>(w) & 15u) == 0);
  int done = 0;
  if (vec) {
    const int n8 = n / 8;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    for (int i = lane; i < n8; i += 32) {
      const uint4 xv = __ldg(x8 + i);
      const float4 wa = __ldg(w4 + 2 * i), wb = __ldg(w4 + 2 * i + 1);
      acc = fmaf(bf16_lo(xv.x), wa.x, acc);
      acc = fmaf(bf16_hi(xv.x), wa.y, acc);
      acc = fmaf(bf16_lo(xv.y), wa.z, acc);
      acc = fmaf(bf16_hi(xv.y), wa.w, acc);
      acc = fmaf(bf16_lo(xv.z), wb.x, acc);
      acc = fmaf(bf16_hi(xv.z), wb.y, acc);
      acc = fmaf(bf16_lo(xv.w), wb.z, acc);
      acc = fmaf(bf16_hi(xv.w), wb.w, acc);
    }
    done = n8 * 8;
  }
  for (int i = done + lane; i < n; i += 32) acc = fmaf(bf16_at(x + i), __ldg(w + i), acc);
  return acc;
}

__global__ void __launch_bounds__(kConfWarps * 32)
    k2_confidence(const uint16_t* __restrict__ h, const uint16_t* __restrict__ W1, const float* __restrict__ w,
                  const float* __restrict__ sts_t, const int32_t* __restrict__ anchors,
                  const int32_t* __restrict__ tokens, int R, int gamma, int d, int rank, int V, float* __restrict__ c_out, float* __restrict__ a_out, int32_t* status) {
  __shared__ float s_c[kMaxGamma];
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < gamma; j += kConfWarps) {
    int prev = j == 0 ? anchors[r] : tokens[static_cast<size_t>(r) * gamma + j - 1];
    if (prev < 0 || prev >= V) {
      if (lane == 0) report(status, DSPARK_STATUS_BAD_TOKEN);
      prev = 0;
    }
    float s = dot_bf16_f32(h + (static_cast<size_t>(r) * gamma + j) * d, w, d, lane);
    s += dot_bf16_f32(W1 + static_cast<size_t>(prev) * rank, w + d, rank, lane);
    s = warp_sum(s);
    if (sts_t != nullptr) {
      float t = __ldg(sts_t + j);
      if (!(t > 0.f) || !(t <= 3.4e38f)) {  // zero, negative, NaN or infinite: no scaling
        if (lane == 0) report(status, DSPARK_STATUS_NONFINITE);
        t = 1.f;
      }
      s = __fdiv_rn(s, t);
    }
    if (lane == 0) s_c[j] = 1.0f / (1.0f + expf(-s));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float run = 1.0f;
    for (int j = 0; j < gamma; ++j) {
      const float cj = s_c[j];
      run = __fmul_rn(run, cj);
      c_out[static_cast<size_t>(r) * gamma + j] = cj;
      a_out[static_cast<size_t>(r) * gamma + j] = run;
    }
  }
}

int launch_confidence(const uint16_t* h, const uint16_t* W1, const float* w, const float* sts_t,
                      const int32_t* anchors, const int32_t* tokens, int R, int gamma, int d, int rank, int V,
                      float* c, float* a, int32_t* status, cudaStream_t stream) {
  const cudaError_t e = launch_pdl(k2_confidence, dim3(R), dim3(kConfWarps * 32), 0, stream, true, h, W1, w, sts_t,
                                   anchors, tokens, R, gamma, d, rank, V, c, a, status);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark
