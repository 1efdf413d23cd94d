// Confidence head and survival products:
//   c_{r,j} = sigma(w_h . h_{r,j} + w_e . W1[x_{r,j-1}])   ("DSpark" §3.1, eq. c_k)
//   a_{r,j} = prod_{i<=j} c_{r,i}, left to right in fp32   (§1.1, eq. a_j)
// With sequential temperature scaling (§3.2, STS) the logit of position j is
// divided by its fitted temperature t_j before the sigmoid.
// The kernel streams h from HBM (R * gamma * d bf16).  One cluster of
// kConfCluster CTAs per request (position j on CTA j % kConfCluster), so that
// even a small batch fills the SMs.  Within a CTA each warp takes a slice of
// the d dimension: it loads its slice of w once and applies it to the h rows
// of up to kConfMaxPos positions at a time, all those loads in flight
// together; the slices' partial sums meet in shared memory.  fp32
// accumulation; each c_j goes to the leader CTA's shared memory (distributed
// shared memory), and after a cluster barrier one thread of the leader forms
// the running product in position order.
#include <cmath>

#include "common.h"
#include "device.cuh"

namespace dspark {

constexpr int kConfWarps = 4;    // warps per CTA
constexpr int kConfCluster = 4;  // CTAs per request (one thread-block cluster)
constexpr int kConfUnroll = 8;
constexpr int kConfMaxPos = 4;   // positions per CTA per round (their h rows share each w slice)

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Stores v into CTA `rank`'s shared-memory word at the address of `local`.
__device__ __forceinline__ void st_cluster_f32(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// sum_i x[i] * w[i] over n elements, x bf16 and w fp32 in global memory (the
// vector path when both are 16-byte aligned).
__device__ __forceinline__ float dot_bf16_f32(const uint16_t* x, const float* w, int n, int lane) {
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) && ((reinterpret_cast<uintptr_t>(w) & 15u) == 0);
  float acc[kConfUnroll];
#pragma unroll
  for (int u = 0; u < kConfUnroll; ++u) acc[u] = 0.f;
  int done = 0;
  if (vec) {
    const int n8 = n / 8;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    // kConfUnroll loads per lane in flight per round; the last round is
    // predicated rather than a serial tail
    for (int i = lane; i < n8; i += kConfUnroll * 32) {
      uint4 xv[kConfUnroll];
#pragma unroll
      for (int u = 0; u < kConfUnroll; ++u)
        xv[u] = i + u * 32 < n8 ? __ldcs(x8 + i + u * 32) : make_uint4(0u, 0u, 0u, 0u);  // all loads in flight first
#pragma unroll
      for (int u = 0; u < kConfUnroll; ++u) {
        if (i + u * 32 >= n8) continue;
        const float4 wa = __ldg(w4 + 2 * (i + u * 32)), wb = __ldg(w4 + 2 * (i + u * 32) + 1);
        float a = acc[u];
        a = fmaf(bf16_lo(xv[u].x), wa.x, a);
        a = fmaf(bf16_hi(xv[u].x), wa.y, a);
        a = fmaf(bf16_lo(xv[u].y), wa.z, a);
        a = fmaf(bf16_hi(xv[u].y), wa.w, a);
        a = fmaf(bf16_lo(xv[u].z), wb.x, a);
        a = fmaf(bf16_hi(xv[u].z), wb.y, a);
        a = fmaf(bf16_lo(xv[u].w), wb.z, a);
        a = fmaf(bf16_hi(xv[u].w), wb.w, a);
        acc[u] = a;
      }
    }
    done = n8 * 8;
  }
  for (int i = done + lane; i < n; i += 32) acc[0] = fmaf(bf16_at(x + i), __ldg(w + i), acc[0]);
  float s = 0.f;
#pragma unroll
  for (int u = 0; u < kConfUnroll; ++u) s += acc[u];
  return s;
}

// Partial sums of one CTA's positions: warp w takes the 8-element groups
// g = w, w + kConfWarps, ... of [0, d) (a slice of w it loads once, in
// registers) and multiplies it into the h rows of every position of the CTA;
// kConfUnroll loads of h per lane are in flight at a time.
__device__ __forceinline__ void slice_dots(const uint16_t* __restrict__ h, const float* __restrict__ w, int d, int r,
                                           int gamma, int j0, int nj, int warp, int lane, float (&part)[kConfMaxPos]) {
  const int n8 = d / 8;
#pragma unroll
  for (int q = 0; q < kConfMaxPos; ++q) part[q] = 0.f;
#pragma unroll 2
  for (int g = warp * 32 + lane; g < n8; g += kConfWarps * 32) {
    const float4 wa = __ldg(reinterpret_cast<const float4*>(w) + 2 * g);
    const float4 wb = __ldg(reinterpret_cast<const float4*>(w) + 2 * g + 1);
    uint4 xv[kConfMaxPos];
#pragma unroll
    for (int q = 0; q < kConfMaxPos; ++q)
      xv[q] = q < nj ? __ldcs(reinterpret_cast<const uint4*>(h + (static_cast<size_t>(r) * gamma + j0 + q * kConfCluster) * d) + g)
                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int q = 0; q < kConfMaxPos; ++q) {
      float a = part[q];
      a = fmaf(bf16_lo(xv[q].x), wa.x, a);
      a = fmaf(bf16_hi(xv[q].x), wa.y, a);
      a = fmaf(bf16_lo(xv[q].y), wa.z, a);
      a = fmaf(bf16_hi(xv[q].y), wa.w, a);
      a = fmaf(bf16_lo(xv[q].z), wb.x, a);
      a = fmaf(bf16_hi(xv[q].z), wb.y, a);
      a = fmaf(bf16_lo(xv[q].w), wb.z, a);
      a = fmaf(bf16_hi(xv[q].w), wb.w, a);
      part[q] = a;
    }
  }
}

__global__ void __launch_bounds__(kConfWarps * 32)
    k2_confidence(const uint16_t* __restrict__ h, const uint16_t* __restrict__ W1, const float* __restrict__ w,
                  const float* __restrict__ sts_t, const int32_t* __restrict__ anchors,
                  const int32_t* __restrict__ tokens, int R, int gamma, int d, int rank, int V, float* __restrict__ c_out,
                  float* __restrict__ a_out, int32_t* status) {
  __shared__ float s_c[kMaxGamma];                      // the leader CTA's copy is the one used
  __shared__ float s_part[kConfWarps][kConfMaxPos];     // per-warp partial sums of the h dots
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t crank = cluster_ctarank();
  const int r = blockIdx.x / kConfCluster;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool vec = (d % 8) == 0 && (reinterpret_cast<uintptr_t>(h) & 15u) == 0 && (reinterpret_cast<uintptr_t>(w) & 15u) == 0;
  // this CTA's positions j = crank + kConfCluster * q, in rounds of kConfMaxPos
  for (int base = static_cast<int>(crank); base < gamma; base += kConfCluster * kConfMaxPos) {
    const int nj = min(kConfMaxPos, (gamma - base + kConfCluster - 1) / kConfCluster);
    if (vec) {
      float part[kConfMaxPos];
      slice_dots(h, w, d, r, gamma, base, nj, warp, lane, part);
#pragma unroll
      for (int q = 0; q < kConfMaxPos; ++q) {
        const float s = warp_sum(part[q]);
        if (lane == 0) s_part[warp][q] = s;
      }
    }
    __syncthreads();
    // one warp per position: the W1 row's dot, the h dot (summed over the
    // slices, or computed here when h or w is not 16-byte aligned), sigmoid
    for (int q = warp; q < nj; q += kConfWarps) {
      const int j = base + q * kConfCluster;
      int prev = j == 0 ? anchors[r] : tokens[static_cast<size_t>(r) * gamma + j - 1];
      if (prev < 0 || prev >= V) {
        if (lane == 0) report(status, DSPARK_STATUS_BAD_TOKEN);
        prev = 0;
      }
      float s = dot_bf16_f32(W1 + static_cast<size_t>(prev) * rank, w + d, rank, lane);
      if (!vec) s += dot_bf16_f32(h + (static_cast<size_t>(r) * gamma + j) * d, w, d, lane);
      s = warp_sum(s);
      if (vec) {
#pragma unroll
        for (int w2 = 0; w2 < kConfWarps; ++w2) s += s_part[w2][q];
      }
      if (sts_t != nullptr) {
        float t = __ldg(sts_t + j);
        if (!(t > 0.f) || !(t <= 3.4e38f)) {  // zero, negative, NaN or infinite: no scaling
          if (lane == 0) report(status, DSPARK_STATUS_NONFINITE);
          t = 1.f;
        }
        s = __fdiv_rn(s, t);
      }
      if (lane == 0) st_cluster_f32(&s_c[j], 0u, 1.0f / (1.0f + expf(-s)));
    }
    __syncthreads();  // s_part is rewritten by the next round
  }
  cluster_sync_all();  // every c_j of the request is in the leader's shared memory
  if (crank == 0 && threadIdx.x == 0) {
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(R * kConfCluster);
  cfg.blockDim = dim3(kConfWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kConfCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k2_confidence, h, W1, w, sts_t, anchors, tokens, R, gamma, d, rank, V,
                                           c, a, status);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark
