// Sampling searches shared by the draft sampler and verify: the first item
// whose running sum of weights exceeds a target, per warp and per block, and
// block-wide max / sum reductions.
#pragma once

#include "device.cuh"

namespace dspark {

// Segmented search across one warp.  Weights w(i), i in [0, n), are summed
// per lane over contiguous segments; returns the first i whose inclusive
// prefix (starting at `base`) exceeds `target`, or the last i with w(i) > 0
// when rounding leaves the total at or below the target.  *before = the
// prefix just before the returned i.  fp32 throughout: GB300's fp64 rate is
// a small fraction of its fp32 rate, and tree-ordered scans keep the
// relative error of every prefix near log2(n) * 2^-24 (about 1e-6 for 1024
// items), well inside the 1e-5 CDF tolerance of the sampled draw.
template <class W>
__device__ int warp_find_crossing(int n, float base, float target, W weight, float* before) {
  const int lane = threadIdx.x & 31;
  const int seg = (n + 31) / 32;
  const int lo = min(n, lane * seg), hi = min(n, lo + seg);
  float mine = 0.f;
  for (int i = lo; i < hi; ++i) mine += weight(i);
  const float incl = warp_incl_scan_f(mine);
  const float excl = incl - mine;
  const unsigned cross = __ballot_sync(0xffffffffu, base + incl > target && mine > 0.f);
  int found = -1;
  float cum = base + excl;
  int owner;
  if (cross) {
    owner = __ffs(cross) - 1;
    if (lane == owner) {
      for (int i = lo; i < hi; ++i) {
        const float w = weight(i);
        if (cum + w > target && w > 0.f) { found = i; break; }
        cum += w;
      }
      if (found < 0) {  // the crossing was lost to rounding inside the segment
        float c2 = base + excl;
        for (int i = lo; i < hi; ++i) {
          const float w = weight(i);
          if (w > 0.f) { found = i; cum = c2; }
          c2 += w;
        }
      }
    }
  } else {
    const unsigned nz = __ballot_sync(0xffffffffu, mine > 0.f);
    owner = nz ? 31 - __clz(nz) : 0;
    if (lane == owner) {
      float c2 = base + excl;
      for (int i = lo; i < hi; ++i) {
        const float w = weight(i);
        if (w > 0.f) { found = i; cum = c2; }
        c2 += w;
      }
      if (found < 0) { found = lo; cum = base + excl; }
    }
  }
  found = __shfl_sync(0xffffffffu, found, owner);
  *before = __shfl_sync(0xffffffffu, cum, owner);
  return max(found, 0);
}

// Block-wide (NT threads) version for long lists: items are split into
// contiguous per-thread segments, the segment sums are scanned across the
// block, and the owning thread walks its segment.  Same contract as
// warp_find_crossing; every thread gets the result.
struct BlockFindScratch {
  float warp_tot[32];
  float before;
  int owner_first, owner_last, found;
};
template <int NT, class W>
__device__ int block_find_crossing(int n, float base, float target, W weight, float* before, BlockFindScratch& sc) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (n + NT - 1) / NT;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  float mine = 0.f;
  for (int i = lo; i < hi; ++i) mine += weight(i);
  const float wincl = warp_incl_scan_f(mine);
  if (tid == 0) { sc.owner_first = 0x7fffffff; sc.owner_last = -1; }
  if (lane == 31) sc.warp_tot[wid] = wincl;
  __syncthreads();
  if (wid == 0) {
    float t = lane < NT / 32 ? sc.warp_tot[lane] : 0.f;
    t = warp_incl_scan_f(t);
    if (lane < NT / 32) sc.warp_tot[lane] = t;
  }
  __syncthreads();
  const float excl = (wincl - mine) + (wid > 0 ? sc.warp_tot[wid - 1] : 0.f);
  if (mine > 0.f) {
    if (base + excl + mine > target) atomicMin(&sc.owner_first, tid);
    atomicMax(&sc.owner_last, tid);
  }
  __syncthreads();
  const bool crossed = sc.owner_first != 0x7fffffff;
  const int owner = crossed ? sc.owner_first : (sc.owner_last >= 0 ? sc.owner_last : 0);
  if (tid == owner) {
    int found = -1;
    float cum = base + excl;
    if (crossed) {
      for (int i = lo; i < hi; ++i) {
        const float w = weight(i);
        if (cum + w > target && w > 0.f) { found = i; break; }
        cum += w;
      }
    }
    if (found < 0) {  // no crossing (rounding): the last positive weight of the segment
      float c2 = base + excl;
      cum = c2;
      for (int i = lo; i < hi; ++i) {
        const float w = weight(i);
        if (w > 0.f) { found = i; cum = c2; }
        c2 += w;
      }
      if (found < 0) found = lo < n ? lo : 0;
    }
    sc.found = found;
    sc.before = cum;
  }
  __syncthreads();
  *before = sc.before;
  const int f = sc.found;
  __syncthreads();
  return f;
}

__device__ __forceinline__ float block_max_f(float v, float* s_red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  if (lane == 0) s_red[wid] = v;
  __syncthreads();
  float r = lane < nw ? s_red[lane] : -INFINITY;
  r = warp_max(r);
  __syncthreads();
  return r;
}
__device__ __forceinline__ float block_sum_f(float v, float* s_red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  if (lane == 0) s_red[wid] = v;
  __syncthreads();
  float r = lane < nw ? s_red[lane] : 0.f;
  r = warp_sum(r);
  __syncthreads();
  return r;
}


}  // namespace dspark
