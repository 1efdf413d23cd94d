// Hardware-aware prefix scheduler ("DSpark" §4.1-4.3; "投机解码的新做法" page,
// section "按负载决定验证多少").  One CTA of 1024 threads, everything in
// shared memory, no host round trip:
//   1. keys (a descending, j ascending, r ascending) packed into 64 bits and
//      bitonic-sorted (warp barriers for the passes inside a warp);
//   2. a -> Q.40 fixed point and an integer inclusive scan: S_b is the same for
//      every summation order;
//   3. Theta(b) = (R + S_b 2^-40) * SPS[R + b] in fp64 for every b;
//   4. b* by mode (first descent / min(K, n) / n) and the global argmax;
//   5. lens[r] = admitted pairs of request r.
#include <cmath>

#include "common.h"
#include "device.cuh"

namespace dspark {

constexpr int kSchedThreads = 1024;

struct SchedSmem {
  uint32_t keys, S, rid, cnt, total;
};
__host__ __device__ inline SchedSmem sched_smem_plan(int npow2, int R) {
  SchedSmem s;
  uint32_t off = 0;
  s.keys = off; off += 8u * (npow2 + 1);   // sorted keys, later Theta(b) (fp64, n + 1 entries)
  s.S = off;    off += 8u * (npow2 + 1);   // Q.40 prefix sums S_0..S_n
  s.rid = off;  off += 2u * npow2;         // request of each sorted entry
  off = (off + 15u) & ~15u;
  s.cnt = off;  off += 4u * R;             // per-request admitted counts
  off = (off + 15u) & ~15u;
  s.total = off + 64;                      // + reduction scratch
  return s;
}

__global__ void __launch_bounds__(kSchedThreads)
    k3_schedule(const float* __restrict__ a, int R, int gamma, const double* __restrict__ sps, int mode, int budget_K,
                int32_t* __restrict__ lens, int32_t* __restrict__ total_b, int32_t* __restrict__ argmax_b,
                double* __restrict__ theta, int32_t* status, int npow2) {
  extern __shared__ __align__(16) uint8_t sm[];
  const SchedSmem plan = sched_smem_plan(npow2, R);
  uint64_t* keys = reinterpret_cast<uint64_t*>(sm + plan.keys);
  int64_t* S = reinterpret_cast<int64_t*>(sm + plan.S);
  uint16_t* rid = reinterpret_cast<uint16_t*>(sm + plan.rid);
  int32_t* cnt = reinterpret_cast<int32_t*>(sm + plan.cnt);
  double* th = reinterpret_cast<double*>(sm + plan.keys);
  __shared__ int s_red_b[32];
  __shared__ unsigned long long s_red_t[32];
  __shared__ int64_t s_warp[32];

  pdl_launch_dependents();
  pdl_wait();
  const int n = R * gamma;
  const int tid = threadIdx.x;
  // 1. keys
  for (int i = tid; i < npow2; i += kSchedThreads) {
    uint64_t key = ~0ull;
    if (i < n) {
      float v = a[i];
      if (!(v >= 0.f) || !(v <= 3.4e38f)) {  // NaN, negative or infinite: schedule it last
        report(status, DSPARK_STATUS_NONFINITE);
        v = 0.f;
      }
      const uint32_t bits = __float_as_uint(v);
      const int r = i / gamma, j = i - r * gamma;
      key = (static_cast<uint64_t>(0xFFFFFFFFu - bits) << 32) | (static_cast<uint64_t>(j) << 16) |
            static_cast<uint64_t>(r);
    }
    keys[i] = key;
  }
  for (int r = tid; r < R; r += kSchedThreads) cnt[r] = 0;
  __syncthreads();
  // 2. bitonic sort, ascending.  Thread t handles indices t + 1024 m, so a warp
  // owns 32 consecutive indices of every block of 1024: passes whose partner
  // distance is below 32 stay inside the warp and need only a warp barrier;
  // the CTA barrier follows the wider passes and each merge size.
  for (int k = 2; k <= npow2; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = tid; i < npow2; i += kSchedThreads) {
        const int ixj = i ^ jj;
        if (ixj > i) {
          const uint64_t x = keys[i], y = keys[ixj];
          const bool up = (i & k) == 0;
          if ((x > y) == up) { keys[i] = y; keys[ixj] = x; }
        }
      }
      if (jj >= 32) __syncthreads(); else __syncwarp();
    }
    // merges up to 32 wide never leave a warp; the next, wider one reads across warps
    if (k >= 32) __syncthreads(); else __syncwarp();
  }
  // 3. fixed-point values and request ids in sorted order; S[0] = 0
  for (int i = tid; i < n; i += kSchedThreads) {
    const uint64_t key = keys[i];
    const float v = __uint_as_float(0xFFFFFFFFu - static_cast<uint32_t>(key >> 32));
    S[i + 1] = __double2ll_rn(static_cast<double>(v) * 0x1p40);
    rid[i] = static_cast<uint16_t>(key & 0xFFFFu);
  }
  if (tid == 0) S[0] = 0;
  __syncthreads();
  // inclusive scan of S[1..n]: each thread owns a contiguous run
  {
    const int per = (n + kSchedThreads - 1) / kSchedThreads;
    const int lo = 1 + tid * per, hi = min(n + 1, lo + per);
    int64_t run = 0;
    for (int i = lo; i < hi; ++i) { run += S[i]; S[i] = run; }
    // exclusive scan of the per-thread totals
    const int lane = tid & 31, wid = tid >> 5;
    int64_t x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int64_t w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int64_t offset = (x - run) + (wid > 0 ? s_warp[wid - 1] : 0);
    for (int i = lo; i < hi; ++i) S[i] += offset;
  }
  __syncthreads();
  // 4. Theta(b) (overwrites the key storage; rid keeps what is still needed)
  for (int b = tid; b <= n; b += kSchedThreads) {
    const double tau = __dadd_rn(static_cast<double>(R), static_cast<double>(S[b]) * 0x1p-40);
    th[b] = __dmul_rn(tau, sps[R + b]);
  }
  __syncthreads();
  // first descent (early stop) and global argmax (lowest b on ties).  The
  // comparisons use an order-preserving integer image of each fp64 Theta
  // (the fp64 pipe of GB300 is slow; the integer compare is exact).
  auto key = [&](int b) -> unsigned long long {
    const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(th[b]));
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
  };
  int my_stop = n;
  unsigned long long my_best = 0ull;
  int my_arg = 0x7fffffff;
  for (int b = tid; b <= n; b += kSchedThreads) {
    const unsigned long long kb = key(b);
    if (b < n && key(b + 1) <= kb && b < my_stop) my_stop = b;
    if (kb > my_best || (kb == my_best && b < my_arg)) { my_best = kb; my_arg = b; }
  }
  {
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      my_stop = min(my_stop, __shfl_xor_sync(0xffffffffu, my_stop, o));
      const unsigned long long ob = __shfl_xor_sync(0xffffffffu, my_best, o);
      const int oa = __shfl_xor_sync(0xffffffffu, my_arg, o);
      if (ob > my_best || (ob == my_best && oa < my_arg)) { my_best = ob; my_arg = oa; }
    }
    if (lane == 0) { s_red_b[wid] = my_stop; s_red_t[wid] = my_best; s_warp[wid] = my_arg; }
    __syncthreads();
    if (wid == 0) {
      my_stop = s_red_b[lane];
      my_best = s_red_t[lane];
      my_arg = static_cast<int>(s_warp[lane]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        my_stop = min(my_stop, __shfl_xor_sync(0xffffffffu, my_stop, o));
        const unsigned long long ob = __shfl_xor_sync(0xffffffffu, my_best, o);
        const int oa = __shfl_xor_sync(0xffffffffu, my_arg, o);
        if (ob > my_best || (ob == my_best && oa < my_arg)) { my_best = ob; my_arg = oa; }
      }
      if (lane == 0) { s_red_b[0] = my_stop; s_warp[0] = my_arg; }
    }
    __syncthreads();
  }
  int bstar;
  if (mode == DSPARK_MODE_EARLY_STOP) bstar = s_red_b[0];
  else if (mode == DSPARK_MODE_TOP_K) bstar = budget_K < 0 ? 0 : (budget_K > n ? n : budget_K);
  else bstar = n;
  // 5. per-request lengths
  for (int i = tid; i < bstar; i += kSchedThreads) atomicAdd(&cnt[rid[i]], 1);
  __syncthreads();
  for (int r = tid; r < R; r += kSchedThreads) lens[r] = cnt[r];
  if (tid == 0) {
    *total_b = bstar;
    *argmax_b = static_cast<int>(s_warp[0]);
    *theta = th[bstar];
  }
}

int launch_schedule(const float* a, int R, int gamma, const double* sps, int mode, int budget_K, int32_t* lens,
                    int32_t* total_b, int32_t* argmax_b, double* theta, int32_t* status, cudaStream_t stream) {
  int npow2 = 1;
  while (npow2 < R * gamma) npow2 <<= 1;
  const SchedSmem plan = sched_smem_plan(npow2, R);
  if (cudaFuncSetAttribute(k3_schedule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sched_smem_plan(kMaxSchedule, kMaxSchedule).total)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  const cudaError_t e = launch_pdl(k3_schedule, dim3(1), dim3(kSchedThreads), plan.total, stream, true, a, R, gamma,
                                   sps, mode, budget_K, lens, total_b, argmax_b, theta, status, npow2);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark
