// Hardware-aware prefix scheduler ("DSpark" §4.1-4.3; "投机解码的新做法" page,
// section "按负载决定验证多少").  One CTA of 1024 threads, everything in
// shared memory, no host round trip:
//   1. keys (a descending, j ascending, r ascending) packed into 64 bits and
//      bitonic-sorted in registers (E keys per thread): partners inside a
//      warp by shuffles, partners in the same thread in registers, partners
//      in other warps through a double-buffered shared array (one CTA
//      barrier per such pass);
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

// One bitonic compare-exchange seen from index i: keep the smaller key when i
// is the lower index of an ascending pair (or the upper of a descending one).
__device__ __forceinline__ uint64_t bitonic_keep(uint64_t x, uint64_t y, int i, int jj, int k) {
  const bool keep_min = ((i & jj) == 0) == ((i & k) == 0);
  return keep_min ? (x < y ? x : y) : (x < y ? y : x);
}

// A pass whose partner index is m ^ MJ in the same thread (MJ fixed at compile
// time, so that the keys stay in registers).
template <int E, int MJ>
__device__ __forceinline__ void bitonic_in_thread(uint64_t (&x)[E], int t, int jj, int k) {
#pragma unroll
  for (int m = 0; m < E; ++m) {
    if ((m ^ MJ) > m && (m ^ MJ) < E) {
      const int m2 = m ^ MJ;
      const uint64_t lo = x[m], hi = x[m2];
      x[m] = bitonic_keep(lo, hi, t + kSchedThreads * m, jj, k);
      x[m2] = bitonic_keep(hi, lo, t + kSchedThreads * m2, jj, k);
    }
  }
}

// Ascending bitonic sort of b0[0, 1024 E); b1 is scratch of the same size.
// Thread t holds indices t + 1024 m, m < E, so a warp owns 32 consecutive
// indices of every block of 1024: partners closer than 32 are exchanged by
// shuffles, partners 1024 apart or more sit in the same thread, and the rest
// go through shared memory (one CTA barrier per pass, the two buffers taking
// turns).  On return b0 holds the sorted keys.  (Measured: 8 consecutive keys
// per thread on fewer warps was slower; the network is latency-bound.)
template <int E>
__device__ void sort_keys(uint64_t* b0, uint64_t* b1) {
  constexpr int n = kSchedThreads * E;
  const int t = threadIdx.x;
  uint64_t x[E];
#pragma unroll
  for (int m = 0; m < E; ++m) x[m] = b0[t + kSchedThreads * m];
  __syncthreads();  // every key is read before the first exchange rewrites b0
  int xp = 0;       // exchanges through shared memory so far (buffer parity)
  for (int k = 2; k <= n; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      if (jj < 32) {
#pragma unroll
        for (int m = 0; m < E; ++m) {
          const uint64_t y = __shfl_xor_sync(0xffffffffu, x[m], jj);
          x[m] = bitonic_keep(x[m], y, t + kSchedThreads * m, jj, k);
        }
      } else if (jj >= kSchedThreads) {
        const int mj = jj / kSchedThreads;  // partner m ^ mj in this thread: 1, 2 or 4
        if (mj == 1) bitonic_in_thread<E, 1>(x, t, jj, k);
        else if (mj == 2) bitonic_in_thread<E, 2>(x, t, jj, k);
        else bitonic_in_thread<E, 4>(x, t, jj, k);
      } else {
        uint64_t* buf = (xp & 1) ? b1 : b0;
#pragma unroll
        for (int m = 0; m < E; ++m) buf[t + kSchedThreads * m] = x[m];
        __syncthreads();
#pragma unroll
        for (int m = 0; m < E; ++m) {
          const int i = t + kSchedThreads * m;
          x[m] = bitonic_keep(x[m], buf[i ^ jj], i, jj, k);
        }
        ++xp;
      }
    }
  }
  __syncthreads();  // the last shared-memory exchange is read everywhere
#pragma unroll
  for (int m = 0; m < E; ++m) b0[t + kSchedThreads * m] = x[m];
  __syncthreads();
}

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
  // 2. bitonic sort, ascending (npow2 = 1024 E, E <= 8: the host pads to 1024);
  // the prefix-sum array is the exchange scratch
  {
    uint64_t* scratch = reinterpret_cast<uint64_t*>(S);
    switch (npow2 / kSchedThreads) {
      case 1: sort_keys<1>(keys, scratch); break;
      case 2: sort_keys<2>(keys, scratch); break;
      case 4: sort_keys<4>(keys, scratch); break;
      default: sort_keys<8>(keys, scratch); break;
    }
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
  int npow2 = kSchedThreads;  // at least one key per thread
  while (npow2 < R * gamma) npow2 <<= 1;
  static_assert(kMaxSchedule <= 8 * kSchedThreads, "the register sort holds at most 8 keys per thread");
  const SchedSmem plan = sched_smem_plan(npow2, R);
  if (cudaFuncSetAttribute(k3_schedule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sched_smem_plan(kMaxSchedule, kMaxSchedule).total)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  const cudaError_t e = launch_pdl(k3_schedule, dim3(1), dim3(kSchedThreads), plan.total, stream, true, a, R, gamma,
                                   sps, mode, budget_K, lens, total_b, argmax_b, theta, status, npow2);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark
