// Hardware-aware prefix scheduler ("DSpark" §4.1-4.3; "投机解码的新做法" page,
// section "按负载决定验证多少").  One CTA of 1024 threads, everything in
// shared memory, no host round trip:
//   1. keys (a descending, j ascending, r ascending) packed into 64 bits and
//      sorted.  Survival products never rise along a request (each step
//      multiplies by a confidence <= 1, and fp32 rounding is monotone), so
//      each request's keys already form a sorted run and the order is a merge
//      of R runs: ceil(log2 R) levels, each a merge path (one diagonal search
//      per thread, then a sequential merge of its keys).  The keys are
//      distinct, so this is exactly the sorted order.  Rows that do rise (a
//      caller's own a, or values reported as non-finite) take the general
//      path: a stable radix sort of the keys written in (j, r) order on their
//      upper 32 bits (four 8-bit passes);
//   2. a -> Q.40 fixed point (an exact integer rounding) and an integer
//      inclusive scan: S_b is the same for every summation order;
//   3. Theta(b) = (R + S_b 2^-40) * SPS[R + b] in fp64 for every b (the sum
//      built exactly from integer bits when it fits 53 bits);
//   4. b* by mode (first descent / min(K, n) / n) and the global argmax;
//   5. lens[r] = admitted pairs of request r.
#include <cmath>

#include "common.h"
#include "device.cuh"

namespace dspark {

constexpr int kSchedThreads = 1024;

constexpr int kRadixDigits = 256;  // 8-bit digits, four passes over the upper 32 key bits
constexpr int kSchedWarps = kSchedThreads / 32;
// SPS entries that fit in the radix counts' shared memory (staged by cp.async)
constexpr int kSpsStaged = (kSchedWarps + 8) * kRadixDigits * 4 / 8;

// Stable LSD radix sort of b0[0, 1024 E) by key bits 32..63, ascending; b1 is
// scratch of the same size and hist holds (32 + 8) x 256 ints.  Thread t =
// 32 w + lane handles elements 32 E w + 32 m + lane, m < E (the keys stay in
// shared memory), so that within a warp the order (slot, lane) is the element
// order and the per-slot ranks from __match_any_sync are stable.  Per pass: each warp counts its digits
// (hist[w][d]), the counts are scanned in (digit, warp) order, and each key
// goes to its digit's base + the keys of that digit in earlier warps + its
// rank in the warp.  On return b0 holds the sorted keys.
template <int E>
__device__ __noinline__ void radix_sort_keys(uint64_t* b0, uint64_t* b1, int* hist) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned below = (1u << lane) - 1u;
  int* gsum = hist + kSchedWarps * kRadixDigits;  // [4][256]: counts of warps 8g .. 8g+7
  int* gbase = gsum + 4 * kRadixDigits;           // [4][256]: first position of (digit, warp group)
  uint64_t* src = b0;
  uint64_t* dst = b1;
  for (int pass = 0; pass < 4; ++pass) {
    const int sh = 32 + 8 * pass;
    for (int i = t; i < kSchedWarps * kRadixDigits; i += kSchedThreads) hist[i] = 0;
    __syncthreads();
    int rd[E];  // rank in the warp << 8 | digit
#pragma unroll
    for (int m = 0; m < E; ++m) {
      const int d = static_cast<int>((src[32 * E * w + 32 * m + lane] >> sh) & 0xFFu);
      const unsigned peers = __match_any_sync(0xffffffffu, d);
      const int before = hist[w * kRadixDigits + d];  // this digit in the warp's earlier slots
      __syncwarp();
      if ((peers & below) == 0) hist[w * kRadixDigits + d] = before + __popc(peers);
      __syncwarp();
      rd[m] = ((before + __popc(peers & below)) << 8) | d;
    }
    __syncthreads();
    {  // exclusive counts over the warps of each group of 8, per digit
      const int d = t & (kRadixDigits - 1), g = t >> 8;
      int run = 0;
      for (int ww = 8 * g; ww < 8 * g + 8; ++ww) {
        const int c = hist[ww * kRadixDigits + d];
        hist[ww * kRadixDigits + d] = run;
        run += c;
      }
      gsum[g * kRadixDigits + d] = run;
    }
    __syncthreads();
    if (w == 0) {  // digit bases (exclusive over digits), then each (digit, group) start
      int tot[8];
      int sum = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int d = 8 * lane + k;
        tot[k] = gsum[d] + gsum[kRadixDigits + d] + gsum[2 * kRadixDigits + d] + gsum[3 * kRadixDigits + d];
        sum += tot[k];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int base = incl - sum;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int d = 8 * lane + k;
        int gb = base;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          gbase[g * kRadixDigits + d] = gb;
          gb += gsum[g * kRadixDigits + d];
        }
        base += tot[k];
      }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < E; ++m) {
      const int d = rd[m] & 0xFF;
      dst[gbase[(w >> 3) * kRadixDigits + d] + hist[w * kRadixDigits + d] + (rd[m] >> 8)] =
          src[32 * E * w + 32 * m + lane];
    }
    __syncthreads();
    uint64_t* const tmp = src;
    src = dst;
    dst = tmp;
  }
  // four passes: the last one wrote b0
}

// Sorts a[0, n) (distinct keys) whose runs [k run, (k + 1) run) are each
// ascending, by merging adjacent runs level by level; b is scratch of the same
// size.  On return a holds the sorted keys.  At every level thread t writes
// the merged keys [E t, E t + E) (merge path): one binary search along the
// diagonal finds how many of the first d keys of its merged run come from the
// left run, then the thread merges its E keys in turn.
__device__ void merge_sorted_runs(uint64_t* a, uint64_t* b, int n, int run, int E) {
  uint64_t* src = a;
  uint64_t* dst = b;
  for (int L = run; L < n; L <<= 1) {
    const int L2 = 2 * L;
    int o = threadIdx.x * E;
    const int oend = min(o + E, n);
    while (o < oend) {
      const int lo = (o / L2) * L2;
      const int mid = min(lo + L, n), hi = min(lo + L2, n);
      const int la = mid - lo, lb = hi - mid, d = o - lo;
      // the smallest m with A[m] > B[d - m - 1]: keys of A among the first d
      int x0 = max(0, d - lb), x1 = min(d, la);
      while (x0 < x1) {
        const int m = (x0 + x1) >> 1;
        if (src[lo + m] < src[mid + d - m - 1]) x0 = m + 1;
        else x1 = m;
      }
      int ia = x0, ib = d - x0;
      const int stop = min(oend, hi);
      for (; o < stop; ++o) {
        const bool take_a = ia < la && (ib >= lb || src[lo + ia] < src[mid + ib]);
        dst[o] = take_a ? src[lo + ia++] : src[mid + ib++];
      }
    }
    __syncthreads();
    uint64_t* const tmp = src;
    src = dst;
    dst = tmp;
  }
  if (src != a) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) a[i] = src[i];
    __syncthreads();
  }
}

__device__ __forceinline__ void cp_async_8(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// round(v 2^40) to nearest, ties to even, for finite v >= 0, in integer
// arithmetic (exactly the fp64 product rounded to int64: v 2^40 needs no more
// than 24 significant bits); saturates at 2^63 - 1 from v >= 2^23 on.
__device__ __forceinline__ int64_t q40(float v) {
  const uint32_t bits = __float_as_uint(v);
  const int e = static_cast<int>(bits >> 23);
  if (e == 0) return 0;  // zero or subnormal: below 2^-86
  const uint64_t mant = (bits & 0x7FFFFFu) | 0x800000u;  // v = mant 2^(e - 150)
  const int sh = e - 110;                                 // v 2^40 = mant 2^sh
  if (sh >= 0) return sh >= 40 ? INT64_MAX : static_cast<int64_t>(mant << sh);
  const int s = -sh;
  if (s > 24) return 0;  // below 1/2
  const uint64_t q = mant >> s, rem = mant & ((1ull << s) - 1), half = 1ull << (s - 1);
  return static_cast<int64_t>(q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0));
}

// R + S 2^-40 in fp64, exactly, for S >= 0 and R 2^40 + S < 2^53: the sum
// needs no rounding, so its double is built from the integer's bits (the fp64
// pipe of GB300 is slow).
__device__ __forceinline__ double tau_exact(int R, int64_t S) {
  const int64_t T = (static_cast<int64_t>(R) << 40) + S;
  const int p = 63 - __clzll(T);  // 40 <= p <= 52 (R >= 1)
  const uint64_t bits = (static_cast<uint64_t>(p - 40 + 1023) << 52) |
                        ((static_cast<uint64_t>(T) << (52 - p)) & ((1ull << 52) - 1));
  return __longlong_as_double(static_cast<long long>(bits));
}

struct SchedSmem {
  uint32_t keys, S, rid, cnt, hist, total;
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
  s.hist = off; off += 4u * (kSchedWarps + 8) * kRadixDigits;  // radix counts and bases
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
  int* hist = reinterpret_cast<int*>(sm + plan.hist);
  double* th = reinterpret_cast<double*>(sm + plan.keys);
  __shared__ int s_red_b[32];
  __shared__ unsigned long long s_red_t[32];
  __shared__ int64_t s_warp[32];

  pdl_launch_dependents();
  pdl_wait();
  const int n = R * gamma;
  const int tid = threadIdx.x;
  // 1. keys, in (r, j) order: each request's run.  NaN, negative or infinite
  // a is scheduled last (as 0) and reported; -0 is 0.
  auto clean = [](float v) -> uint32_t {
    return (!(v >= 0.f) || !(v <= 3.4e38f) || v == 0.f) ? 0u : __float_as_uint(v);
  };
  int rises = 0;  // some request's a rises along its positions
  for (int i = tid; i < npow2; i += kSchedThreads) {
    uint64_t key = ~0ull;
    if (i < n) {
      const float v = a[i];
      if (!(v >= 0.f) || !(v <= 3.4e38f)) report(status, DSPARK_STATUS_NONFINITE);
      const uint32_t bits = clean(v);
      const int r = i / gamma, j = i - r * gamma;
      if (j > 0 && clean(a[i - 1]) < bits) rises = 1;
      key = (static_cast<uint64_t>(0xFFFFFFFFu - bits) << 32) | (static_cast<uint64_t>(j) << 16) |
            static_cast<uint64_t>(r);
    }
    keys[i] = key;
  }
  for (int r = tid; r < R; r += kSchedThreads) cnt[r] = 0;
  rises = __syncthreads_or(rises);
  // 2. sort, ascending key; the prefix-sum array is the scratch buffer
  {
    uint64_t* scratch = reinterpret_cast<uint64_t*>(S);
    if (!rises) {
      merge_sorted_runs(keys, scratch, n, gamma, npow2 / kSchedThreads);
      // the SPS entries of step 4 go to shared memory now, asynchronously, so
      // that their latency hides behind steps 3 and the scan: into the radix
      // counts' space, which the merge leaves unused (when they fit; otherwise
      // step 4 reads them itself)
      if (n + 1 <= kSpsStaged) {
        for (int b = tid; b <= n; b += kSchedThreads) cp_async_8(reinterpret_cast<double*>(hist) + b, sps + R + b);
        cp_async_commit();
      }
    } else {
      // the keys in (j, r) order, the low key bits ascending, so that a stable
      // sort by the upper 32 bits is the full 64-bit order (npow2 = 1024 E,
      // E <= 8: the host pads to 1024; the padding keys stay at the end)
      for (int i = tid; i < n; i += kSchedThreads) scratch[i] = keys[i];
      __syncthreads();
      for (int i = tid; i < n; i += kSchedThreads) {
        const int r = i / gamma, j = i - r * gamma;
        keys[j * R + r] = scratch[i];
      }
      __syncthreads();
      switch (npow2 / kSchedThreads) {
        case 1: radix_sort_keys<1>(keys, scratch, hist); break;
        case 2: radix_sort_keys<2>(keys, scratch, hist); break;
        case 4: radix_sort_keys<4>(keys, scratch, hist); break;
        default: radix_sort_keys<8>(keys, scratch, hist); break;
      }
    }
  }
  // 3. fixed-point values and request ids in sorted order; S[0] = 0
  for (int i = tid; i < n; i += kSchedThreads) {
    const uint64_t key = keys[i];
    const float v = __uint_as_float(0xFFFFFFFFu - static_cast<uint32_t>(key >> 32));
    S[i + 1] = q40(v);
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
  const bool staged = !rises && n + 1 <= kSpsStaged;  // SPS(R + b) in shared memory
  if (staged) cp_async_wait_all();
  __syncthreads();
  // 4. Theta(b) (overwrites the key storage; rid keeps what is still needed)
  // S_b never falls as b grows (Q.40 values are >= 0; a sum that overflowed
  // is negative), so S_n decides for every b whether tau is exact
  if (S[n] >= 0 && (static_cast<int64_t>(R) << 40) + S[n] < (1ll << 53)) {
    for (int b = tid; b <= n; b += kSchedThreads)
      th[b] = __dmul_rn(tau_exact(R, S[b]), staged ? reinterpret_cast<const double*>(hist)[b] : sps[R + b]);
  } else {
    for (int b = tid; b <= n; b += kSchedThreads)
      th[b] = __dmul_rn(__dadd_rn(static_cast<double>(R), static_cast<double>(S[b]) * 0x1p-40), sps[R + b]);
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
