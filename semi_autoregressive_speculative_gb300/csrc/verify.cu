// Rejection-sampling verification (standard speculative verification:
// "DSpark" introduction and §2.2; "DSpark: Speculative decodingを活用した…",
// "問題定義").  Only rows 0..lens[r] of each request are read.
//
//  k4_prepare       one CTA: verify-row offsets (exclusive scan of lens + 1),
//                   clears the rejection list.
//  k4_target_stats  one warp per (verify row, 1024-column chunk; row owners from a
//                   shared-memory copy of the row offsets): softmax
//                   partials of T / temperature (or max / argmax), and the
//                   target logit at the drafted token.
//  k4_accept        one CTA per request: per row max and normaliser, the
//                   accept tests u < p_t(x) / p_d(x) of all positions at once
//                   (the first rejection is the lowest rejected position), the
//                   bonus draw from row lens[r] when everything is accepted,
//                   otherwise the request joins the rejection list.
//  k_residual_partials  tensor-core recompute of the draft rows at the
//                   rejected positions fused with max(0, p_t - p_d) partial sums.
//  k4_residual_sample  one CTA per rejected request: inverse CDF of the
//                   residual (or of p_t when its mass is zero).
//
// Optional output: the analytic acceptance c*_j = 1 - 1/2 ||p_d - p_t||_1
// ("DSpark" §3.1, eq. c_k*) of every verify row j <= lens[r] that has a draft
// position (j < gamma).  Then the residual pass covers all those rows instead
// of the rejected ones only, k4_c_star sums each row's partials, and the
// rejection sampler reads its rows' partials from the same pass.  Greedy: the
// two distributions are point masses and k4_accept writes c* = [x_j == argmax].
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.h"
#include "device.cuh"
#include "search.cuh"
#include "residual.cuh"
#include "vocab_common.h"

namespace dspark {

struct VerifyArgs {
  const float* T;          // [R, gamma+1, V]
  const float* U;          // [R, gamma, V]
  const uint16_t* W1;
  const uint16_t* W2;
  const int32_t* anchors;
  const int32_t* tokens;   // [R, gamma]
  const float* pd_tok;     // [R, gamma]
  const float* logZd;      // [R, gamma]
  const int32_t* lens;     // [R]
  int32_t* n_accept;       // [R]
  int32_t* next_token;     // [R]
  float* c_star;           // [R, gamma] or null
  float2* tstats;          // [R*(gamma+1)][n_vc]
  float4* trow;            // [R*(gamma+1)]: (max, Z, t(x), -) base-2 units
  int32_t* rowoff;         // [R+1]
  int32_t* rej;            // [R_pad + 1]
  const float2* coarse;    // residual partials [row][residual_chunks(rows, res_grid, n_tiles)]
  const float2* fine;      // [2*n_tiles][R_pad]
  int32_t* status;
  int R, R_pad, gamma, V, rank, n_vc, n_tiles;
  int res_grid;            // CTAs of the residual pass
  float scale;             // log2(e) / T (1 when greedy)
  int greedy;
  int all_rows;            // residual partials cover every verify row with a draft position
  uint64_t seed;
  uint32_t round;
};

__device__ __forceinline__ int clamp_len(int l, int gamma, int32_t* status) {
  if (l < 0 || l > gamma) {
    report(status, DSPARK_STATUS_BAD_LENGTH);
    return l < 0 ? 0 : gamma;
  }
  return l;
}

__global__ void __launch_bounds__(1024) k4_prepare(const VerifyArgs p) {
  __shared__ int32_t s_warp[32];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (p.R + 1023) / 1024;
  const int lo = tid * per, hi = min(p.R, lo + per);
  int run = 0;
  for (int r = lo; r < hi; ++r) run += clamp_len(p.lens[r], p.gamma, p.status) + 1;
  int x = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  int off = (x - run) + (wid > 0 ? s_warp[wid - 1] : 0);
  for (int r = lo; r < hi; ++r) {
    p.rowoff[r] = off;
    off += clamp_len(p.lens[r], p.gamma, nullptr) + 1;
  }
  if (tid == 1023) p.rowoff[p.R] = s_warp[31];
  if (tid == 0) p.rej[p.R_pad] = 0;
}

__global__ void __launch_bounds__(256) k4_target_stats(const VerifyArgs p) {
  extern __shared__ int32_t s_rowoff[];  // [R + 1]
  pdl_launch_dependents();
  pdl_wait();
  for (int i = threadIdx.x; i <= p.R; i += blockDim.x) s_rowoff[i] = p.rowoff[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int nw = gridDim.x * 8;
  const int rows = s_rowoff[p.R];
  const long long items = static_cast<long long>(rows) * p.n_vc;
  for (long long it = gw; it < items; it += nw) {
    const int gi = static_cast<int>(it / p.n_vc);
    const int c = static_cast<int>(it - static_cast<long long>(gi) * p.n_vc);
    // request owning verify row gi: the last r with rowoff[r] <= gi (shared-memory copy)
    int lo = 0, hi = p.R - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_rowoff[mid] <= gi) lo = mid; else hi = mid - 1;
    }
    const int r = lo, j = gi - s_rowoff[r];
    const size_t trw = static_cast<size_t>(r) * (p.gamma + 1) + j;
    const float* row = p.T + trw * p.V;
    const int c0 = c * kVerifyChunk;
    const int ncol = min(kVerifyChunk, p.V - c0);
    constexpr int kPer = kVerifyChunk / 32;  // values per lane (16-byte loads, all in flight)
    float t[kPer];
#pragma unroll
    for (int k = 0; k < kPer / 4; ++k) {
      const int col = (k * 32 + lane) * 4;
      float4 v = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (col < ncol) v = __ldcs(reinterpret_cast<const float4*>(row + c0 + col));
      t[4 * k] = v.x; t[4 * k + 1] = v.y; t[4 * k + 2] = v.z; t[4 * k + 3] = v.w;
    }
    float2 res;
    if (p.greedy) {
      float mx = -INFINITY;
      int ix = 0x7fffffff;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int col = c0 + (k >> 2) * 128 + lane * 4 + (k & 3);
        if (t[k] > mx || (t[k] == mx && col < ix)) { mx = t[k]; ix = col; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
        if (om > mx || (om == mx && oi < ix)) { mx = om; ix = oi; }
      }
      res = make_float2(mx, __int_as_float(ix));
    } else {
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < kPer; ++k) { t[k] *= p.scale; mx = fmaxf(mx, t[k]); }
      mx = warp_max(mx);
      float s = 0.f;
      if (mx > -INFINITY) {
#pragma unroll
        for (int k = 0; k < kPer; ++k) s += ex2(t[k] - mx);
      }
      s = warp_sum(s);
      res = make_float2(mx, s);
    }
    if (lane == 0) {
      p.tstats[trw * p.n_vc + c] = res;
      if (j < p.gamma) {
        const int x = p.tokens[static_cast<size_t>(r) * p.gamma + j];
        if (x >= c0 && x < c0 + ncol) p.trow[trw].z = row[x];
      }
    }
  }
}

// row max / normaliser from the chunk partials (base-2 units)
__device__ __forceinline__ void row_stats(const float2* st, int n_vc, float* M_out, float* Z_out) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, z = 0.f;  // online (max, sum) per lane, then merged across the warp
  for (int c = lane; c < n_vc; c += 32) {
    const float2 e = st[c];
    if (e.x > -INFINITY) {
      if (e.x > m) {
        z = (m > -INFINITY ? z * exp2f(m - e.x) : 0.f) + e.y;
        m = e.x;
      } else {
        z += e.y * exp2f(e.x - m);
      }
    }
  }
  const float M = warp_max(m);
  *M_out = M;
  *Z_out = warp_sum(m > -INFINITY ? z * exp2f(m - M) : 0.f);
}
__device__ __forceinline__ int row_argmax(const float2* st, int n_vc) {
  const int lane = threadIdx.x & 31;
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  for (int c = lane; c < n_vc; c += 32) {
    const float2 e = st[c];
    const int ei = __float_as_int(e.y);
    if (e.x > best || (e.x == best && ei < bidx)) { best = e.x; bidx = ei; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
  }
  return bidx;
}

// Inverse CDF of softmax(T_row * scale) with target u * Z, via the chunk
// partials and a scan of the selected kVerifyChunk-column chunk.
// Block-wide (256 threads); every thread gets the result.
__device__ int sample_target_row(const VerifyArgs& p, size_t trw, float M, float Z, float u, BlockFindScratch& sc) {
  const float2* st = p.tstats + trw * p.n_vc;
  const float target = u * Z;
  float before = 0.f;
  const int c = block_find_crossing<256>(
      p.n_vc, 0.f, target,
      [&](int i) -> float { const float2 e = st[i]; return e.x > -INFINITY ? e.y * exp2f(e.x - M) : 0.f; }, &before,
      sc);
  const float* row = p.T + trw * p.V;
  const int c0 = c * kVerifyChunk;
  const int ncol = min(kVerifyChunk, p.V - c0);
  float b2 = 0.f;
  const int i = block_find_crossing<256>(
      ncol, before, target, [&](int k) -> float { return exp2f(row[c0 + k] * p.scale - M); }, &b2, sc);
  return c0 + i;
}

// One CTA per request: warp w computes the statistics of rows w, w+8, ...;
// then thread j runs the accept test of position j (all at once: the tests
// are independent, and the first rejection is the lowest rejected j).
__global__ void __launch_bounds__(256) k4_accept(const VerifyArgs p) {
  __shared__ BlockFindScratch sc;
  __shared__ float s_M[kMaxGamma + 1], s_Z[kMaxGamma + 1], s_tz[kMaxGamma + 1];
  __shared__ int s_am[kMaxGamma + 1];
  __shared__ unsigned s_rej[2];  // rejected positions 0..31 and 32..63
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int r = blockIdx.x;
  const int len = clamp_len(p.lens[r], p.gamma, nullptr);
  const size_t base_row = static_cast<size_t>(r) * (p.gamma + 1);
  // the accept test's own inputs (thread j < len: position j), read and drawn
  // before the row statistics
  int tok = 0;
  float pd = 0.f, u = 0.f;
  if (tid < len) {
    tok = p.tokens[static_cast<size_t>(r) * p.gamma + tid];
    if (!p.greedy) {
      pd = p.pd_tok[static_cast<size_t>(r) * p.gamma + tid];
      u = uniform24(p.seed, p.round, static_cast<uint64_t>(r), static_cast<uint64_t>(tid), kAcceptTest);
    }
  }
  for (int j = wid; j <= len; j += 8) {
    const float2* st = p.tstats + (base_row + j) * p.n_vc;
    if (p.greedy) {
      const int am = row_argmax(st, p.n_vc);
      if (lane == 0) s_am[j] = am;
    } else {
      float M, Z;
      row_stats(st, p.n_vc, &M, &Z);
      if (lane == 0) {
        const float tz = p.trow[base_row + j].z;
        s_M[j] = M;
        s_Z[j] = Z;
        s_tz[j] = tz;
        p.trow[base_row + j] = make_float4(M, Z, tz, 0.f);
      }
    }
  }
  __syncthreads();
  bool rejected = false, nonfinite = false;
  if (tid < len) {
    if (p.greedy) {
      rejected = tok != s_am[tid];
    } else {
      const float M = s_M[tid], Z = s_Z[tid];
      if (!(fabsf(M) <= 3.4e38f) || !(Z > 0.f) || !(Z <= 3.4e38f)) {
        rejected = nonfinite = true;
      } else {
        const float pt = exp2f(s_tz[tid] * p.scale - M) / Z;
        // accept iff u < p_t / p_d, evaluated as u * p_d < p_t (p_d > 0)
        rejected = !(!(pd > 0.f) || u * pd < pt);
      }
    }
  }
  const unsigned rej_bits = __ballot_sync(0xffffffffu, rejected);
  if (wid < 2 && lane == 0) s_rej[wid] = rej_bits;
  __syncthreads();
  const int n = s_rej[0] ? __ffs(s_rej[0]) - 1 : s_rej[1] ? 32 + __ffs(s_rej[1]) - 1 : len;
  if (tid == n && nonfinite) report(p.status, DSPARK_STATUS_NONFINITE);  // the first rejection's row
  if (tid == 0) p.n_accept[r] = n;
  if (p.greedy) {
    if (tid == 0) {
      const int nxt = s_am[n];
      p.next_token[r] = (nxt >= 0 && nxt < p.V) ? nxt : 0;
    }
    if (p.c_star != nullptr) {
      for (int j = tid; j < p.gamma; j += 256) {
        const float cs = j <= len ? (p.tokens[static_cast<size_t>(r) * p.gamma + j] == s_am[j] ? 1.f : 0.f)
                                  : __int_as_float(0x7fc00000);  // NaN: no target row read
        p.c_star[static_cast<size_t>(r) * p.gamma + j] = cs;
      }
    }
    return;
  }
  if (n == len) {
    const float M = s_M[n], Z = s_Z[n];
    if (!(fabsf(M) <= 3.4e38f) || !(Z > 0.f) || !(Z <= 3.4e38f)) {
      if (tid == 0) {
        report(p.status, DSPARK_STATUS_NONFINITE);
        p.next_token[r] = 0;
      }
      return;
    }
    const float u2 = uniform24(p.seed, p.round, static_cast<uint64_t>(r), static_cast<uint64_t>(n), kResidualOrBonus);
    const int x = sample_target_row(p, base_row + n, M, Z, u2, sc);
    if (tid == 0) p.next_token[r] = min(x, p.V - 1);
  } else if (tid == 0) {
    const int slot = atomicAdd(&p.rej[p.R_pad], 1);
    p.rej[slot] = r;
  }
}

__global__ void __launch_bounds__(256) k4_residual_sample(const __grid_constant__ CUtensorMap tm_slab,
                                                          const VerifyArgs p) {
  __shared__ BlockFindScratch sc;
  __shared__ float s_redz[32];
  __shared__ float s_e[256];
  __shared__ float s_part[8][32];
  __shared__ __align__(128) uint16_t s_slab[256 * kSubN];  // W2 columns of the chosen sub-tile, [rank][32]
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_landed;
  __shared__ volatile int s_no_abort;  // the slab wait's abort word: never set
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const uint32_t bar = smem_u32(&s_bar);
  if (tid == 0) {
    s_no_abort = 0;
    mbar_init(bar, 1);
    fence_barrier_init();
    prefetch_tensormap(&tm_slab);
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x;
  if (i >= p.rej[p.R_pad]) return;
  const int r = p.rej[i];
  const int n = p.n_accept[r];
  const size_t trw = static_cast<size_t>(r) * (p.gamma + 1) + n;
  const float4 ts = p.trow[trw];
  const float Mt = ts.x;
  const float Zt = ts.y;
  const float u2 = uniform24(p.seed, p.round, static_cast<uint64_t>(r), static_cast<uint64_t>(n), kResidualOrBonus);
  // partials of this row: by rejection slot, or (all verify rows covered) by
  // verify row for the chunk sums and by request for the sub-tile sums
  const int prow = p.all_rows ? p.rowoff[r] + n : i;
  const int fcol = p.all_rows ? r : i;
  const int n_chunks = residual_chunks(p.all_rows ? p.rowoff[p.R] : p.rej[p.R_pad], p.res_grid, p.n_tiles);
  const float2* crow = p.coarse + static_cast<size_t>(prow) * n_chunks;
  float zl = 0.f;
  for (int c = tid; c < n_chunks; c += 256) zl += crow[c].x;
  const float Zr = block_sum_f(zl, s_redz);
  if (!(Zr > 0.f) || !(Zr <= 3.4e38f)) {
    // zero residual mass: draw from p_t
    const int x = sample_target_row(p, trw, Mt, Zt, u2, sc);
    if (tid == 0) p.next_token[r] = min(max(x, 0), p.V - 1);
    return;
  }
  const float target = u2 * Zr;
  float before_c = 0.f;
  const int cstar = block_find_crossing<256>(
      n_chunks, 0.f, target, [&](int c) -> float { return crow[c].x; }, &before_c, sc);
  const int tb = static_cast<int>((static_cast<long long>(cstar) * p.n_tiles) / n_chunks);
  const int te = static_cast<int>((static_cast<long long>(cstar + 1) * p.n_tiles) / n_chunks);
  const float2* frow = p.fine + fcol;
  float before_s = 0.f;
  const int sstar = 2 * tb + block_find_crossing<256>(
                                 2 * (te - tb), before_c, target,
                                 [&](int k) -> float { return frow[static_cast<size_t>(2 * tb + k) * p.R_pad].x; },
                                 &before_s, sc);
  // recompute the 32 residual weights of that sub-tile: the W2 columns come in
  // as one TMA box (rank x 32), each warp sums 32 rank rows for lane = column
  const int v0 = sstar * kSubN;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(p.rank) * kSubN * 2u);
    tma_load_2d(smem_u32(s_slab), &tm_slab, bar, v0, 0, policy_evict_normal());
  }
  const int prev_raw = n == 0 ? p.anchors[r] : p.tokens[static_cast<size_t>(r) * p.gamma + n - 1];
  const int prev = (prev_raw >= 0 && prev_raw < p.V) ? prev_raw : 0;
  for (int k = tid; k < p.rank; k += 256) s_e[k] = bf16_at(p.W1 + static_cast<size_t>(prev) * p.rank + k);
  // the sub-tile's U and T values, read while the slab is in flight
  const int v = v0 + lane;
  float u_v = 0.f, t_v = 0.f;
  if (wid == 0 && v < p.V) {
    u_v = p.U[(static_cast<size_t>(r) * p.gamma + n) * p.V + v];
    t_v = p.T[trw * p.V + v];
  }
  if (tid == 0) s_landed = mbar_wait(bar, 0, &s_no_abort) ? 1 : 0;  // bounded; one waiter, result shared
  __syncthreads();
  float acc = 0.f;
  if (s_landed) {
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const int j = wid * 32 + k;
      if (j < p.rank) acc = fmaf(s_e[j], __uint_as_float(static_cast<uint32_t>(s_slab[j * kSubN + lane]) << 16), acc);
    }
  } else if (tid == 0) {
    report(p.status, DSPARK_STATUS_TIMEOUT);
  }
  s_part[wid][lane] = acc;
  __syncthreads();
  if (wid == 0) {
    float w = 0.f;
    if (v < p.V) {
      float b = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) b += s_part[k][lane];
      const float l2zd = p.logZd[static_cast<size_t>(r) * p.gamma + n] * 1.4426950408889634f;
      const float pd = exp2f((b + u_v) * p.scale - l2zd);
      const float pt = exp2f(t_v * p.scale - Mt) / Zt;
      w = fmaxf(pt - pd, 0.f);
    }
    const float incl = before_s + warp_incl_scan_f(w);
    const unsigned cross = __ballot_sync(0xffffffffu, incl > target && w > 0.f);
    int pick;
    if (cross) {
      pick = __ffs(cross) - 1;
    } else {
      const unsigned nz = __ballot_sync(0xffffffffu, w > 0.f);
      pick = nz ? 31 - __clz(nz) : 0;
    }
    if (lane == 0) p.next_token[r] = min(max(v0 + pick, 0), p.V - 1);
  }
}

// c*_{r,j} = 1 - sum over the vocabulary of max(0, p_t - p_d), from the chunk
// partials of verify row rowoff[r] + j; one warp per (r, j), a fixed summation
// order; NaN for positions past the rows verify read.
__global__ void __launch_bounds__(256) k4_c_star(const VerifyArgs p) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (gw >= p.R * p.gamma) return;
  const int r = gw / p.gamma, j = gw - r * p.gamma;
  const int len = clamp_len(p.lens[r], p.gamma, nullptr);
  float cs = __int_as_float(0x7fc00000);
  if (j <= len) {
    const int n_chunks = residual_chunks(p.rowoff[p.R], p.res_grid, p.n_tiles);
    const float2* crow = p.coarse + static_cast<size_t>(p.rowoff[r] + j) * n_chunks;
    float s = 0.f;
    for (int c = lane; c < n_chunks; c += 32) s += crow[c].x;
    cs = 1.f - warp_sum(s);
  }
  if (lane == 0) p.c_star[gw] = cs;
}

// The residual pass of verify, chained to the accept kernel with programmatic
// dependent launch.
static cudaError_t launch_residual_partials(const CUtensorMap& tm_w2, const CUtensorMap& tm_u, const ResidualArgs& a,
                                            cudaStream_t stream) {
  const ResidualSmem plan = residual_smem_plan(a.rank);
  const dim3 grid(a.grid);
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(k_residual_partials, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(residual_smem_plan(256).total));
  });
  return launch_pdl(k_residual_partials, grid, dim3(kDraftThreads), plan.total, stream, true, tm_w2, tm_u, a);
}

int launch_verify(const float* T, const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* anchors,
                  const int32_t* tokens, const float* pd_tok, const float* logZ, const int32_t* lens, int R, int gamma,
                  int V, int rank, float temperature, uint64_t seed, uint32_t round, int32_t* n_accept,
                  int32_t* next_token, float* c_star, void* workspace, cudaStream_t stream) {
  const WorkspaceLayout L = workspace_layout(R, gamma, V);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  VerifyArgs p = {};
  p.T = T; p.U = U; p.W1 = W1; p.W2 = W2; p.anchors = anchors; p.tokens = tokens; p.pd_tok = pd_tok;
  p.logZd = logZ; p.lens = lens; p.n_accept = n_accept; p.next_token = next_token; p.c_star = c_star;
  p.tstats = reinterpret_cast<float2*>(ws + L.tstats);
  p.trow = reinterpret_cast<float4*>(ws + L.trow);
  p.rowoff = reinterpret_cast<int32_t*>(ws + L.rowoff);
  p.rej = reinterpret_cast<int32_t*>(ws + L.rej);
  p.coarse = reinterpret_cast<const float2*>(ws + L.coarse);
  p.fine = reinterpret_cast<const float2*>(ws + L.fine);
  p.status = reinterpret_cast<int32_t*>(ws + L.status);
  p.R = R; p.gamma = gamma; p.V = V; p.rank = rank;
  const int n_mtiles = ceil_div(R, kMTile);
  p.R_pad = n_mtiles * kMTile;
  p.n_vc = ceil_div(V, kVerifyChunk);
  p.n_tiles = ceil_div(V, kTileN);
  p.greedy = temperature == 0.0f ? 1 : 0;
  // residual rows: the rejected requests (<= R), or every verify row (<= R (gamma + 1))
  p.all_rows = (c_star != nullptr && !p.greedy) ? 1 : 0;
  // one CTA per SM at least, one per M-tile of the most rows there can be
  const int res_mtiles = p.all_rows ? ceil_div(R * (gamma + 1), kMTile) : n_mtiles;
  p.res_grid = std::max(sm_count(), res_mtiles);
  // the chunk partials of every residual row (at most 128 x max(grid, M-tiles)
  // entries) must fit the workspace's partials region
  if (static_cast<size_t>(p.res_grid) * kMTile > static_cast<size_t>(kMaxChunks) * p.R_pad)
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  p.scale = p.greedy ? 1.0f : static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  p.seed = seed; p.round = round;

  if (launch_pdl(k4_prepare, dim3(1), dim3(1024), 0, stream, true, p) != cudaSuccess) return DSPARK_ERR_CUDA;
  const long long max_items = static_cast<long long>(R) * (gamma + 1) * p.n_vc;
  long long blocks = (max_items + 7) / 8;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const size_t rowoff_bytes = (static_cast<size_t>(R) + 1) * sizeof(int32_t);
  if (rowoff_bytes > 48 * 1024 &&
      cudaFuncSetAttribute(k4_target_stats, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(rowoff_bytes)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (launch_pdl(k4_target_stats, dim3(static_cast<unsigned>(blocks)), dim3(256), rowoff_bytes, stream, true, p) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (launch_pdl(k4_accept, dim3(R), dim3(256), 0, stream, true, p) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (p.greedy) return DSPARK_OK;

  ResidualArgs a = {};
  a.U = U; a.W1 = W1; a.W2 = W2; a.anchors = anchors; a.tokens = tokens;
  a.T = T; a.rej = p.rej; a.n_acc = n_accept; a.trow = p.trow; a.logZd = logZ;
  a.rowoff = p.all_rows ? p.rowoff : nullptr;
  a.coarse = reinterpret_cast<float2*>(ws + L.coarse);
  a.fine = reinterpret_cast<float2*>(ws + L.fine);
  a.status = p.status;
  a.R = R; a.R_pad = p.R_pad; a.gamma = gamma; a.V = V; a.rank = rank;
  a.n_tiles = p.n_tiles; a.grid = p.res_grid;
  a.scale = p.scale;
  CUtensorMap tm_w2, tm_u;
  if (encode_w2_map(&tm_w2, W2, V, rank) != DSPARK_OK || encode_u_rows_map(&tm_u, U, R, gamma, V) != DSPARK_OK)
    return DSPARK_ERR_CUDA;
  if (launch_residual_partials(tm_w2, tm_u, a, stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (p.all_rows &&
      launch_pdl(k4_c_star, dim3(ceil_div(R * gamma, 8)), dim3(256), 0, stream, true, p) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  CUtensorMap tm_slab;
  if (encode_w2_slab_map(&tm_slab, W2, V, rank) != DSPARK_OK) return DSPARK_ERR_CUDA;
  if (launch_pdl(k4_residual_sample, dim3(R), dim3(256), 0, stream, true, tm_slab, p) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

}  // namespace dspark
