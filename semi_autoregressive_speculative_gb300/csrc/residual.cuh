// Tensor-core residual pass of verify (included by verify.cu only): for up to
// 128 rows per M-tile — the rejected positions, or, when the analytic
// acceptance c* is wanted, every verify row that has a draft position — each
// with the previous token x_i of its position,
// the draft bias row W1[x_i] . W2 ("DSpark" §2.3, B = W1 W2) is re-formed 64
// vocabulary columns at a time by a tcgen05 UMMA (M = 128 rows, N = 64,
// K = rank, bf16 x bf16 -> fp32 in tensor memory) and reduced on the fly —
// logits never reach HBM:
//
//   p_d = exp2(y - log2 Z_d) with y = (bias + U) * log2(e)/T,
//   p_t = exp2(T_row * log2(e)/T - M_t) / Z_t,   w = max(0, p_t - p_d),
//   per 32-column sub-tile and per CTA chunk: sum of w.
//
// Summed over the vocabulary, w gives 1 - c* for that row ("DSpark" §3.1,
// eq. c_k*: sum max(0, p_t - p_d) = 1/2 ||p_d - p_t||_1).
//
// One CTA per (contiguous V-chunk, M-tile), 10 warps.  The number of rows is
// decided on the device (rejections, or the verify lengths), so the launch
// has at least one CTA per SM and the split of the vocabulary into chunks is
// taken on the device from the actual row count (residual_chunks); the
// kernels that read the partials take the same split.
//   warp 0     producer: W2 tiles by TMA (MN-major, 128B-swizzled) into a
//              kStages-deep ring freed by the UMMA, and the gathered U rows by
//              tile::gather4 loads (four rows per instruction: the TMA unit's
//              issue rate, not HBM, bounds per-row copies) into a second ring
//              freed by the epilogue;
//   warp 1     allocates tensor memory and issues the UMMAs (one thread);
//   warps 2-9  gather W1[x_i] into tensor memory as the A operand (one row per
//              lane), then run the epilogue, two warps per tensor-memory lane
//              quarter (one per 32-column half).
// Every wait is bounded.
#pragma once

#include <cuda.h>

#include "common.h"
#include "device.cuh"
#include "vocab_common.h"

namespace dspark {

constexpr int kStages = 3;  // W2 tiles and U rows in flight per CTA

struct ResidualArgs {
  const float* U;          // [R, gamma, V]
  const uint16_t* W1;      // [V, rank]
  const uint16_t* W2;      // [rank, V]
  const int32_t* anchors;  // [R]
  const int32_t* tokens;   // [R, gamma]
  const float* T;          // [R, gamma+1, V]
  const int32_t* rej;      // [R_pad + 1]: rejected requests; rej[R_pad] = their number
  const int32_t* n_acc;    // [R] rejected position of each request
  const int32_t* rowoff;   // [R+1] verify row offsets; non-null: one row per verify row with a draft position
  const float4* trow;      // [R*(gamma+1)] (max, Z) of each target row, base-2 units
  const float* logZd;      // [R, gamma] draft log-normaliser (natural log)
  float2* coarse;          // [row][residual_chunks(rows)]: x = sum of w over the chunk
  float2* fine;            // [2 * n_tiles][R_pad]: x = sum of w over the 32-column sub-tile, rejected
                           // rows only (column = rejection slot, or request when rowoff is set)
  int32_t* status;
  int R, R_pad, gamma, V, rank;
  int n_tiles;
  int grid;                // CTAs launched
  float scale;             // log2(e) / T
};

// Vocabulary chunks per M-tile for `rows` residual rows and `grid` CTAs: as
// many as keep every CTA busy, at most one 64-column tile each.
__host__ __device__ inline int residual_chunks(int rows, int grid, int n_tiles) {
  const int mt = rows > 0 ? (rows + kMTile - 1) / kMTile : 1;
  int c = grid / mt;
  if (c < 1) c = 1;
  if (c > n_tiles) c = n_tiles;
  if (c > kMaxChunks) c = kMaxChunks;
  return c;
}

// Ring stages by arithmetic (w0 + s * wstride): a runtime-indexed array of
// offsets would live in local memory.
constexpr int kResURow = kTileN * 4;  // bytes per gathered U row in a stage (four rows per gather4)
struct ResidualSmem {
  uint32_t w0, wstride, u0, half, bars, rows, total;
  __host__ __device__ uint32_t w(int s) const { return w0 + static_cast<uint32_t>(s) * wstride; }
  __host__ __device__ uint32_t u(int s) const { return u0 + static_cast<uint32_t>(s) * (kMTile * kResURow); }
};
__host__ __device__ inline ResidualSmem residual_smem_plan(int rank) {
  ResidualSmem s;
  uint32_t off = 0;
  s.w0 = off; s.wstride = 128u * rank; off += kStages * s.wstride;  // rank x 64 bf16, MN-major SW128
  s.u0 = off; off += kStages * kMTile * kResURow;                     // 128 rows x 64 fp32 (1024-aligned)
  s.half = off; off += kMTile * 8;   // second-half chunk partials
  s.bars = off; off += 256;          // mbarriers, tmem slot, abort flag
  s.rows = off; off += kMTile * 16;  // residual rows: token, request, position, fine column
  s.total = off + 1024;              // alignment slack
  return s;
}

__global__ void __launch_bounds__(kDraftThreads, 1)
    k_residual_partials(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u,
                        const ResidualArgs p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const ResidualSmem plan = residual_smem_plan(p.rank);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  const int nrows = p.rowoff != nullptr ? p.rowoff[p.R] : p.rej[p.R_pad];
  const int n_mt = (nrows + kMTile - 1) / kMTile;
  const int n_chunks = residual_chunks(nrows, p.grid, p.n_tiles);
  if (static_cast<int>(blockIdx.x) >= n_mt * n_chunks) return;  // no work for this CTA
  const int mtile = blockIdx.x % n_mt;
  const int chunk = blockIdx.x / n_mt;
  // the rows are spread evenly over the M-tiles (a CTA's time grows with its
  // live rows), M-tile k holding rows [k * rpt, (k + 1) * rpt)
  const int rpt = (nrows + n_mt - 1) / n_mt;
  const int r0 = mtile * rpt;
  const int rows_valid = min(rpt, nrows - r0);
  const int t_begin = static_cast<int>((static_cast<long long>(chunk) * p.n_tiles) / n_chunks);
  const int t_end = static_cast<int>((static_cast<long long>(chunk + 1) * p.n_tiles) / n_chunks);
  const int ntile = t_end - t_begin;

  const uint32_t bar_wfull = base + plan.bars;         // [kStages]
  const uint32_t bar_wempty = bar_wfull + 8 * kStages; // [kStages]
  const uint32_t bar_ufull = bar_wempty + 8 * kStages; // [kStages]
  const uint32_t bar_uempty = bar_ufull + 8 * kStages; // [kStages]
  const uint32_t bar_tfull = bar_uempty + 8 * kStages; // [2]
  const uint32_t bar_tempty = bar_tfull + 16;          // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + plan.bars + 32 * kStages + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + plan.bars + 32 * kStages + 36);
  int4* s_rows = reinterpret_cast<int4*>(gbase + plan.rows);  // (token, request, position, fine column)
  float2* s_half = reinterpret_cast<float2*>(gbase + plan.half);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_wfull + 8 * s, 1);
      mbar_init(bar_wempty + 8 * s, 1);
      mbar_init(bar_ufull + 8 * s, 1);
      mbar_init(bar_uempty + 8 * s, 8);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_tfull + 8 * s, 1);
      mbar_init(bar_tempty + 8 * s, 8);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tm_w2);
    prefetch_tensormap(&tm_u);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // residual rows: previous token, request, position, fine-partials column
  // (-1: none); a row with token -1 is idle (a bonus row j == gamma, which has
  // no draft distribution, or past the last row)
  if (threadIdx.x < kMTile) {
    const int m = threadIdx.x;
    int4 row = make_int4(-1, 0, 0, -1);
    if (m < rows_valid) {
      int req, n, fcol;
      if (p.rowoff != nullptr) {
        const int gi = r0 + m;
        int lo = 0, hi = p.R - 1;  // the request owning verify row gi
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (p.rowoff[mid] <= gi) lo = mid; else hi = mid - 1;
        }
        req = lo;
        n = gi - p.rowoff[req];
        const int len = p.rowoff[req + 1] - p.rowoff[req] - 1;
        fcol = (n == p.n_acc[req] && n < len) ? req : -1;
      } else {
        req = p.rej[r0 + m];
        n = p.n_acc[req];
        fcol = r0 + m;
      }
      if (n < p.gamma) {
        int tok = n == 0 ? p.anchors[req] : p.tokens[static_cast<size_t>(req) * p.gamma + n - 1];
        if (tok < 0 || tok >= p.V) {
          report(p.status, DSPARK_STATUS_BAD_TOKEN);
          tok = 0;
        }
        row = make_int4(tok, req, n, fcol);
      }
    }
    s_rows[m] = row;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tmem_a = tmem_base + kAccCols;  // A operand columns
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // waits by lane 0, decisions broadcast: the warp stays converged
    const uint64_t pol_w = policy_evict_last();
    const uint64_t pol_u = policy_evict_first();
    const uint32_t wbytes = 128u * p.rank;
    int filled = 0;
    for (int i = 0; i < ntile; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      const int v0 = (t_begin + i) * kTileN;
      bool ok = lane == 0 ? mbar_wait(bar_wempty + 8 * s, ph ^ 1, abort_flag) : true;
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        *abort_flag = 1;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_wfull + 8 * s, wbytes);
        tma_load_2d(base + plan.w(s), &tm_w2, bar_wfull + 8 * s, v0, 0, pol_w);
      }
      ok = lane == 0 ? mbar_wait(bar_uempty + 8 * s, ph ^ 1, abort_flag) : true;
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        *abort_flag = 1;
        break;
      }
      // rows 4g .. 4g+3 by lane g (idle rows read U row 0; the box counts in
      // full, columns past V zero-filled)
      const int ngroups = (rows_valid + 3) >> 2;
      if (lane == 0) mbar_arrive_expect_tx(bar_ufull + 8 * s, static_cast<uint32_t>(ngroups) * 4u * kResURow);
      __syncwarp();
      if (lane < ngroups) {
        int rc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int m = 4 * lane + k;
          const int4 row = m < rows_valid ? s_rows[m] : make_int4(-1, 0, 0, -1);
          rc[k] = row.x >= 0 ? row.y * p.gamma + row.z : 0;
        }
        tma_gather4(base + plan.u(s) + lane * 4 * kResURow, &tm_u, bar_ufull + 8 * s, v0, rc[0], rc[1], rc[2], rc[3],
                    pol_u);
      }
      __syncwarp();
      ++filled;
    }
    if (*abort_flag && lane == 0) {
      // let copies already in flight land before the CTA exits
      for (int i = max(0, filled - kStages); i < filled; ++i) {
        const uint32_t s = i % kStages, ph = (i / kStages) & 1;
        const uint64_t t0 = global_ns();
        while (!(mbar_try_wait(bar_wfull + 8 * s, ph) && mbar_try_wait(bar_ufull + 8 * s, ph)) &&
               global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- UMMA issuer
    named_barrier(2, kDraftThreads - 32);  // A operand in tensor memory
    tc_fence_after_sync();
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kMTile, kTileN, false, true);
      const int ksteps = p.rank / 16;
      int issued = 0;
      for (int i = 0; i < ntile; ++i) {
        const int s = i % kStages, acc = i & 1;
        if (!mbar_wait(bar_wfull + 8 * s, (i / kStages) & 1, abort_flag) ||
            !mbar_wait(bar_tempty + 8 * acc, ((i >> 1) & 1) ^ 1, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kTileN);
        for (int ks = 0; ks < ksteps; ++ks) {
          const uint32_t b_addr = base + plan.w(s) + ks * 2048;
          umma_bf16_ts(d, tmem_a + ks * 8, smem_desc_sw128(b_addr, 1024, 1024), idesc, ks > 0 ? 1u : 0u);
        }
        umma_commit(bar_wempty + 8 * s);
        umma_commit(bar_tfull + 8 * acc);
        ++issued;
      }
      if (*abort_flag && issued > 0) {
        const int i = issued - 1;
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(bar_tfull + 8 * (i & 1), (i >> 1) & 1) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue warps 2..9
    const int q = warp & 3;         // tensor-memory lane quarter of this warp
    const int h = (warp - 2) >> 2;  // 32-column half of each tile; half of A's columns
    const int row = q * 32 + lane;
    const int r = r0 + row;
    const bool valid = s_rows[row].x >= 0;
    const int fcol = s_rows[row].w;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;

    // A operand: W1[x_row] into tensor memory, K elements [h*rank/2, (h+1)*rank/2)
    const int tok = s_rows[row].x;
    {
      const int half_cols = p.rank / 4;  // 32-bit columns per half (2 bf16 each)
      const uint4* src = reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(tok < 0 ? 0 : tok) * p.rank) +
                         h * (p.rank / 16);
      for (int c0 = 0; c0 < half_cols; c0 += 32) {
        uint32_t a[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint4 w = make_uint4(0, 0, 0, 0);
          if (tok >= 0 && c0 + 4 * k < half_cols) w = __ldg(src + c0 / 4 + k);
          a[4 * k] = w.x; a[4 * k + 1] = w.y; a[4 * k + 2] = w.z; a[4 * k + 3] = w.w;
        }
        const uint32_t dst = tmem_a + lane_off + static_cast<uint32_t>(h * half_cols + c0);
        if (c0 + 32 <= half_cols) {
          tmem_st_32x32(dst, a);
        } else {
          tmem_st_32x16(dst, a);  // the 16-column remainder (rank 64 or 192)
        }
      }
      tmem_wait_st();
    }
    tc_fence_before_sync();
    named_barrier(2, kDraftThreads - 32);

    const float* trow_ptr = nullptr;
    float mt = 0.f, inv_zt = 0.f, l2zd = 0.f;
    if (valid) {
      const int4 rr = s_rows[row];
      const size_t tr = static_cast<size_t>(rr.y) * (p.gamma + 1) + rr.z;
      trow_ptr = p.T + tr * p.V;
      const float4 st = p.trow[tr];
      mt = st.x;
      inv_zt = 1.0f / st.y;
      l2zd = p.logZd[static_cast<size_t>(rr.y) * p.gamma + rr.z] * 1.4426950408889634f;
    }
    float runS = 0.f;  // running sum of w over this warp's half of the chunk
    // a warp with no live row in its lane quarter only keeps the rings moving
    const bool warp_works = __any_sync(0xffffffffu, valid);
    // this row's 32 target values of the next tile, loaded one tile ahead
    float tn[32];
    auto load_t = [&](int i) {
      const int v0 = (t_begin + i) * kTileN + h * kSubN;
      const int ncol = min(kSubN, p.V - v0);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid && 4 * k < ncol) t4 = __ldg(reinterpret_cast<const float4*>(trow_ptr + v0) + k);
        tn[4 * k] = t4.x; tn[4 * k + 1] = t4.y; tn[4 * k + 2] = t4.z; tn[4 * k + 3] = t4.w;
      }
    };
    if (warp_works && ntile > 0) load_t(0);
    for (int i = 0; i < ntile; ++i) {
      const int s = i % kStages, acc = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8 * acc, (i >> 1) & 1, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      if (!warp_works) {
        if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
        if (!__all_sync(0xffffffffu, mbar_wait(bar_ufull + 8 * s, (i / kStages) & 1, abort_flag))) {
          *abort_flag = 1;
          break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_uempty + 8 * s);
        continue;
      }
      tc_fence_after_sync();
      float v[32];
      tmem_ld_32x32(tmem_base + lane_off + static_cast<uint32_t>(acc * kTileN + h * kSubN), v);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
      if (!__all_sync(0xffffffffu, mbar_wait(bar_ufull + 8 * s, (i / kStages) & 1, abort_flag))) {
        *abort_flag = 1;
        break;
      }
      float u[32];
      const float4* urow = reinterpret_cast<const float4*>(gbase + plan.u(s) + row * kResURow + h * 128);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 t4 = urow[k];
        u[4 * k] = t4.x; u[4 * k + 1] = t4.y; u[4 * k + 2] = t4.z; u[4 * k + 3] = t4.w;
      }
      // the stage is refilled by bulk copies (async proxy) once released: order
      // these generic-proxy reads before that write
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_uempty + 8 * s);

      const int v0 = (t_begin + i) * kTileN + h * kSubN;
      const int ncol = min(kSubN, p.V - v0);  // <= 0 for a fully masked last half
      const size_t fidx = static_cast<size_t>(2 * (t_begin + i) + h) * p.R_pad + fcol;
      float tv[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) tv[k] = tn[k];
      if (i + 1 < ntile) load_t(i + 1);
      float sw = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float pd = ex2((v[k] + u[k]) * p.scale - l2zd);
        const float pt = ex2(tv[k] * p.scale - mt) * inv_zt;
        sw += (k < ncol) ? fmaxf(pt - pd, 0.f) : 0.f;
      }
      if (valid && fcol >= 0) p.fine[fidx] = make_float2(sw, 0.f);
      runS += sw;
    }
    // combine the two column halves of this CTA's chunk
    if (h == 1) s_half[row] = make_float2(0.f, runS);
    named_barrier(1, 256);
    if (h == 0 && valid) p.coarse[static_cast<size_t>(r) * n_chunks + chunk] = make_float2(runS + s_half[row].y, 0.f);
  }
  if (*abort_flag && threadIdx.x == 0) report(p.status, DSPARK_STATUS_TIMEOUT);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace dspark
