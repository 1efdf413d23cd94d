// Tensor-core vocabulary pass shared by the draft and by verify's residual
// step: for a set of up to 128 rows per M-tile, each row i having a previous
// token x_i, the bias row W1[x_i] . W2 ("DSpark" §2.3, B = W1 W2) is formed
// 64 vocabulary columns at a time by a tcgen05 UMMA (M = 128 rows, N = 64,
// K = rank, bf16 x bf16 -> fp32 in tensor memory) and reduced on the fly —
// logits never reach HBM:
//
//   kDraft    : y = (bias + U) * log2(e)/T; per 32-column sub-tile and per
//               CTA chunk the softmax partial (max y, sum exp2(y - max)), or
//               (max, argmax) when greedy.
//   kResidual : p_d = exp2(y - log2 Z_d), p_t = exp2(T * log2(e)/T - M_t) / Z_t,
//               w = max(0, p_t - p_d); per sub-tile and per chunk sum of w.
//
// One CTA per (contiguous V-chunk, M-tile), 10 warps: warp 0 issues TMA (W2
// tile, MN-major 128B-swizzled) and per-row bulk copies of U; warp 1 gathers
// nothing and issues the UMMAs (one thread); warps 2..9 are the epilogue, two
// per tensor-memory lane quarter (one per 32-column half).  Two smem stages,
// two tensor-memory accumulators.  Every wait is bounded.
#pragma once

#include <cuda.h>

#include "common.h"
#include "device.cuh"

namespace dspark {

enum class VocabMode { kDraft, kResidual };

struct VocabArgs {
  const float* U;          // [R, gamma, V]
  const uint16_t* W1;      // [V, rank]
  const uint16_t* W2;      // [rank, V]
  const int32_t* anchors;  // [R]
  const int32_t* tokens;   // [R, gamma]
  float2* coarse;          // [n_chunks][R_pad]
  float2* fine;            // [2 * n_tiles][R_pad]
  int32_t* status;
  int R, R_pad, gamma, V, rank, step;
  int n_tiles, n_chunks, n_mtiles;
  float scale;             // log2(e) / T  (1 when greedy)
  int greedy;
  // kResidual only
  const float* T;          // [R, gamma+1, V]
  const int32_t* rej;      // [R_pad + 1]: rej[R_pad] = number of residual rows
  const int32_t* n_acc;    // [R] rejected position of each request
  const float4* trow;      // [R*(gamma+1)] (max, Z) of each target row, base-2 units
  const float* logZd;      // [R, gamma] draft log-normaliser (natural log)
};

struct VocabSmem {
  uint32_t a, w[2], u[2], half, bars, rows, total;
};
__host__ __device__ inline VocabSmem vocab_smem_plan(int rank) {
  VocabSmem s;
  uint32_t off = 0;
  s.a = off;    off += 256u * rank;        // 128 rows x rank bf16, K-major SW128
  s.w[0] = off; off += 128u * rank;        // rank x 64 bf16, MN-major SW128
  s.w[1] = off; off += 128u * rank;
  s.u[0] = off; off += kMTile * kUStride;  // 128 rows x 64 fp32 (+16 B per row)
  s.u[1] = off; off += kMTile * kUStride;
  s.half = off; off += kMTile * 8;         // second-half chunk partials
  s.bars = off; off += 128;                // 8 mbarriers, tmem slot, abort flag
  s.rows = off; off += kMTile * 16;        // per row: token, request, position, pad / constants
  s.total = off + 1024;                    // alignment slack
  return s;
}

// A-tile byte offset of (row m, 16-byte chunk c): K-major, 128B swizzle,
// K blocks of 64 elements (16 KB each), 8-row groups of 1024 bytes.
__device__ __forceinline__ uint32_t a_tile_offset(int m, int c) {
  const int kb = c >> 3, cc = c & 7;
  return static_cast<uint32_t>(kb * (kMTile * 128) + m * 128 + ((cc ^ (m & 7)) << 4));
}

template <VocabMode MODE>
__global__ void __launch_bounds__(kDraftThreads, 1)
    k_vocab_partials(const __grid_constant__ CUtensorMap tm_w2, const VocabArgs p) {
  constexpr bool kRes = MODE == VocabMode::kResidual;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const VocabSmem plan = vocab_smem_plan(p.rank);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mtile = blockIdx.x % p.n_mtiles;
  const int chunk = blockIdx.x / p.n_mtiles;
  const int r0 = mtile * kMTile;

  int nrows = p.R;
  if constexpr (kRes) {
    pdl_wait();
    nrows = p.rej[p.R_pad];
    if (r0 >= nrows) return;  // no residual rows for this M-tile
  }
  const int rows_valid = min(kMTile, nrows - r0);
  const int t_begin = static_cast<int>((static_cast<long long>(chunk) * p.n_tiles) / p.n_chunks);
  const int t_end = static_cast<int>((static_cast<long long>(chunk + 1) * p.n_tiles) / p.n_chunks);
  const int ntile = t_end - t_begin;

  const uint32_t bar_full = base + plan.bars;  // [2]
  const uint32_t bar_empty = bar_full + 16;    // [2]
  const uint32_t bar_tfull = bar_full + 32;    // [2]
  const uint32_t bar_tempty = bar_full + 48;   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + plan.bars + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + plan.bars + 68);
  int4* s_rows = reinterpret_cast<int4*>(gbase + plan.rows);  // (token, request, position, -)
  float2* s_half = reinterpret_cast<float2*>(gbase + plan.half);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1 + 8);
      mbar_init(bar_tfull + 8 * s, 1);
      mbar_init(bar_tempty + 8 * s, 8);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tm_w2);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * kTileN);
    tmem_relinquish();
  }
  if constexpr (kRes) {
    // residual rows: request, rejected position, previous token
    if (threadIdx.x < kMTile) {
      const int m = threadIdx.x;
      int4 row = make_int4(-1, 0, 0, 0);
      if (m < rows_valid) {
        const int req = p.rej[r0 + m];
        const int n = p.n_acc[req];
        int tok = n == 0 ? p.anchors[req] : p.tokens[static_cast<size_t>(req) * p.gamma + n - 1];
        if (tok < 0 || tok >= p.V) {
          report(p.status, DSPARK_STATUS_BAD_TOKEN);
          tok = 0;
        }
        row = make_int4(tok, req, n, 0);
      }
      s_rows[m] = row;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    // In the draft, W2 and U are inputs of the round, so their loads may start
    // before the previous kernel in the stream has finished.
    const uint64_t pol_w = policy_evict_last();
    const uint64_t pol_u = policy_evict_first();
    const uint32_t wbytes = 128u * p.rank;
    int filled = 0;
    for (int i = 0; i < ntile; ++i) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag)) {
        *abort_flag = 1;
        break;
      }
      const int v0 = (t_begin + i) * kTileN;
      const int cols = min(kTileN, p.V - v0);
      const uint32_t ubytes = static_cast<uint32_t>(cols) * 4u;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_full + 8 * s, wbytes + ubytes * static_cast<uint32_t>(rows_valid));
        tma_load_2d(base + plan.w[s], &tm_w2, bar_full + 8 * s, v0, 0, pol_w);
      }
      __syncwarp();
      for (int m = lane; m < rows_valid; m += 32) {
        size_t urow;
        if constexpr (kRes) {
          const int4 row = s_rows[m];
          urow = static_cast<size_t>(row.y) * p.gamma + row.z;
        } else {
          urow = static_cast<size_t>(r0 + m) * p.gamma + p.step;
        }
        bulk_load(base + plan.u[s] + m * kUStride, p.U + urow * p.V + v0, ubytes, bar_full + 8 * s, pol_u);
      }
      ++filled;
    }
    if (*abort_flag && lane == 0) {
      // let copies already in flight land before the CTA exits
      for (int i = max(0, filled - 2); i < filled; ++i) {
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(bar_full + 8 * (i & 1), (i >> 1) & 1) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ---------------------------------------------------------- gather W1 rows into the A tile
    if constexpr (!kRes) {
      pdl_wait();  // tokens of the previous position come from the previous kernel
      const int t = threadIdx.x - 32;
      if (t < kMTile) {
        int tok = -1;
        if (t < rows_valid) {
          const int r = r0 + t;
          tok = p.step == 0 ? p.anchors[r] : p.tokens[static_cast<size_t>(r) * p.gamma + p.step - 1];
          if (tok < 0 || tok >= p.V) {
            report(p.status, DSPARK_STATUS_BAD_TOKEN);
            tok = 0;
          }
        }
        s_rows[t] = make_int4(tok, r0 + t, p.step, 0);
      }
      named_barrier(2, kDraftThreads - 32);
    }
    const int tid = threadIdx.x - 32;  // 0..287
    const int cpr = p.rank / 8;        // 16-byte chunks per row
    for (int idx = tid; idx < kMTile * cpr; idx += kDraftThreads - 32) {
      const int m = idx / cpr, c = idx - m * cpr;
      const int tok = s_rows[m].x;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (tok >= 0) val = __ldg(reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(tok) * p.rank) + c);
      *reinterpret_cast<uint4*>(gbase + plan.a + a_tile_offset(m, c)) = val;
    }
    fence_proxy_async_smem();
    named_barrier(2, kDraftThreads - 32);

    if (warp == 1) {
      // -------------------------------------------------------- UMMA issuer
      if (lane == 0) {
        const uint32_t idesc = idesc_bf16_f32(kMTile, kTileN, false, true);
        const int ksteps = p.rank / 16;
        int issued = 0;
        for (int i = 0; i < ntile; ++i) {
          const int s = i & 1, acc = i & 1;
          const uint32_t ph = (i >> 1) & 1;
          if (!mbar_wait(bar_full + 8 * s, ph, abort_flag) || !mbar_wait(bar_tempty + 8 * acc, ph ^ 1, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kTileN);
          for (int ks = 0; ks < ksteps; ++ks) {
            const uint32_t a_addr = base + plan.a + (ks >> 2) * (kMTile * 128) + (ks & 3) * 32;
            const uint32_t b_addr = base + plan.w[s] + ks * 2048;
            umma_bf16(d, smem_desc_sw128(a_addr, 16, 1024), smem_desc_sw128(b_addr, 1024, 1024), idesc,
                      ks > 0 ? 1u : 0u);
          }
          umma_commit(bar_empty + 8 * s);
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
      // -------------------------------------------------------- epilogue (warps 2..9)
      const int q = warp & 3;         // tensor-memory lane quarter of this warp
      const int h = (warp - 2) >> 2;  // 32-column half of each tile
      const int row = q * 32 + lane;
      const int r = r0 + row;
      const bool valid = row < rows_valid;
      // residual-mode row constants
      const float* trow_ptr = nullptr;
      float mt = 0.f, inv_zt = 0.f, l2zd = 0.f;
      if constexpr (kRes) {
        if (valid) {
          const int4 rr = s_rows[row];
          const size_t tr = static_cast<size_t>(rr.y) * (p.gamma + 1) + rr.z;
          trow_ptr = p.T + tr * p.V;
          const float4 st = p.trow[tr];
          mt = st.x;
          inv_zt = 1.0f / st.y;
          l2zd = p.logZd[static_cast<size_t>(rr.y) * p.gamma + rr.z] * 1.4426950408889634f;
        }
      }
      float runM = -INFINITY, runS = 0.f;  // draft: running (max, sum exp2); residual: runS = sum w
      int runIdx = 0;                      // greedy: running argmax
      for (int i = 0; i < ntile; ++i) {
        const int s = i & 1, acc = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait(bar_tfull + 8 * acc, ph, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after_sync();
        float v[32];
        tmem_ld_32x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kTileN + h * kSubN),
                      v);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
        if (!mbar_wait(bar_full + 8 * s, ph, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        const float4* urow = reinterpret_cast<const float4*>(gbase + plan.u[s] + row * kUStride + h * 128);
        float u[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 t4 = urow[k];
          u[4 * k] = t4.x; u[4 * k + 1] = t4.y; u[4 * k + 2] = t4.z; u[4 * k + 3] = t4.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);

        const int v0 = (t_begin + i) * kTileN + h * kSubN;
        const int ncol = min(kSubN, p.V - v0);  // <= 0 for a fully masked last half
        const size_t fidx = static_cast<size_t>(2 * (t_begin + i) + h) * p.R_pad + r;
        if constexpr (kRes) {
          float tv[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (valid && 4 * k < ncol) t4 = __ldg(reinterpret_cast<const float4*>(trow_ptr + v0) + k);
            tv[4 * k] = t4.x; tv[4 * k + 1] = t4.y; tv[4 * k + 2] = t4.z; tv[4 * k + 3] = t4.w;
          }
          float sw = 0.f;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float pd = exp2f((v[k] + u[k]) * p.scale - l2zd);
            const float pt = exp2f(tv[k] * p.scale - mt) * inv_zt;
            sw += (k < ncol) ? fmaxf(pt - pd, 0.f) : 0.f;
          }
          if (valid) p.fine[fidx] = make_float2(sw, 0.f);
          runS += sw;
        } else if (p.greedy) {
          float mx = -INFINITY;
          int ix = v0;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float y = v[k] + u[k];
            if (k < ncol && y > mx) { mx = y; ix = v0 + k; }
          }
          if (valid) p.fine[fidx] = make_float2(mx, __int_as_float(ix));
          if (mx > runM) { runM = mx; runIdx = ix; }
        } else {
          float y[32];
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            y[k] = (v[k] + u[k]) * p.scale;
            if (k < ncol) mx = fmaxf(mx, y[k]);
          }
          float sm = 0.f;
          if (mx > -INFINITY) {
#pragma unroll
            for (int k = 0; k < 32; ++k) sm += (k < ncol) ? exp2f(y[k] - mx) : 0.f;
          }
          if (valid) p.fine[fidx] = make_float2(mx, sm);
          if (mx > -INFINITY) {
            if (mx > runM) {
              runS = (runM > -INFINITY ? runS * exp2f(runM - mx) : 0.f) + sm;
              runM = mx;
            } else {
              runS += sm * exp2f(mx - runM);
            }
          }
        }
      }
      // combine the two column halves of this CTA's chunk
      if (h == 1) s_half[row] = p.greedy ? make_float2(runM, __int_as_float(runIdx)) : make_float2(runM, runS);
      named_barrier(1, 256);
      if (h == 0 && valid) {
        const float2 o = s_half[row];
        float2 outv;
        if constexpr (kRes) {
          outv = make_float2(runS + o.y, 0.f);
        } else if (p.greedy) {
          const int oi = __float_as_int(o.y);
          if (o.x > runM || (o.x == runM && oi < runIdx)) { runM = o.x; runIdx = oi; }
          outv = make_float2(runM, __int_as_float(runIdx));
        } else {
          const float M = fmaxf(runM, o.x);
          float S = 0.f;
          if (M > -INFINITY) {
            if (runM > -INFINITY) S += runS * exp2f(runM - M);
            if (o.x > -INFINITY) S += o.y * exp2f(o.x - M);
          }
          outv = make_float2(M, S);
        }
        p.coarse[static_cast<size_t>(chunk) * p.R_pad + r] = outv;
      }
    }
  }
  if (*abort_flag && threadIdx.x == 0) report(p.status, DSPARK_STATUS_TIMEOUT);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 2 * kTileN);
  }
}

// Segmented search across one warp.  Weights w(i), i in [0, n), are summed
// per lane over contiguous segments; returns the first i whose inclusive
// prefix (starting at `base`) exceeds `target`, or the last i with w(i) > 0
// when rounding leaves the total at or below the target.  *before = the
// prefix just before the returned i.
template <class W>
__device__ int warp_find_crossing(int n, double base, double target, W weight, double* before) {
  const int lane = threadIdx.x & 31;
  const int seg = (n + 31) / 32;
  const int lo = min(n, lane * seg), hi = min(n, lo + seg);
  double mine = 0.0;
  for (int i = lo; i < hi; ++i) mine += static_cast<double>(weight(i));
  const double incl = warp_incl_scan_d(mine);
  const double excl = incl - mine;
  const unsigned cross = __ballot_sync(0xffffffffu, base + incl > target && mine > 0.0);
  int found = -1;
  double cum = base + excl;
  int owner;
  if (cross) {
    owner = __ffs(cross) - 1;
    if (lane == owner) {
      for (int i = lo; i < hi; ++i) {
        const double w = static_cast<double>(weight(i));
        if (cum + w > target && w > 0.0) { found = i; break; }
        cum += w;
      }
      if (found < 0) {  // the crossing was lost to rounding inside the segment
        double c2 = base + excl;
        for (int i = lo; i < hi; ++i) {
          const double w = static_cast<double>(weight(i));
          if (w > 0.0) { found = i; cum = c2; }
          c2 += w;
        }
      }
    }
  } else {
    const unsigned nz = __ballot_sync(0xffffffffu, mine > 0.0);
    owner = nz ? 31 - __clz(nz) : 0;
    if (lane == owner) {
      double c2 = base + excl;
      for (int i = lo; i < hi; ++i) {
        const double w = static_cast<double>(weight(i));
        if (w > 0.0) { found = i; cum = c2; }
        c2 += w;
      }
      if (found < 0) { found = lo; cum = base + excl; }
    }
  }
  found = __shfl_sync(0xffffffffu, found, owner);
  *before = __shfl_sync(0xffffffffu, cum, owner);
  return max(found, 0);
}

// Host: tensor map over W2 and launch of the vocabulary pass.
int encode_w2_map(CUtensorMap* tm, const uint16_t* W2, int V, int rank);
int vocab_chunks(int n_tiles, int n_mtiles);
cudaError_t launch_vocab_partials(VocabMode mode, const CUtensorMap& tm, const VocabArgs& a, cudaStream_t stream);

}  // namespace dspark
