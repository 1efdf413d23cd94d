// Markov-head sequential draft ("DSpark" §2.2 eq. p_k, §2.3 eq. B = W1 W2,
// and the position-by-position loop of §6.2).  Per draft position j:
//
//  k_vocab_partials<kDraft> — the tensor-core bias pass of vocab_gemm.cuh:
//    softmax partials of z_j = (U_j + W1[x_{j-1}] W2) / T per 32-column
//    sub-tile and per CTA chunk, without writing logits to HBM.
//  k1_sample — one CTA per request: combines the chunk partials into the
//    row's max and normaliser, finds the chunk, then the 32-column sub-tile,
//    in which the cumulative mass first exceeds u * Z, recomputes that
//    sub-tile's 32 logits on CUDA cores (the rank dimension split over the
//    CTA's 8 warps) and picks the token; writes x_j, p_d(x_j) and log Z_j.
//    Greedy: the argmax of the chunk partials.
//
// Both kernels and consecutive positions are chained with programmatic
// dependent launch: the next position's W2 / U loads overlap the sampling.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <utility>

#include "common.h"
#include "device.cuh"
#include "search.cuh"
#include "vocab_gemm.cuh"

namespace dspark {

constexpr int kSampleThreads = 256;

struct SampleArgs {
  const float* U;
  const uint16_t* W1;
  const uint16_t* W2;
  const int32_t* anchors;
  int32_t* tokens;
  float* pd_tok;
  float* logZ;
  const float2* coarse;  // [R_pad][n_chunks]
  const float2* fine;    // [2 * n_tiles][R_pad]
  int32_t* status;
  int R, R_pad, gamma, V, rank, step, n_tiles, n_chunks;
  float scale;
  int greedy;
  uint64_t seed;
  uint32_t round;
};

__global__ void __launch_bounds__(kSampleThreads) k1_sample(const SampleArgs p) {
  __shared__ BlockFindScratch sc;
  __shared__ float s_redf[32];
  __shared__ float s_redz[32];
  __shared__ int s_redi[32];
  __shared__ float s_e[256];
  __shared__ float s_part[kSampleThreads / 32][32];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int r = blockIdx.x;
  const size_t out = static_cast<size_t>(r) * p.gamma + p.step;
  const float2* crow = p.coarse + static_cast<size_t>(r) * p.n_chunks;

  if (p.greedy) {
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    for (int c = tid; c < p.n_chunks; c += kSampleThreads) {
      const float2 e = crow[c];
      const int ei = __float_as_int(e.y);
      if (e.x > best || (e.x == best && ei < bidx)) { best = e.x; bidx = ei; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
      if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
    }
    if (lane == 0) { s_redf[wid] = best; s_redi[wid] = bidx; }
    __syncthreads();
    if (wid == 0) {
      best = lane < kSampleThreads / 32 ? s_redf[lane] : -INFINITY;
      bidx = lane < kSampleThreads / 32 ? s_redi[lane] : 0x7fffffff;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
      }
      if (lane == 0) {
        if (!(fabsf(best) <= 3.4e38f) || bidx < 0 || bidx >= p.V) {
          report(p.status, DSPARK_STATUS_NONFINITE);
          bidx = 0;
        }
        p.tokens[out] = bidx;
        p.pd_tok[out] = 1.0f;
        p.logZ[out] = best;
      }
    }
    return;
  }

  // the previous token's W1 row, needed by the recompute at the end
  const int prev_raw = p.step == 0 ? p.anchors[r] : p.tokens[static_cast<size_t>(r) * p.gamma + p.step - 1];
  const int prev = (prev_raw >= 0 && prev_raw < p.V) ? prev_raw : 0;
  for (int i = tid; i < p.rank; i += kSampleThreads) s_e[i] = bf16_at(p.W1 + static_cast<size_t>(prev) * p.rank + i);

  // row maximum and normaliser (base-2 units) in one pass: each thread merges
  // its chunks online, then the block merges the (max, sum) pairs
  float m = -INFINITY, zs = 0.f;
  for (int c = tid; c < p.n_chunks; c += kSampleThreads) {
    const float2 e = crow[c];
    if (e.x > -INFINITY) {
      if (e.x > m) {
        zs = (m > -INFINITY ? zs * exp2f(m - e.x) : 0.f) + e.y;
        m = e.x;
      } else {
        zs += e.y * exp2f(e.x - m);
      }
    }
  }
  const float M = block_max_f(m, s_redf);
  const float Z = block_sum_f(m > -INFINITY ? zs * exp2f(m - M) : 0.f, s_redz);
  auto chunk_w = [&](int c) -> float {
    const float2 e = crow[c];
    return e.x > -INFINITY ? e.y * exp2f(e.x - M) : 0.f;
  };
  if (!(fabsf(M) <= 3.4e38f) || !(Z > 0.f) || !(Z <= 3.4e38f)) {
    if (tid == 0) {
      report(p.status, DSPARK_STATUS_NONFINITE);
      p.tokens[out] = 0;
      p.pd_tok[out] = 0.f;
      p.logZ[out] = NAN;
    }
    return;
  }
  const float u = uniform24(p.seed, p.round, static_cast<uint64_t>(r), static_cast<uint64_t>(p.step), kDraftSample);
  const float target = u * Z;
  float before_c = 0.f;
  const int cstar = block_find_crossing<kSampleThreads>(p.n_chunks, 0.f, target, chunk_w, &before_c, sc);
  const int tb = static_cast<int>((static_cast<long long>(cstar) * p.n_tiles) / p.n_chunks);
  const int te = static_cast<int>((static_cast<long long>(cstar + 1) * p.n_tiles) / p.n_chunks);
  const float2* frow = p.fine + r;
  auto sub_w = [&](int i) -> float {
    const float2 e = frow[static_cast<size_t>(2 * tb + i) * p.R_pad];
    return e.x > -INFINITY ? e.y * exp2f(e.x - M) : 0.f;
  };
  float before_s = 0.f;
  const int sstar = 2 * tb + block_find_crossing<kSampleThreads>(2 * (te - tb), before_c, target, sub_w, &before_s, sc);

  // recompute the 32 logits of that sub-tile: column = lane, rank split over
  // the warps; every W2 load of a thread is issued before the first FMA
  const int v = sstar * kSubN + lane;
  const int per = p.rank / (kSampleThreads / 32);  // <= 32
  float acc = 0.f;
  if (v < p.V) {
    const uint16_t* col = p.W2 + static_cast<size_t>(wid * per) * p.V + v;
    uint16_t wv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) wv[i] = i < per ? col[static_cast<size_t>(i) * p.V] : 0;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < per) acc = fmaf(s_e[wid * per + i], __uint_as_float(static_cast<uint32_t>(wv[i]) << 16), acc);
  }
  s_part[wid][lane] = acc;
  __syncthreads();
  if (wid == 0) {
    float y = -INFINITY, w = 0.f;
    if (v < p.V) {
      float b = 0.f;
#pragma unroll
      for (int k = 0; k < kSampleThreads / 32; ++k) b += s_part[k][lane];
      y = (b + p.U[(static_cast<size_t>(r) * p.gamma + p.step) * p.V + v]) * p.scale;
      w = exp2f(y - M);
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
    const float ypick = __shfl_sync(0xffffffffu, y, pick);
    if (lane == 0) {
      const int x = min(sstar * kSubN + pick, p.V - 1);
      p.tokens[out] = x;
      p.pd_tok[out] = exp2f(ypick - M) / Z;
      p.logZ[out] = (M + log2f(Z)) * 0.69314718f;
    }
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// W2 [rank, V] bf16 as a 2-D tensor (x = vocabulary, y = rank); box 64 x rank
// with 128-byte swizzle: the MN-major SW128 operand layout of the UMMA.
int encode_w2_map(CUtensorMap* tm, const uint16_t* W2, int V, int rank) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(rank)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileN), static_cast<cuuint32_t>(rank)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W2), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// U [R, gamma, V] fp32 as a 3-D tensor (x = vocabulary, y = position,
// z = request); box 32 x 1 x 128 with 128-byte swizzle.
int encode_u_map(CUtensorMap* tm, const float* U, int R, int gamma, int V) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(gamma), static_cast<cuuint64_t>(R)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(V) * 4, static_cast<cuuint64_t>(V) * 4 * gamma};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kSubN), 1, static_cast<cuuint32_t>(kMTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(U), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? DSPARK_OK : DSPARK_ERR_CUDA;
}

int vocab_chunks(int n_tiles, int n_mtiles) {
  int c = sm_count() / n_mtiles;
  if (c < 1) c = 1;
  if (c > n_tiles) c = n_tiles;
  if (c > kMaxChunks) c = kMaxChunks;
  return c;
}

// pdl: whether this launch may overlap the tail of the previous kernel in the
// stream.  A draft pass reads U and W2 before its griddepcontrol.wait, so the
// first pass of a call is launched without it: whatever precedes the call on
// the stream (for instance the kernel that produced U) completes first.
cudaError_t launch_vocab_partials(VocabMode mode, const CUtensorMap& tm_w2, const CUtensorMap& tm_u,
                                  const VocabArgs& a, cudaStream_t stream, bool pdl) {
  const VocabSmem plan = vocab_smem_plan(a.rank);
  const dim3 grid(a.n_chunks * a.n_mtiles);
  const int max_smem = static_cast<int>(vocab_smem_plan(256).total);
  if (mode == VocabMode::kDraft) {
    static std::once_flag once;
    std::call_once(once, [&] {
      cudaFuncSetAttribute(k_vocab_partials<VocabMode::kDraft>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    });
    return launch_pdl(k_vocab_partials<VocabMode::kDraft>, grid, dim3(kDraftThreads), plan.total, stream, pdl, tm_w2,
                      tm_u, a);
  }
  static std::once_flag once_r;
  std::call_once(once_r, [&] {
    cudaFuncSetAttribute(k_vocab_partials<VocabMode::kResidual>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  });
  return launch_pdl(k_vocab_partials<VocabMode::kResidual>, grid, dim3(kDraftThreads), plan.total, stream, pdl, tm_w2,
                    tm_u, a);
}

int launch_markov_draft(const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* anchors, int R,
                        int gamma, int V, int rank, float temperature, uint64_t seed, uint32_t round,
                        int32_t* tokens, float* pd_tok, float* logZ, void* workspace, cudaStream_t stream) {
  const WorkspaceLayout L = workspace_layout(R, gamma, V);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  VocabArgs a = {};
  a.U = U; a.W1 = W1; a.W2 = W2; a.anchors = anchors; a.tokens = tokens;
  a.coarse = reinterpret_cast<float2*>(ws + L.coarse);
  a.fine = reinterpret_cast<float2*>(ws + L.fine);
  a.status = reinterpret_cast<int32_t*>(ws + L.status);
  a.R = R;
  a.n_mtiles = ceil_div(R, kMTile);
  a.R_pad = a.n_mtiles * kMTile;
  a.gamma = gamma; a.V = V; a.rank = rank;
  a.n_tiles = ceil_div(V, kTileN);
  a.n_chunks = vocab_chunks(a.n_tiles, a.n_mtiles);
  a.greedy = temperature == 0.0f ? 1 : 0;
  a.scale = a.greedy ? 1.0f : static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));

  SampleArgs s = {};
  s.U = U; s.W1 = W1; s.W2 = W2; s.anchors = anchors; s.tokens = tokens; s.pd_tok = pd_tok; s.logZ = logZ;
  s.coarse = a.coarse; s.fine = a.fine; s.status = a.status;
  s.R = R; s.R_pad = a.R_pad; s.gamma = gamma; s.V = V; s.rank = rank;
  s.n_tiles = a.n_tiles; s.n_chunks = a.n_chunks; s.scale = a.scale; s.greedy = a.greedy;
  s.seed = seed; s.round = round;

  CUtensorMap tm_w2, tm_u;
  if (encode_w2_map(&tm_w2, W2, V, rank) != DSPARK_OK || encode_u_map(&tm_u, U, R, gamma, V) != DSPARK_OK)
    return DSPARK_ERR_CUDA;
  for (int step = 0; step < gamma; ++step) {
    a.step = step;
    s.step = step;
    if (launch_vocab_partials(VocabMode::kDraft, tm_w2, tm_u, a, stream, step > 0) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (launch_pdl(k1_sample, dim3(R), dim3(kSampleThreads), 0, stream, true, s) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  }
  return DSPARK_OK;
}

}  // namespace dspark
