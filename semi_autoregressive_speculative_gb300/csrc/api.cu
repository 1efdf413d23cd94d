// extern "C" entry points of libdspark.so: argument validation, workspace
// layout and dispatch to the kernels.  See include/dspark.h for the contract.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.h"

namespace dspark {

int launch_markov_draft(const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* anchors, int R,
                        int gamma, int V, int rank, float temperature, uint64_t seed, uint32_t round,
                        int32_t* tokens, float* pd_tok, float* logZ, void* workspace, cudaStream_t stream);
int launch_markov_draft_lmhead(const uint16_t* h, const uint16_t* W_lm, int d, const uint16_t* W1, const uint16_t* W2,
                               const int32_t* anchors, int R, int gamma, int V, int rank, float temperature,
                               uint64_t seed, uint32_t round, int32_t* tokens, float* pd_tok, float* logZ,
                               void* workspace, cudaStream_t stream);
int launch_confidence(const uint16_t* h, const uint16_t* W1, const float* w, const float* sts_t,
                      const int32_t* anchors, const int32_t* tokens, int R, int gamma, int d, int rank, int V,
                      float* c, float* a, int32_t* status, cudaStream_t stream);
int launch_schedule(const float* a, int R, int gamma, const double* sps, int mode, int budget_K, int32_t* lens,
                    int32_t* total_b, int32_t* argmax_b, double* theta, int32_t* status, cudaStream_t stream);
int launch_verify(const float* T, const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* anchors,
                  const int32_t* tokens, const float* pd_tok, const float* logZ, const int32_t* lens, int R, int gamma,
                  int V, int rank, float temperature, uint64_t seed, uint32_t round, int32_t* n_accept,
                  int32_t* next_token, float* c_star, void* workspace, cudaStream_t stream);
int launch_load_verified_rows(const float* T_host, const int32_t* lens, int R, int gamma, int V, float* T,
                              int32_t* status, cudaStream_t stream);

int sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    count[dev] = n;
  }
  return count[dev];
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool finite_nonneg(float t) { return t >= 0.0f && t <= 3.4e38f; }
static bool rank_ok(int rank) { return rank == 64 || rank == 128 || rank == 192 || rank == 256; }

}  // namespace dspark

using namespace dspark;

extern "C" {

size_t dspark_workspace_size(int R, int gamma, int V, int rank, int d) {
  (void)rank;
  (void)d;
  if (R < 0 || gamma < 0 || gamma > kMaxGamma || V <= 0) return 0;
  return workspace_layout(R, gamma, V).total;
}

int dspark_clear_status(void* workspace, void* stream) {
  if (!workspace) return DSPARK_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_ERR_CUDA;
}

int dspark_markov_draft(const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* anchors, int R,
                        int gamma, int V, int rank, float temperature, uint64_t seed, uint32_t round, int32_t* tokens,
                        float* pd_tok, float* logZ, void* workspace, size_t workspace_bytes, void* stream) {
  if (R < 0 || gamma < 1 || V < 8 || rank < 1 || !finite_nonneg(temperature)) return DSPARK_ERR_INVALID_ARG;
  if (gamma > kMaxGamma || V % 8 != 0 || !rank_ok(rank)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return DSPARK_OK;
  if (!U || !W1 || !W2 || !anchors || !tokens || !pd_tok || !logZ || !workspace) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DSPARK_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_layout(R, gamma, V).total) return DSPARK_ERR_INVALID_ARG;
  return launch_markov_draft(U, W1, W2, anchors, R, gamma, V, rank, temperature, seed, round, tokens, pd_tok, logZ,
                             workspace, static_cast<cudaStream_t>(stream));
}

int dspark_markov_draft_lmhead(const uint16_t* h, const uint16_t* W_lm, const uint16_t* W1, const uint16_t* W2,
                               const int32_t* anchors, int R, int gamma, int V, int rank, int d, float temperature,
                               uint64_t seed, uint32_t round, int32_t* tokens, float* pd_tok, float* logZ,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (R < 0 || gamma < 1 || V < 8 || rank < 1 || d < 1 || !finite_nonneg(temperature)) return DSPARK_ERR_INVALID_ARG;
  if (gamma > kMaxGamma || V % 8 != 0 || !rank_ok(rank) || d % 128 != 0 || d > kMaxLmHeadD)
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return DSPARK_OK;
  if (!h || !W_lm || !W1 || !W2 || !anchors || !tokens || !pd_tok || !logZ || !workspace) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W_lm) || !aligned16(W1) || !aligned16(W2) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DSPARK_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_layout(R, gamma, V).total) return DSPARK_ERR_INVALID_ARG;
  return launch_markov_draft_lmhead(h, W_lm, d, W1, W2, anchors, R, gamma, V, rank, temperature, seed, round, tokens,
                                    pd_tok, logZ, workspace, static_cast<cudaStream_t>(stream));
}

int dspark_confidence(const uint16_t* h, const uint16_t* W1, const float* w, const float* sts_temperature,
                      const int32_t* anchors, const int32_t* tokens, int R, int gamma, int d, int rank, int V,
                      float* c, float* a, void* workspace, size_t workspace_bytes, void* stream) {
  if (R < 0 || gamma < 1 || d < 1 || rank < 1 || V < 1) return DSPARK_ERR_INVALID_ARG;
  if (gamma > kMaxGamma) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return DSPARK_OK;
  if (!h || !W1 || !w || !anchors || !tokens || !c || !a || !workspace) return DSPARK_ERR_INVALID_ARG;
  if (workspace_bytes < sizeof(int32_t)) return DSPARK_ERR_INVALID_ARG;
  return launch_confidence(h, W1, w, sts_temperature, anchors, tokens, R, gamma, d, rank, V, c, a,
                           static_cast<int32_t*>(workspace), static_cast<cudaStream_t>(stream));
}

int dspark_schedule(const float* a, int R, int gamma, const double* sps, int sps_len, int mode, int budget_K,
                    int32_t* lens, int32_t* total_b, int32_t* argmax_b, double* theta, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (R < 1 || gamma < 1 || mode < 0 || mode > 2) return DSPARK_ERR_INVALID_ARG;
  if (gamma > kMaxGamma || static_cast<long long>(R) * gamma > kMaxSchedule) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (sps_len < R * (1 + gamma) + 1) return DSPARK_ERR_INVALID_ARG;
  if (!a || !sps || !lens || !total_b || !argmax_b || !theta || !workspace) return DSPARK_ERR_INVALID_ARG;
  if (workspace_bytes < sizeof(int32_t)) return DSPARK_ERR_INVALID_ARG;
  return launch_schedule(a, R, gamma, sps, mode, budget_K, lens, total_b, argmax_b, theta,
                         static_cast<int32_t*>(workspace), static_cast<cudaStream_t>(stream));
}

int dspark_verify(const float* T, const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* anchors,
                  const int32_t* tokens, const float* pd_tok, const float* logZ, const int32_t* lens, int R, int gamma,
                  int V, int rank, float temperature, uint64_t seed, uint32_t round, int32_t* n_accept,
                  int32_t* next_token, float* c_star, void* workspace, size_t workspace_bytes, void* stream) {
  if (R < 0 || gamma < 1 || V < 8 || rank < 1 || !finite_nonneg(temperature)) return DSPARK_ERR_INVALID_ARG;
  if (gamma > kMaxGamma || V % 8 != 0 || !rank_ok(rank) || R > kMaxVerifyR) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return DSPARK_OK;
  if (!T || !U || !W1 || !W2 || !anchors || !tokens || !pd_tok || !logZ || !lens || !n_accept || !next_token ||
      !workspace)
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(T) || !aligned16(U) || !aligned16(W1) || !aligned16(W2) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DSPARK_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_layout(R, gamma, V).total) return DSPARK_ERR_INVALID_ARG;
  return launch_verify(T, U, W1, W2, anchors, tokens, pd_tok, logZ, lens, R, gamma, V, rank, temperature, seed, round,
                       n_accept, next_token, c_star, workspace, static_cast<cudaStream_t>(stream));
}

int dspark_load_verified_rows(const float* T_host, const int32_t* lens, int R, int gamma, int V, float* T,
                              void* workspace, void* stream) {
  if (R < 0 || gamma < 1 || V < 8) return DSPARK_ERR_INVALID_ARG;
  if (gamma > kMaxGamma || V % 8 != 0) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (R == 0) return DSPARK_OK;
  if (!T_host || !lens || !T || !workspace) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(T_host) || !aligned16(T) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DSPARK_ERR_INVALID_ARG;
  return launch_load_verified_rows(T_host, lens, R, gamma, V, T, static_cast<int32_t*>(workspace),
                                   static_cast<cudaStream_t>(stream));
}

}  // extern "C"
