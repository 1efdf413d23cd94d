// dspark_markov_draft_noalloc: the Markov-head draft for callers that cannot
// hand the library a workspace.
//
// Some callers have no way to obtain device memory at the point where they
// draft.  Examples:
//  - An engine that records the whole decode step into a CUDA graph. It may
//    not call cudaMalloc while capture is open.
//  - A latency-critical serving loop that forbids allocator calls on its hot
//    path, because cudaMalloc / cudaFree can synchronise the device.
//  - A plug-in whose host program owns all device memory and gives the plug-in
//    no allocator.
// For them this file keeps the draft's scratch (the status word and the
// per-chunk and per-32-column softmax partials) in one file-scope device array
// of fixed size. The caller passes only the inputs and outputs.
//
// Properties a caller has to know:
//  - Every GPU that loads libdspark.so holds kNoAllocScratchBytes (16 MiB) for
//    this array until the process exits.
//  - Shapes whose scratch does not fit are rejected with
//    DSPARK_ERR_STATIC_SCRATCH_TOO_SMALL before anything is enqueued.
//  - All calls on a device share the one array, and it keeps the contents of
//    the previous call. Each call clears the status word before its kernels
//    run; the partials are fully rewritten before they are read. Two calls
//    whose kernels overlap on the GPU (different streams, no ordering between
//    them) race on the array and give wrong results.
//  - The first call on each device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current) and caches it. Make that
//    first call before any stream capture begins.
//  - Nothing here calls cudaMalloc, cudaFree or an allocating library routine.
#include <cstdint>
#include <mutex>

#include "common.h"

namespace dspark {

int launch_markov_draft(const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* anchors, int R,
                        int gamma, int V, int rank, float temperature, uint64_t seed, uint32_t round,
                        int32_t* tokens, float* pd_tok, float* logZ, void* workspace, cudaStream_t stream);

constexpr size_t kNoAllocScratchBytes = DSPARK_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes == (size_t(16) << 20), "16 MiB");

// The draft's scratch.  In host code this name is only a host-side handle of
// the symbol, never a device address: kernels get the address that
// cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Bytes of the workspace layout the draft touches: the status word, the chunk
// partials and the 32-column partials (the verify regions come after them).
size_t draft_scratch_bytes(int R, int gamma, int V) {
  const WorkspaceLayout L = workspace_layout(R, gamma, V);
  const size_t R_pad = static_cast<size_t>(ceil_div(R, kMTile)) * kMTile;
  const size_t n_sub = 2 * static_cast<size_t>(ceil_div(V, kTileN));
  return L.fine + n_sub * R_pad * sizeof(float2);
}

// Device address of the array on the current device (looked up once per device).
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSPARK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DSPARK_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" int dspark_markov_draft_noalloc(const float* U, const uint16_t* W1, const uint16_t* W2,
                                           const int32_t* anchors, int R, int gamma, int V, int rank,
                                           float temperature, uint64_t seed, uint32_t round, int32_t* tokens,
                                           float* pd_tok, float* logZ, int32_t* status, void* stream) {
  // the same argument rules as dspark_markov_draft
  if (R < 0 || gamma < 1 || V < 8 || rank < 1 || !(temperature >= 0.0f && temperature <= 3.4e38f))
    return DSPARK_ERR_INVALID_ARG;
  if (gamma > kMaxGamma || V % 8 != 0 || !(rank == 64 || rank == 128 || rank == 192 || rank == 256))
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (draft_scratch_bytes(R, gamma, V) > kNoAllocScratchBytes) return DSPARK_ERR_STATIC_SCRATCH_TOO_SMALL;
  if (R == 0) return DSPARK_OK;
  if (!U || !W1 || !W2 || !anchors || !tokens || !pd_tok || !logZ) return DSPARK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(U) | reinterpret_cast<uintptr_t>(W1) | reinterpret_cast<uintptr_t>(W2)) & 15u)
    return DSPARK_ERR_INVALID_ARG;

  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != DSPARK_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the previous call's status bits must not leak into this one
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), st) != cudaSuccess) return DSPARK_ERR_CUDA;
  const int lr = launch_markov_draft(U, W1, W2, anchors, R, gamma, V, rank, temperature, seed, round, tokens, pd_tok,
                                     logZ, scratch, st);
  if (lr != DSPARK_OK) return lr;
  if (status &&
      cudaMemcpyAsync(status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}
