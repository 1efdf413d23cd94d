// Host-side shared definitions of libdspark: workspace layout, launch
// geometry and small utilities.  Device helpers live in device.cuh.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "dspark.h"

namespace dspark {

// ------------------------------------------------------------------ draft geometry
constexpr int kMTile = 128;        // rows (requests) per tensor-core tile (UMMA M)
constexpr int kTileN = 64;         // vocabulary columns per tile (UMMA N)
constexpr int kSubN = 32;          // columns per fine softmax partial (one epilogue warp)
constexpr int kMaxChunks = 1024;   // upper bound on contiguous V-chunks per M-tile
constexpr int kUStride = kTileN * 4 + 16;  // bytes per bulk-copied U row (padded: conflict-free)
constexpr int kPfTiles = 4;        // tiles per L2 prefetch group (a 256-column span per row)
constexpr int kDraftThreads = 320; // warp 0 TMA producer, warp 1 MMA, warps 2..9 epilogue
constexpr int kVerifyChunk = 1024; // target columns per verify statistics item (32 per lane)
constexpr int kMaxGamma = 64;
constexpr int kMaxLmHeadD = 65536;  // hidden size bound of the fused LM-head draft
constexpr int kMaxSchedule = 8192; // R * gamma handled by the one-CTA scheduler
constexpr int kMaxVerifyR = 32768; // verify keeps R + 1 row offsets in shared memory

constexpr int kMaxSampleChunks = 256; // chunk partials per row the draft sampler holds in registers

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct WorkspaceLayout {
  size_t status = 0;     // int32 status word (+ padding)
  size_t coarse = 0;     // float2 [R_pad][kMaxChunks] per-chunk softmax partials
  size_t fine = 0;       // float2 [n_sub][R_pad] per-32-column softmax partials
  size_t tstats = 0;     // float2 [R*(gamma+1)][n_vchunks] target-row partials
  size_t trow = 0;       // float4 [R*(gamma+1)] per target row: (max, sum, t(x), unused)
  size_t rowoff = 0;     // int32 [R+1] verify row offsets
  size_t rej = 0;        // int32 [R_pad] rejecting requests (-1 = none) + count
  size_t total = 0;
  // The draft's synchronisation words, in the tail of the chunk-partials
  // region that the draft never uses (it keeps <= kMaxSampleChunks chunks per
  // row): a done counter and a ready counter per M-tile and the abort word,
  // each on its own 64-byte line.  Zeroed at the start of every draft call.
  size_t dsync = 0;
  size_t dsync_bytes = 0;
  // The draft's staging copy of each row's next A operand (the W1 row of the
  // token just drawn), 512 bytes per row, in the same unused tail, laid out so
  // that a gather warp reads whole 128-byte lines: uint4 index
  // (((mtile * 4 + quarter) * 2 + half) * 16 + k) * 32 + lane.
  size_t abuf = 0;
  size_t abuf_bytes = 0;
};

inline WorkspaceLayout workspace_layout(int R, int gamma, int V) {
  WorkspaceLayout L;
  const size_t R_pad = static_cast<size_t>(ceil_div(R > 0 ? R : 1, kMTile)) * kMTile;
  const size_t n_tiles = static_cast<size_t>(ceil_div(V, kTileN));
  const size_t n_sub = 2 * n_tiles;
  const size_t rows = static_cast<size_t>(R) * static_cast<size_t>(gamma + 1);
  const size_t n_vchunks = static_cast<size_t>(ceil_div(V, kVerifyChunk));
  size_t off = 256;
  L.coarse = off; off = align256(off + static_cast<size_t>(kMaxChunks) * R_pad * 8);
  L.fine = off;   off = align256(off + n_sub * R_pad * 8);
  L.tstats = off; off = align256(off + rows * n_vchunks * 8);
  L.trow = off;   off = align256(off + rows * 16);
  L.rowoff = off; off = align256(off + (static_cast<size_t>(R) + 1) * 4);
  L.rej = off;    off = align256(off + (R_pad + 4) * 4);
  L.total = off;
  L.dsync = L.coarse + R_pad * kMaxSampleChunks * 8;
  L.dsync_bytes = 64 * (2 * (R_pad / kMTile) + 1);
  L.abuf = align256(L.dsync + L.dsync_bytes);
  L.abuf_bytes = R_pad * 512;
  return L;
}

// SM count of the current device (cached per device).
int sm_count();

// Launch helper: programmatic dependent launch on `stream`.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dspark
