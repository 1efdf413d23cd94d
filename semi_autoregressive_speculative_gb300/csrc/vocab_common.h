// Shared by the two tensor-core vocabulary passes (the draft kernel in
// markov_draft.cu and the residual pass of verify): tensor-memory budget,
// tensor maps over W2 and U, and the split of the vocabulary into per-CTA
// chunks.
#pragma once

#include <cuda.h>

#include "common.h"

namespace dspark {

constexpr int kAccCols = 2 * kTileN;  // two fp32 accumulators of 64 columns
constexpr int kTmemCols = 256;        // accumulators + the A operand (rank / 2 columns, rank <= 256)

// W2 [rank, V] bf16 as a 2-D tensor; box 64 x rank, 128-byte swizzle (the
// MN-major SW128 B-operand layout of the UMMA).
int encode_w2_map(CUtensorMap* tm, const uint16_t* W2, int V, int rank);
// W2 again, box 32 x rank without swizzle: the 32 columns of one sub-tile as
// [rank][32] (the samplers' recompute of a sub-tile's bias).
int encode_w2_slab_map(CUtensorMap* tm, const uint16_t* W2, int V, int rank);
// U [R, gamma, V] fp32 as a 2-D tensor of R * gamma rows (row = request *
// gamma + position), box 64 x 1, no swizzle: rows gathered four at a time
// (tile::gather4) by the verify residual pass.
int encode_u_rows_map(CUtensorMap* tm, const float* U, int R, int gamma, int V);
// Contiguous V-chunks per M-tile so that chunks x M-tiles fills the SMs once.
int vocab_chunks(int n_tiles, int n_mtiles);

}  // namespace dspark
