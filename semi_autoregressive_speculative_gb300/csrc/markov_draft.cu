// Markov-head sequential draft ("DSpark" §2.2 eq. p_k, §2.3 eq. B = W1 W2,
// and the position-by-position loop of §6.2) as ONE persistent cooperative
// kernel per call: every CTA stays resident for all gamma positions.  A small
// prologue kernel before it clears the call's tagged words and stages the
// anchors' W1 rows (k_draft_prologue).  A compile-time variant takes the
// pre-LM-head hidden states instead of U and forms U = h . W_lm in the same
// MMAs (kLm, "DSpark: Speculative decodingを活用した…", "隠れ状態通信").
//
// Per position j, on every CTA (one contiguous V-chunk of one 128-row M-tile):
//   gather   each row's W1[x_{j-1}] goes into tensor memory as the UMMA A
//            operand, once the samplers of the M-tile have published the
//            previous tokens (a per-M-tile counter; the publishing sampler
//            has already staged the row in gather order)
//   tiles    W2 in 128-row K-chunks (L2-resident after the first position)
//            and U tiles (128 rows x 64 columns) come in through TMA rings,
//            each fed by its own producer warp; U is copied into the fp32
//            accumulators in tensor memory and tcgen05.mma adds the bias on
//            top, two 64-column tiles per instruction (below); the epilogue
//            takes a pair of tiles per iteration, scales z = U + bias by
//            log2(e)/T and reduces each 32-column sub-tile and the whole
//            chunk to softmax partials (max, sum exp2) — (max, argmax) when
//            greedy.  Logits never reach HBM.  Each row's chunk partial is
//            published as one tagged 64-bit entry (chunk_entry).
//   sample   the CTA's requests (all 8 epilogue warps per request; one warp
//            per request when greedy): the leader polls the row's chunk
//            entries, merges them into the row's max and normaliser, finds
//            the chunk, then the 32-column sub-tile, where the cumulative
//            mass first exceeds u * Z, and the warps recompute those 32
//            logits from a slab of W2 columns; the leader picks x_j, writes
//            x_j, p_d(x_j) and log Z_j, stages W1[x_j] for the next gather
//            and counts x_j as published on its M-tile.  Greedy: argmax of
//            the entries.
// The producer warps never wait for the samplers: W2 and U do not depend on
// the drafted tokens, so they stream the next position's first tiles into the
// rings while the samplers run.  Every wait is bounded (kWaitLimitNs); a CTA
// that gives up raises a grid-wide abort word and DSPARK_STATUS_TIMEOUT.
// Waits are polled by one thread per group (a CTA's gather, a sampler warp)
// with a short sleep, and shared through named barriers or shuffles.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <utility>

#include "common.h"
#include "device.cuh"
#include "search.cuh"
#include "vocab_common.h"

namespace dspark {

// Tiles are multiplied in pairs.  An M=128, K=16 tcgen05.mma costs about 66
// cycles at N=64 and 80 at N=128 (microbenchmark, one CTA), so one N=128
// instruction per K-step covers two 64-column tiles at 0.62 cycles per column
// against 1.03.
// W2 comes in K-chunks: a ring stage holds 128 rank rows of both tiles of a
// pair (two 128 x 64 boxes, 128-byte swizzled, 16 KB apart: the B descriptor
// spans them as two swizzle atoms along N).  A stage is released as soon as
// its 8 MMAs are done.  The issuing thread pays for every wait and commit
// (about 110 and 220 cycles: 16 MMAs cost 1 430 cycles back to back and 2 770
// with a wait and a commit every 4), so a pair takes two chunks, not four.
constexpr int kDraftKChunk = 128;    // rank rows per W2 stage (fewer, when the rank is smaller)
constexpr int kDraftWBox = kDraftKChunk * 128;  // bytes of one 64-column box of a stage
constexpr int kDraftWStages = 4;     // W2 K-chunk stages (L2-resident after the first position)
constexpr int kDraftUStages = 2;     // U tiles staged in shared memory (tensor memory holds 3 pairs more)
constexpr int kDraftAccPairs = 3;    // fp32 accumulator pairs (2 x 64 columns each) in tensor memory
constexpr int kDraftACol = kDraftAccPairs * 2 * kTileN;  // first tensor-memory column of the A operand
constexpr int kDraftTmemCols = 512;                      // accumulators + A (rank / 2 <= 128 columns)
static_assert(kDraftACol + 128 <= kDraftTmemCols, "tensor-memory plan");
// warp 0 W2 producer, warp 1 MMA issuer, warps 2..9 epilogue and samplers,
// warp 10 U producer, warp 11 U copier
constexpr int kDraftKThreads = kDraftThreads + 64;
constexpr int kUWarp = 10;
constexpr int kCopyWarp = 11;
// U never passes through registers: each 128-row x 64-column U tile lands in
// shared memory by TMA in the 128-byte-swizzled K-major layout and is copied
// into its accumulator pair in tensor memory (tcgen05.cp, by the copier warp)
// before the MMA, which then accumulates the Markov bias on top of it.  The
// copier runs as far ahead as the accumulator slots allow: while the samplers
// of a position run, the next position's first three pairs are already in
// tensor memory and the ring refills behind them, so the HBM stream no longer
// stops between positions.
//   fast layout (R % 8 == 0, a whole tile): one 5-D TMA box {32 columns,
//     8 rows, 2 halves, 16 row groups} per tile, so that each request row's
//     256 contiguous bytes are fetched together (a box per 32-column half
//     streams at about 70 % of that rate).  Row group g holds half h of its
//     8 rows at byte g * 2048 + h * 1024 (SBO 2048).
//   general layout (a ragged last tile, or R % 8 != 0): two 3-D boxes
//     {32, 1, 128} per tile, columns past V and rows past R zero-filled; half
//     h at byte h * 16384, rows at 128 bytes (SBO 1024).
constexpr int kDraftUBytes = kMTile * kTileN * 4;  // one U tile (32 KB, 1024-aligned stages)
constexpr int kEpiThreads = kDraftThreads - 64;  // warps 2..9
constexpr int kMaxDraftV = 1 << 24;               // vocabulary bound of the 32-bit chunk arithmetic

// Phase tracing (compiled only with -DDSPARK_DRAFT_TRACE, into a separate
// build of the library used by the draft_trace tool; the product build has
// none of it).  Every CTA stamps the global timer (ns) at each event of each
// position into trace[(position * n_ctas + cta) * kTraceEvents + event].
enum TraceEvent {
  kEvAReady = 0,      // the position's A operand is in tensor memory (gather done)
  kEvFirstAcc = 1,    // the first accumulator pair of the position is ready
  kEvTilesDone = 2,   // the CTA's last tile pair of the position is reduced
  kEvEntry = 3,       // the CTA's chunk entries are published
  kEvPollDone = 4,    // sampler (the CTA's first request): every chunk entry seen
  kEvChunkFound = 5,  // sampler: crossing chunk found
  kEvFineLoaded = 6,  // sampler: the crossing chunk's sub-tile partials loaded
  kEvSlabIssued = 7,  // sampler: crossing sub-tile found, slab copy issued
  kEvSlabLanded = 8,  // sampler: slab in shared memory
  kEvPicked = 9,      // sampler: token picked
  kEvPublished = 10,  // sampler: token published (W1 row staged, counted)
  kEvReadySeen = 11,  // the previous position's tokens of the M-tile are all published
  kEvCopyFirst = 12,  // copier: the position's first pair of U is in tensor memory (issued)
  kEvCopyThird = 13,  // copier: the position's third pair of U is in tensor memory (issued)
  kEvStart = 14,      // the CTA's set-up is done (position 0's slot only)
  kEvEnd = 15,        // the CTA is about to free its tensor memory and exit (position 0's slot only)
  kEvLaunch = 16,     // the CTA's first instruction (position 0's slot only)
  kEvProStart = 17,   // prologue block b (b < the draft's CTA count) starts (position 0, CTA b)
  kEvProEnd = 18,     // prologue block b is done (position 0, CTA b)
  kTraceEvents = 19
};
#ifdef DSPARK_DRAFT_TRACE
#define DRAFT_TRACE(p, step, ev)                                                                         \
  do {                                                                                                   \
    if ((p).trace)                                                                                       \
      (p).trace[(static_cast<size_t>(step) * gridDim.x + blockIdx.x) * kTraceEvents + (ev)] = global_ns(); \
  } while (0)
#else
#define DRAFT_TRACE(p, step, ev) \
  do {                           \
  } while (0)
#endif

struct DraftArgs {
  const float* U;          // [R, gamma, V] (null with the LM head)
  const uint16_t* h;       // [R, gamma, d] bf16 pre-LM-head hidden states (LM head only)
  const uint16_t* W1;      // [V, rank]
  const uint16_t* W2;      // [rank, V]
  const int32_t* anchors;  // [R]
  int32_t* tokens;         // [R, gamma]
  float* pd_tok;           // [R, gamma]
  float* logZ;             // [R, gamma]
  unsigned long long* centry;  // [R_pad][n_chunks] tagged chunk entries (see chunk_entry)
  unsigned long long* fine;  // [2 * n_tiles][R_pad] tagged sub-tile partials (sampled draws only; see fine_word)
  int32_t* status;
  uint32_t* ready;         // [n_mtiles] tokens published, 16 words apart
  uint32_t* abort;         // any CTA gave up on a wait
  uint4* abuf;             // each row's next A operand (W1 row of its last token), gather-ordered
#ifdef DSPARK_DRAFT_TRACE
  unsigned long long* trace;  // [gamma][n_ctas][kTraceEvents] or null
#endif
  int R, R_pad, gamma, V, rank, n_tiles, n_chunks, n_mtiles;
  int d;                   // hidden size (LM head only; 0 otherwise)
  float scale;             // log2(e) / T (1 when greedy)
  uint64_t seed;
  uint32_t round;
};

// Offsets in dynamic shared memory.  Ring stages are found by arithmetic
// (w0 + s * wstride), never by indexing an array with the stage number: a
// runtime-indexed array would put the whole plan in local memory.
struct DraftSmem {
  uint32_t w0, wstride, u0, half, bars, slots, part, wts, ev, slab, total;  // u0 and w0 1024-aligned
  __host__ __device__ uint32_t w(int s) const { return w0 + static_cast<uint32_t>(s) * wstride; }
  __host__ __device__ uint32_t u(int s) const { return u0 + static_cast<uint32_t>(s) * kDraftUBytes; }
};
__host__ __device__ inline DraftSmem draft_smem_plan(int rank) {
  DraftSmem s;
  uint32_t off = 0;
  s.w0 = off; s.wstride = 2u * kDraftWBox; off += kDraftWStages * s.wstride;  // 2 x (128 rows x 64 bf16), SW128
  s.u0 = off; off += kDraftUStages * kDraftUBytes;
  s.half = off; off += kMTile * 8;
  s.bars = off; off += 320;
  s.slots = off; off += 32;                      // the sampler's SampleSlot
  s.part = off; off += 8 * 32 * 4;               // each epilogue warp's 32 column shares
  s.wts = off; off += kMaxSampleChunks * 4;      // the leader's search weights
  s.ev = off; off += 256 * 4;                    // the previous token's W1 row
  off = (off + 127u) & ~127u;
  s.slab = off; off += (rank > 256 ? 64u * rank : 64u * 256u) + 32 * 4;  // [<=256][32] bf16 columns, then 32 U values
  s.total = off + 1024;  // alignment slack
  return s;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Relaxed (single-copy atomic, unordered) 64-bit accesses: the chunk entries
// and the sub-tile partials carry their position tag in the word itself, so a
// reader needs no ordering against other writes, only a tag that matches.
__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Waits until *word >= target (acquire).  Gives up after kWaitLimitNs or once
// any CTA has raised the abort word; then raises it too and returns false.
// One thread per waiting group polls, with a short sleep between polls, so
// that waiters do not crowd L2 while other CTAs still stream.
__device__ __forceinline__ bool wait_at_least(const uint32_t* word, uint32_t target, uint32_t* abort_word) {
  if (ld_acquire_gpu(word) >= target) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(64);
    if (ld_acquire_gpu(word) >= target) return true;
    if ((i & 15u) == 0u) {
      if (ld_relaxed_gpu(abort_word)) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicExch(abort_word, 1u);
        return false;
      }
    }
  }
}

// First item of a contiguous list of weights w[0..n) (shared memory, n <= 256)
// whose running sum (from `base`) exceeds `target`.  Each lane sums its own
// contiguous segment of ceil(n/32) items, one warp scan over the segment sums
// finds the lane that crosses, and that lane walks its segment: a single scan
// however long the list.  Rounding can leave the total at or below the target:
// then the last item with positive weight.  `before` = the running sum just
// before the returned item.
struct Crossing {
  int idx;
  float before;
};
__device__ __forceinline__ Crossing warp_crossing(const float* w, int n, float base, float target) {
  const int lane = threadIdx.x & 31;
  const int seg = (n + 31) >> 5;
  const int lo = min(n, lane * seg), hi = min(n, lo + seg);
  float mine = 0.f;
  for (int i = lo; i < hi; ++i) mine += w[i];
  const float incl = warp_incl_scan_f(mine);
  const float start = base + (incl - mine);  // running sum before this lane's segment
  const unsigned cross = __ballot_sync(0xffffffffu, base + incl > target && mine > 0.f);
  const unsigned nz = __ballot_sync(0xffffffffu, mine > 0.f);
  // the owner: the first crossing lane, else the last lane holding mass
  const int owner = cross ? __ffs(cross) - 1 : (nz ? 31 - __clz(nz) : 0);
  Crossing c = {lo, start};
  if (lane == owner) {
    float run = start;
    int found = -1, last = -1;
    float last_before = start;
    for (int i = lo; i < hi; ++i) {
      const float wi = w[i];
      if (wi > 0.f) {
        if (cross && run + wi > target) { found = i; break; }
        last = i;
        last_before = run;
      }
      run += wi;
    }
    if (found >= 0) {
      c = Crossing{found, run};
    } else if (last >= 0) {  // no crossing inside the segment (rounding): its last positive item
      c = Crossing{last, last_before};
    }
  }
  c.idx = __shfl_sync(0xffffffffu, c.idx, owner);
  c.before = __shfl_sync(0xffffffffu, c.before, owner);
  return c;
}

// The i-th tile a CTA sweeps at position `step`: forwards at even positions,
// backwards at odd ones, so that the W2 tiles a position uses last (the most
// recently used in L2) are the first the next position needs.
__device__ __forceinline__ int tile_of(int step, int i, int ntile) { return (step & 1) ? ntile - 1 - i : i; }

// First 64-column tile of chunk c when n_tiles tiles are split into n_chunks
// contiguous chunks.  32-bit: c <= kMaxSampleChunks and n_tiles < 2^18 (the
// host limits V to 2^24), so c * n_tiles < 2^26.
__device__ __forceinline__ int chunk_first_tile(int c, int n_tiles, int n_chunks) {
  return static_cast<int>(static_cast<uint32_t>(c) * static_cast<uint32_t>(n_tiles) / static_cast<uint32_t>(n_chunks));
}

// Tree reductions over 32 registers (depth 5 instead of a 31-long chain).
__device__ __forceinline__ float tree_max32(const float (&z)[32]) {
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = fmaxf(z[i], z[i + 16]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
  return t[0];
}
__device__ __forceinline__ float tree_sum32(const float (&z)[32]) {
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = z[i] + z[i + 16];
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] += t[i + w];
  return t[0];
}
// Maximum and the lowest column index attaining it (z[k] is column k).
__device__ __forceinline__ float tree_argmax32(const float (&z)[32], int* idx) {
  float t[16];
  int ix[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    // pairs (i, i + 16): the right one wins only when strictly larger
    const bool r = z[i + 16] > z[i];
    t[i] = r ? z[i + 16] : z[i];
    ix[i] = r ? i + 16 : i;
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const bool r = t[i + w] > t[i] || (t[i + w] == t[i] && ix[i + w] < ix[i]);
      t[i] = r ? t[i + w] : t[i];
      ix[i] = r ? ix[i + w] : ix[i];
    }
  *idx = ix[0];
  return t[0];
}

// Publishes request r's token x (one warp): copies W1[x] into the row's slot
// of the A-operand staging buffer, in the order the gather reads it (for each
// 16-byte piece k, the 32 rows of a lane quarter are contiguous, so a gather
// warp reads whole 128-byte lines), then lane 0 counts the token on the M-tile
// (a release fence, then a relaxed add: the ready counter's pollers pair it
// with their own acquire).
__device__ __forceinline__ void publish_token(const DraftArgs& p, int r, int step, int x) {
  if (step + 1 >= p.gamma) return;
  const int lane = threadIdx.x & 31;
  const int half_u4 = p.rank / 16;  // uint4 per half row; a row is 2 * half_u4 <= 32 of them
  if (lane < 2 * half_u4) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(x) * p.rank) + lane);
    const int rr = r % kMTile, h = lane / half_u4, k = lane - h * half_u4;
    p.abuf[((((static_cast<size_t>(r / kMTile) * 4 + (rr >> 5)) * 2 + h) * 16 + k) << 5) + (rr & 31)] = v;
  }
  __syncwarp();
  if (lane == 0) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(p.ready + 16 * (r / kMTile)) : "memory");
  }
}

// A 32-column sub-tile partial of one row, as one 64-bit word written with a
// relaxed store: the low word is the sub-tile's reference o (its maximum y in
// the log2 domain, with the low kFineTagBits mantissa bits replaced by the
// position tag), the high word is sum over the columns of 2^(y - o).  (o, sum)
// states the sub-tile's mass exactly as (max, sum) would: o moves the
// reference by at most 2^-16 relative, and the sum is taken against o itself.
// An empty sub-tile (columns past V only) has o = -FLT_MAX (tagged) and sum 0.
// The words are zeroed at the start of every call, so only this call's
// position can match a tag.
constexpr uint32_t kFineTagBits = 7;  // tags 1..kMaxGamma
constexpr uint32_t kFineTagMask = (1u << kFineTagBits) - 1u;
static_assert(kMaxGamma <= static_cast<int>(kFineTagMask), "position tags");
__device__ __forceinline__ float fine_ref(float ymax, uint32_t tag) {
  const float o = ymax > -INFINITY ? ymax : -3.4028234663852886e38f;
  return __uint_as_float((__float_as_uint(o) & ~kFineTagMask) | tag);
}
__device__ __forceinline__ unsigned long long fine_word(float o, float sum) {
  return (static_cast<unsigned long long>(__float_as_uint(sum)) << 32) | __float_as_uint(o);
}

// A chunk's partial for one row, published by its CTA in one 64-bit relaxed
// store: the low word is a float (sampled: the chunk's log2-sum-exp2
// L = max + log2(sum), greedy: its maximum), the high word carries the
// position tag (position + 1) in its top 8 bits and, greedy, the argmax in its
// low 24 bits.  The samplers poll their row's entries directly: no CTA count,
// and each chunk is folded in as soon as it lands.  Entries are zeroed at the
// start of every call, so a tag from an earlier call never matches.  No data
// is ordered behind an entry (the sub-tile partials carry their own tags), so
// it needs no release and its readers no acquire.
__device__ __forceinline__ unsigned long long chunk_entry(float lo, uint32_t tag, uint32_t idx) {
  return (static_cast<unsigned long long>((tag << 24) | idx) << 32) | __float_as_uint(lo);
}

constexpr int kEntriesPerLane = kMaxSampleChunks / 32;

// One warp waits until every chunk entry of row r carries `tag`; lane l gets
// the entries of chunks k * 32 + l in e[k] (0 past n_chunks).  Polls with a
// relaxed load per pending entry, two rounds in flight (a round is checked
// while the next is already issued, which halves the time between an entry
// landing and its round returning); gives up (false, the same in every lane,
// abort word raised) after kWaitLimitNs or on abort.
__device__ __forceinline__ bool poll_row(const DraftArgs& p, int r, uint32_t tag,
                                         unsigned long long (&e)[kEntriesPerLane]) {
  const int lane = threadIdx.x & 31;
  const unsigned long long* row = p.centry + static_cast<size_t>(r) * p.n_chunks;
  uint32_t pending = 0;
#pragma unroll
  for (int k = 0; k < kEntriesPerLane; ++k) {
    e[k] = 0ull;
    if (k * 32 + lane < p.n_chunks) pending |= 1u << k;
  }
  const uint64_t t0 = global_ns();
  unsigned long long prev[kEntriesPerLane];
#pragma unroll
  for (int k = 0; k < kEntriesPerLane; ++k) prev[k] = (pending & (1u << k)) ? ld_relaxed_gpu_u64(row + k * 32 + lane) : 0ull;
  for (uint32_t it = 0;; ++it) {
    // the next round is in flight while the previous one is checked
    unsigned long long cur[kEntriesPerLane];
#pragma unroll
    for (int k = 0; k < kEntriesPerLane; ++k) cur[k] = (pending & (1u << k)) ? ld_relaxed_gpu_u64(row + k * 32 + lane) : 0ull;
#pragma unroll
    for (int k = 0; k < kEntriesPerLane; ++k) {
      if ((pending & (1u << k)) && static_cast<uint32_t>(prev[k] >> 56) == tag) {
        e[k] = prev[k];
        pending &= ~(1u << k);
      }
      prev[k] = cur[k];
    }
    if (__all_sync(0xffffffffu, pending == 0)) break;
    if ((it & 15u) == 15u) {
      int bad = 0;
      if (lane == 0) bad = ld_relaxed_gpu(p.abort) != 0 || global_ns() - t0 > kWaitLimitNs;
      if (__shfl_sync(0xffffffffu, bad, 0)) {
        if (lane == 0) atomicExch(p.abort, 1u);
        return false;
      }
    }
  }
  __syncwarp();
  return true;
}

// One warp loads the sub-tile partials [tb2, tb2 + nsub) of row r (lane l
// gets sub-tile k * 32 + l in fw[k], 0 past nsub), re-reading any whose tag
// is not yet `tag` (a partial written before its chunk entry may still be in
// flight).  False (the same in every lane, abort word raised) after
// kWaitLimitNs or on abort.
__device__ __forceinline__ bool load_fine(const DraftArgs& p, int r, int tb2, int nsub, uint32_t tag,
                                          unsigned long long (&fw)[kEntriesPerLane]) {
  const int lane = threadIdx.x & 31;
  uint32_t pending = 0;
#pragma unroll
  for (int k = 0; k < kEntriesPerLane; ++k) {
    fw[k] = 0ull;
    if (k * 32 + lane < nsub) pending |= 1u << k;
  }
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
#pragma unroll
    for (int k = 0; k < kEntriesPerLane; ++k) {
      if (pending & (1u << k)) {
        const unsigned long long v = ld_relaxed_gpu_u64(p.fine + static_cast<size_t>(tb2 + k * 32 + lane) * p.R_pad + r);
        if ((static_cast<uint32_t>(v) & kFineTagMask) == tag) {
          fw[k] = v;
          pending &= ~(1u << k);
        }
      }
    }
    if (__all_sync(0xffffffffu, pending == 0)) return true;
    if ((it & 15u) == 15u) {
      int bad = 0;
      if (lane == 0) bad = ld_relaxed_gpu(p.abort) != 0 || global_ns() - t0 > kWaitLimitNs;
      if (__shfl_sync(0xffffffffu, bad, 0)) {
        if (lane == 0) atomicExch(p.abort, 1u);
        return false;
      }
    }
  }
}

// Greedy sampler for request r (one warp): waits for every chunk entry of the
// row, then takes the argmax, lowest index on ties.  False when the wait gave up.  Partials
// and tokens that other CTAs write during the call are read through L2
// (ld.global.cg): this SM's L1 may hold the previous position's lines.
__device__ __forceinline__ bool sample_greedy(const DraftArgs& p, int r, int step) {
  const int lane = threadIdx.x & 31;
  const size_t out = static_cast<size_t>(r) * p.gamma + step;
  unsigned long long ent[kEntriesPerLane];
  if (!poll_row(p, r, static_cast<uint32_t>(step + 1), ent)) return false;
  if (lane == 0 && r == static_cast<int>(blockIdx.x)) DRAFT_TRACE(p, step, kEvPollDone);
  float best = -INFINITY;
  int bidx = 0x7fffffff;
#pragma unroll
  for (int k = 0; k < kEntriesPerLane; ++k) {
    if (k * 32 + lane >= p.n_chunks) continue;
    const float ex = __uint_as_float(static_cast<uint32_t>(ent[k]));
    const int ei = static_cast<int>((ent[k] >> 32) & 0xFFFFFFu);
    if (ex > best || (ex == best && ex > -INFINITY && ei < bidx)) { best = ex; bidx = ei; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
  }
  if (!(fabsf(best) <= 3.4e38f) || bidx < 0 || bidx >= p.V) {
    if (lane == 0) report(p.status, DSPARK_STATUS_NONFINITE);
    bidx = 0;
  }
  if (lane == 0) {
    if (r == static_cast<int>(blockIdx.x)) DRAFT_TRACE(p, step, kEvPicked);
    p.tokens[out] = bidx;
    p.pd_tok[out] = 1.0f;
    p.logZ[out] = best;
  }
  publish_token(p, r, step, bidx);
  if (lane == 0 && r == static_cast<int>(blockIdx.x)) DRAFT_TRACE(p, step, kEvPublished);
  return true;
}

// What the leader warp hands to the other sampling warps of its CTA.
struct SampleSlot {
  int state;  // 0: gave up waiting (abort), 1: non-finite row, 2: sample
  int sstar;  // 32-column sub-tile holding the crossing
  float M, Z, target, before_s;
  int pad[2];
};
constexpr int kSlotSample = 2, kSlotNonFinite = 1, kSlotAbort = 0;

// Shared-memory pieces of the sampler (one per CTA).
struct SampleSmem {
  SampleSlot* slot;
  float* part;      // [8 warps][32 columns] shares of the bias
  float* wts;       // [kMaxSampleChunks] search weights of the leader
  float* ev;        // [256] the previous token's W1 row (fp32); with the LM head, then a chunk of h
  uint8_t* slab;    // [rank][32] bf16: W2 columns of the chosen sub-tile, then U of the sub-tile (32 fp32);
                    // with the LM head, then [256][32] chunks of W_lm's columns
  uint32_t slab_s;  // shared-space address of `slab`
  uint32_t bar;     // mbarrier of the slab copies
};

// Inverse-CDF sampler for request r, run by all 8 epilogue warps of the CTA
// (`sub` = warp index 0..7, named barrier 5).  `phase` counts the slab copies
// this CTA has waited for.  The leader warp (sub 0) waits until every chunk
// partial of the M-tile is visible, merges the chunk partials into the row's
// max M and normaliser Z (base 2), finds the chunk, then the 32-column
// sub-tile, where the running mass first exceeds u * Z (search weights in
// shared memory), and copies that sub-tile's W2 columns (one TMA box,
// rank x 32) and U values (one bulk copy) into shared memory.  Each warp then
// sums its 32 rank rows for the 32 columns (a lane per column), and the leader
// adds the shares and U and picks the token.  With the LM head (kLm) there is
// no U to copy: the warps add h . W_lm of the 32 columns instead, from
// 256-row chunks of W_lm's columns copied into the slab one after another
// (each thread stages one value of the row's h per chunk).  Returns the number
// of slab copies waited for (add it to `phase`), or -1 (the same in every
// warp: it follows the slot, read after a barrier) when the leader's wait gave
// up.  The arguments are plain values so that nothing of the sampler lives in
// local memory.
template <bool kLm>
__device__ __forceinline__ int sample_cta(const DraftArgs& p, const CUtensorMap* tm_slab,
                                          const CUtensorMap* tm_lmslab, int r, int step, int sub,
                                          const SampleSmem sm, const uint32_t phase, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const size_t out = static_cast<size_t>(r) * p.gamma + step;
  SampleSlot& slot = *sm.slot;

  // issued before the wait: the previous token's W1 entry of this lane's rank row
  const int prev_raw = step == 0 ? p.anchors[r] : __ldcg(p.tokens + out - 1);
  const int prev = (prev_raw >= 0 && prev_raw < p.V) ? prev_raw : 0;
  const int j = sub * 32 + lane;  // this lane's rank row (rank <= 256: one row per lane)
  sm.ev[j] = j < p.rank ? bf16_at(p.W1 + static_cast<size_t>(prev) * p.rank + j) : 0.f;

  if (sub == 0) {
    const float u = uniform24(p.seed, p.round, static_cast<uint64_t>(r), static_cast<uint64_t>(step), kDraftSample);
    constexpr int KC = kEntriesPerLane;
    unsigned long long ent[KC];
    const bool ok = poll_row(p, r, static_cast<uint32_t>(step + 1), ent);
    const bool traced = lane == 0 && r == static_cast<int>(blockIdx.x);
    if (traced) DRAFT_TRACE(p, step, kEvPollDone);
    int state = kSlotAbort, sstar = 0;
    float M = 0.f, Z = 0.f, target = 0.f, before_s = 0.f;
    if (ok) {
      // each chunk's log2-sum-exp2; chunks past n_chunks count as empty
      float L[KC];
#pragma unroll
      for (int k = 0; k < KC; ++k)
        L[k] = k * 32 + lane < p.n_chunks ? __uint_as_float(static_cast<uint32_t>(ent[k])) : -INFINITY;
      // two passes: the row maximum, then each chunk's mass in units of 2^M
      // (the chunk search reuses the masses as its weights)
      float m = -INFINITY;
      bool nan_seen = false;
#pragma unroll
      for (int k = 0; k < KC; ++k) {
        m = fmaxf(m, L[k]);
        nan_seen |= L[k] != L[k];
      }
      M = __any_sync(0xffffffffu, nan_seen) ? NAN : warp_max(m);
      float zs = 0.f;
#pragma unroll
      for (int k = 0; k < KC; ++k) {
        const float wk = L[k] > -INFINITY ? ex2(L[k] - M) : 0.f;
        sm.wts[k * 32 + lane] = wk;
        zs += wk;
      }
      Z = warp_sum(zs);
      if (!(fabsf(M) <= 3.4e38f) || !(Z > 0.f) || !(Z <= 3.4e38f)) {
        state = kSlotNonFinite;
      } else {
        state = kSlotSample;
        target = u * Z;
        __syncwarp();
        const Crossing cc = warp_crossing(sm.wts, p.n_chunks, 0.f, target);
        const int tb = chunk_first_tile(cc.idx, p.n_tiles, p.n_chunks);
        const int te = chunk_first_tile(cc.idx + 1, p.n_tiles, p.n_chunks);
        const int nsub = 2 * (te - tb);  // <= kMaxSampleChunks (host check)
        if (traced) DRAFT_TRACE(p, step, kEvChunkFound);
        unsigned long long fw[KC];
        const bool fine_ok = load_fine(p, r, 2 * tb, nsub, static_cast<uint32_t>(step + 1), fw);
        if (traced) DRAFT_TRACE(p, step, kEvFineLoaded);
        __syncwarp();  // every lane is done reading the chunk weights
#pragma unroll
        for (int k = 0; k < KC; ++k) {
          // each sub-tile's mass in units of 2^M
          const float o = __uint_as_float(static_cast<uint32_t>(fw[k]));
          const float sw = __uint_as_float(static_cast<uint32_t>(fw[k] >> 32));
          sm.wts[k * 32 + lane] = sw > 0.f ? sw * ex2(o - M) : 0.f;
        }
        __syncwarp();
        const Crossing cs = warp_crossing(sm.wts, nsub, cc.before, target);
        sstar = 2 * tb + cs.idx;
        before_s = cs.before;
        if (!fine_ok) state = kSlotAbort;
        if (lane == 0 && fine_ok) {
          // the previous request's readers of the slab are past the barrier
          fence_proxy_async_smem();
          // W2[:, v0 .. v0+31] (columns past V zero-filled) and U[r, step, v0 .. v0+31]
          const int v0 = sstar * kSubN;
          const uint32_t ubytes = kLm ? 0u : static_cast<uint32_t>(min(kSubN, p.V - v0)) * 4u;  // a multiple of 32
          mbar_arrive_expect_tx(sm.bar, static_cast<uint32_t>(p.rank) * 64u + ubytes);
          tma_load_2d(sm.slab_s, tm_slab, sm.bar, v0, 0, policy_evict_normal());
          if (!kLm) bulk_load(sm.slab_s + p.rank * 64, p.U + out * p.V + v0, ubytes, sm.bar, policy_evict_first());
          if (traced) DRAFT_TRACE(p, step, kEvSlabIssued);
        }
      }
    }
    if (lane == 0) {
      slot.state = state;
      slot.sstar = sstar;
      slot.M = M;
      slot.Z = Z;
      slot.target = target;
      slot.before_s = before_s;
    }
  }
  named_barrier(5, kEpiThreads);
  const int state = *reinterpret_cast<volatile int*>(&slot.state);
  const int sstar = *reinterpret_cast<volatile int*>(&slot.sstar);

  bool landed = true;
  if (state == kSlotSample) {
    landed = __all_sync(0xffffffffu, mbar_wait(sm.bar, phase & 1u, abort_flag));
    if (!landed) *abort_flag = 1;
    if (sub == 0 && lane == 0 && r == static_cast<int>(blockIdx.x)) DRAFT_TRACE(p, step, kEvSlabLanded);
    // this warp's share of the 32 bias values: lane l sums column v0 + l over
    // the warp's rank rows (W1 entries read as shared-memory broadcasts)
    float acc = 0.f;
    const uint16_t* slab = reinterpret_cast<const uint16_t*>(sm.slab);
    if (landed) {
#pragma unroll 8
      for (int k = 0; k < 32; ++k) {
        const int jk = sub * 32 + k;
        if (jk < p.rank) acc = fmaf(sm.ev[jk], __uint_as_float(static_cast<uint32_t>(slab[jk * 32 + lane]) << 16), acc);
      }
    }
    if constexpr (kLm) {
      // + h[r, step, :] . W_lm[:, v0 + lane], 256 rows of W_lm per copy
      const int v0 = sstar * kSubN;
      const int nlm = (p.d + 255) / 256;
      for (int c = 0; c < nlm; ++c) {
        named_barrier(5, kEpiThreads);  // every warp is done with the slab and ev of the previous copy
        const int jt = sub * 32 + lane, jj = c * 256 + jt;
        sm.ev[jt] = jj < p.d ? bf16_at(p.h + out * p.d + jj) : 0.f;
        if (sub == 0 && lane == 0 && !*abort_flag) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(sm.bar, 256u * 64u);  // rows past d are zero-filled
          tma_load_2d(sm.slab_s, tm_lmslab, sm.bar, v0, c * 256, policy_evict_first());
        }
        named_barrier(5, kEpiThreads);  // ev is written
        const bool got = __all_sync(0xffffffffu, mbar_wait(sm.bar, (phase + 1u + static_cast<uint32_t>(c)) & 1u,
                                                           abort_flag));
        if (!got) {
          *abort_flag = 1;
          landed = false;
        }
        if (got) {
#pragma unroll 8
          for (int k = 0; k < 32; ++k) {
            const int jk = sub * 32 + k;
            acc = fmaf(sm.ev[jk], __uint_as_float(static_cast<uint32_t>(slab[jk * 32 + lane]) << 16), acc);
          }
        }
      }
    }
    sm.part[sub * 32 + lane] = acc;
  }
  named_barrier(5, kEpiThreads);
  // A copy that never landed has set the abort flag (reported as
  // DSPARK_STATUS_TIMEOUT); the row is finished with zero shares so that every
  // warp takes the same path through the barriers.

  if (sub == 0 && state != kSlotAbort) {
    int x = 0;
    if (state == kSlotNonFinite) {
      if (lane == 0) {
        report(p.status, DSPARK_STATUS_NONFINITE);
        p.tokens[out] = 0;
        p.pd_tok[out] = 0.f;
        p.logZ[out] = NAN;
      }
    } else {
      const float M = slot.M, Z = slot.Z, target = slot.target, before_s = slot.before_s;
      float bias = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < kEpiThreads / 32; ++s2) bias += sm.part[s2 * 32 + lane];
      const int v0 = sstar * kSubN;
      const int v = v0 + lane;
      float y = -INFINITY, w = 0.f;
      if (v < p.V) {
        y = (kLm ? bias : bias + reinterpret_cast<const float*>(sm.slab + p.rank * 64)[lane]) * p.scale;
        w = ex2(y - M);
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
      x = min(v0 + pick, p.V - 1);
      if (lane == 0) {
        if (r == static_cast<int>(blockIdx.x)) DRAFT_TRACE(p, step, kEvPicked);
        p.tokens[out] = x;
        p.pd_tok[out] = __fdividef(ex2(ypick - M), Z);
        p.logZ[out] = (M + __log2f(Z)) * 0.69314718f;
      }
    }
    publish_token(p, r, step, x);
    if (lane == 0 && r == static_cast<int>(blockIdx.x)) DRAFT_TRACE(p, step, kEvPublished);
  }
  // the slot, the shares and the slab are rewritten for the next request only
  // after that request's first barrier, which the leader reaches only after
  // it has finished reading them here
  return state == kSlotAbort ? -1 : (state == kSlotSample ? (kLm ? 1 + (p.d + 255) / 256 : 1) : 0);
}

// 5-D tiled tensor load (coordinates in elements, innermost first).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0, int32_t c1,
                                            int32_t c2, int32_t c3, int32_t c4, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar), "l"(policy)
      : "memory");
}
// Shared memory -> tensor memory, 128 lanes x 256 bits (8 fp32 columns), one
// thread; completion through tcgen05.commit.  A later MMA that accumulates
// into the same columns is NOT ordered after it: wait on the commit first.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Whether the U tile starting at column v0 uses the fast 5-D layout (see
// kDraftUBytes): R a multiple of 8 and the whole tile inside the vocabulary.
__device__ __forceinline__ bool u_fast_tile(const DraftArgs& p, int v0) { return (p.R & 7) == 0 && v0 + kTileN <= p.V; }

// Copies one U tile from its shared-memory stage into 64 accumulator columns
// (8 copies of 32 bytes per row), in the tile's layout.
__device__ __forceinline__ void copy_u_tile(uint32_t stage, uint32_t dst_col, bool fast) {
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t desc = fast ? smem_desc_sw128(stage + h * 1024 + k * 32, 16, 2048)
                                 : smem_desc_sw128(stage + h * 16384 + k * 32, 16, 1024);
      tmem_cp_128x256b(dst_col + h * 32 + k * 8, desc);
    }
}

// Folds a sub-tile partial (max y, sum exp2(y - max y)) into a running one.
__device__ __forceinline__ void merge_partial(float mx, float sm, float& runM, float& runS) {
  if (mx > -INFINITY) {
    if (mx > runM) {
      runS = (runM > -INFINITY ? runS * ex2(runM - mx) : 0.f) + sm;
      runM = mx;
    } else {
      runS += sm * ex2(mx - runM);
    }
  }
}

// The call's prologue, one launch before the draft kernel: zeroes the chunk
// entries, the synchronisation words and (sampled draws) the 32-column
// partials, so that no tag from an earlier call can match, and stages each
// row's anchor W1 row in the gather order of the A-operand staging copy, so
// that position 0 gathers its A operand from L2 in whole lines like every
// later position (read straight from W1, the rows are cold HBM misses queued
// behind the producers' first TMA streams).  An anchor outside [0, V) is
// reported and replaced by token 0.
__global__ void __launch_bounds__(256) k_draft_prologue(const DraftArgs p, uint4* coarse, size_t coarse_u4,
                                                        uint4* dsync, size_t dsync_u4, uint4* fine, size_t fine_u4) {
#ifdef DSPARK_DRAFT_TRACE
  const bool stamp = p.trace && threadIdx.x == 0 && static_cast<int>(blockIdx.x) < p.n_chunks * p.n_mtiles;
  if (stamp) p.trace[static_cast<size_t>(blockIdx.x) * kTraceEvents + kEvProStart] = global_ns();
#endif
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nth = static_cast<size_t>(gridDim.x) * blockDim.x;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (size_t i = tid; i < coarse_u4; i += nth) coarse[i] = z;
  for (size_t i = tid; i < dsync_u4; i += nth) dsync[i] = z;
  for (size_t i = tid; i < fine_u4; i += nth) fine[i] = z;
  const int half_u4 = p.rank / 16;  // uint4 (8 bf16) per half of a W1 row
  const size_t staged = static_cast<size_t>(p.R) * 32;
  for (size_t i = tid; i < staged; i += nth) {
    const int r = static_cast<int>(i >> 5), u = static_cast<int>(i & 31);
    if (u >= 2 * half_u4) continue;
    int tok = p.anchors[r];
    if (tok < 0 || tok >= p.V) {
      if (u == 0) report(p.status, DSPARK_STATUS_BAD_TOKEN);
      tok = 0;
    }
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(tok) * p.rank) + u);
    const int rr = r % kMTile, h = u / half_u4, k = u - h * half_u4;
    p.abuf[((((static_cast<size_t>(r / kMTile) * 4 + (rr >> 5)) * 2 + h) * 16 + k) << 5) + (rr & 31)] = v;
  }
#ifdef DSPARK_DRAFT_TRACE
  __syncthreads();
  if (stamp) p.trace[static_cast<size_t>(blockIdx.x) * kTraceEvents + kEvProEnd] = global_ns();
#endif
}

// kLm: the fused LM head.  U is not read: each pair's accumulators start from
// h_j . W_lm, computed by the same MMAs over d more rank rows (A = h rows of
// the M-tile by TMA through the U stages, B = W_lm K-chunks through the W2
// ring), and then take the bias on top.  tm_u5 and tm_u3 are then the W_lm
// K-chunk and h maps, and tm_lmslab the sampler's W_lm column map.
template <bool kGreedy, bool kLm>
__global__ void __launch_bounds__(kDraftKThreads, 1)
    k_markov_draft(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_u5,
                   const __grid_constant__ CUtensorMap tm_u3, const __grid_constant__ CUtensorMap tm_slab,
                   const __grid_constant__ CUtensorMap tm_lmslab, const DraftArgs p) {
  if (threadIdx.x == 0) DRAFT_TRACE(p, 0, kEvLaunch);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const DraftSmem plan = draft_smem_plan(p.rank);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mtile = blockIdx.x % p.n_mtiles;
  const int chunk = blockIdx.x / p.n_mtiles;
  const int r0 = mtile * kMTile;
  const int rows_valid = min(kMTile, p.R - r0);
  const int t_begin = chunk_first_tile(chunk, p.n_tiles, p.n_chunks);
  const int t_end = chunk_first_tile(chunk + 1, p.n_tiles, p.n_chunks);
  const int ntile = t_end - t_begin;
  const int total_tiles = ntile * p.gamma;

  const uint32_t bar_wfull = base + plan.bars;               // [kDraftWStages]
  const uint32_t bar_wempty = bar_wfull + 8 * kDraftWStages;  // [kDraftWStages]
  const uint32_t bar_ufull = bar_wempty + 8 * kDraftWStages;  // [kDraftUStages]
  const uint32_t bar_uempty = bar_ufull + 8 * kDraftUStages;  // [kDraftUStages]
  const uint32_t bar_tfull = bar_uempty + 8 * kDraftUStages;   // [kDraftAccPairs]
  const uint32_t bar_tempty = bar_tfull + 8 * kDraftAccPairs;  // [kDraftAccPairs]
  const uint32_t bar_ucopied = bar_tempty + 8 * kDraftAccPairs;  // [kDraftAccPairs] U copied into the pair
  const uint32_t bar_slab = bar_ucopied + 8 * kDraftAccPairs;   // the sampler's slab copies
  const uint32_t bar_drain = bar_slab + 8;                      // the MMA issuer's last commit on abort
  const uint32_t bar_cdrain = bar_drain + 8;                    // the copier's last commit
  constexpr uint32_t kBarBytes = 16 * (kDraftWStages + kDraftUStages) + 24 * kDraftAccPairs + 24;
  static_assert(kBarBytes + 8 <= 320, "barrier block");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + plan.bars + kBarBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + plan.bars + kBarBytes + 4);
  float2* s_half = reinterpret_cast<float2*>(gbase + plan.half);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDraftWStages; ++s) {
      mbar_init(bar_wfull + 8 * s, 1);
      mbar_init(bar_wempty + 8 * s, 1);
    }
    for (int s = 0; s < kDraftUStages; ++s) {
      mbar_init(bar_ufull + 8 * s, 1);
      mbar_init(bar_uempty + 8 * s, 1);  // the copier's commit
    }
    for (int s = 0; s < kDraftAccPairs; ++s) {
      mbar_init(bar_tfull + 8 * s, 1);
      mbar_init(bar_tempty + 8 * s, 8);
      mbar_init(bar_ucopied + 8 * s, 1);
    }
    mbar_init(bar_slab, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_cdrain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tm_w2);
    if (kLm || (p.R & 7) == 0) prefetch_tensormap(&tm_u5);
    prefetch_tensormap(&tm_u3);
    prefetch_tensormap(&tm_slab);
    if (kLm) prefetch_tensormap(&tm_lmslab);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kDraftTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tmem_a = tmem_base + kDraftACol;  // A operand columns
  if (threadIdx.x == 0) DRAFT_TRACE(p, 0, kEvStart);
  // tile i of a position belongs to pair i / 2; pair gp of the call uses
  // accumulator pair gp % kDraftAccPairs and W2 K-chunks g = gp * nkc + kc,
  // in ring stage g % kDraftWStages
  const int npair = (ntile + 1) >> 1;
  // W2 K-chunks of a pair: kc_rows rank rows each (the TMA box height), the
  // last one partial when the rank is not a multiple of it (rows past the
  // rank are zero-filled and skipped by the MMA)
  const int kc_rows = min(kDraftKChunk, p.rank);
  const int nkc = (p.rank + kc_rows - 1) / kc_rows;
  const uint32_t w_box = static_cast<uint32_t>(kc_rows) * 128u;  // bytes of one 64-column box
  // with the LM head, a pair first takes nkl K-chunks of W_lm (d % 128 == 0),
  // then the nkc of W2: nkw ring stages per pair in all
  const int nkl = kLm ? p.d / kDraftKChunk : 0;
  const int nkw = nkl + nkc;
  // with the LM head, pairs go through the MMA two at a time (a group), so
  // that each h K-chunk is loaded once for both: a group's ring stages are
  // its W_lm chunks, the two pairs' interleaved chunk by chunk, then the W2
  // chunks of its first pair, then of its second.  Group m of a position
  // holds pairs 2m and 2m + 1; without the LM head a group is one pair.
  constexpr int kGroup = kLm ? 2 : 1;
  const int ngroup = (npair + kGroup - 1) / kGroup;

  if (warp == 0) {
    // ---------------------------------------------------------- W2 producer (all positions, lane 0)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_lm = policy_evict_first();
      uint32_t wlast = 0;  // per stage s: bit 2s = filled, bit 2s + 1 = parity of its last fill
      bool ok = true;
      for (int step = 0; step < p.gamma && ok; ++step) {
        for (int j0 = 0; j0 < npair && ok; j0 += kGroup) {
          const int nb = min(kGroup, npair - j0);
          for (int t = 0; t < nb * nkw; ++t) {
            // the group's t-th ring stage: W_lm chunk kc of member b, or W2 chunk kw of member b
            int b, kc, kw;
            if (t < nkl * nb) {
              b = t % nb;
              kc = t / nb;
              kw = -1;
            } else {
              b = (t - nkl * nb) / nkc;
              kw = t - nkl * nb - b * nkc;
              kc = -1;
            }
            const int j = j0 + b;
            const bool two = 2 * j + 1 < ntile;
            const int va = (t_begin + tile_of(step, 2 * j, ntile)) * kTileN;
            const int vb = two ? (t_begin + tile_of(step, 2 * j + 1, ntile)) * kTileN : 0;
            const int g = (step * npair + j0) * nkw + t;
            const int sw = g % kDraftWStages;
            const uint32_t par = static_cast<uint32_t>(g / kDraftWStages) & 1u;
            if (!mbar_wait(bar_wempty + 8 * sw, par ^ 1u, abort_flag)) {
              *abort_flag = 1;
              ok = false;
              break;
            }
            if (kLm && kc >= 0) {
              // W_lm rows [kc * 128, kc * 128 + 128) of both tiles (streamed: evict first)
              mbar_arrive_expect_tx(bar_wfull + 8 * sw, (two ? 2u : 1u) * kDraftWBox);
              tma_load_2d(base + plan.w(sw), &tm_u5, bar_wfull + 8 * sw, va, kc * kDraftKChunk, pol_lm);
              if (two) tma_load_2d(base + plan.w(sw) + kDraftWBox, &tm_u5, bar_wfull + 8 * sw, vb, kc * kDraftKChunk, pol_lm);
            } else {
              // rank rows [kw * kc_rows, (kw + 1) * kc_rows) of both tiles; rows past the
              // rank and columns past V are zero-filled
              mbar_arrive_expect_tx(bar_wfull + 8 * sw, (two ? 2u : 1u) * w_box);
              tma_load_2d(base + plan.w(sw), &tm_w2, bar_wfull + 8 * sw, va, kw * kc_rows, pol_w);
              if (two) tma_load_2d(base + plan.w(sw) + w_box, &tm_w2, bar_wfull + 8 * sw, vb, kw * kc_rows, pol_w);
            }
            wlast = (wlast & ~(3u << (2 * sw))) | ((1u | (par << 1)) << (2 * sw));
          }
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA exits
        const uint64_t t0 = global_ns();
        for (int s = 0; s < kDraftWStages; ++s)
          if ((wlast >> (2 * s)) & 1u)
            while (!mbar_try_wait(bar_wfull + 8 * s, (wlast >> (2 * s + 1)) & 1u) && global_ns() - t0 < kWaitLimitNs) {
            }
      }
    }
    __syncwarp();
  } else if (kLm && warp == kUWarp) {
    // ---------------------------------------------------------- h producer (LM head; all positions, lane 0)
    // each LM K-chunk of a group of pairs: the M-tile's h rows at this
    // position, K elements [kc * 128, kc * 128 + 128) as two 64-element SW128
    // boxes (rows past R zero-filled), into a U stage
    if (lane == 0) {
      const uint64_t pol_h = policy_evict_last();  // reread by every group of the position
      int hfilled = 0;
      for (int gg = 0; gg < ngroup * p.gamma && !*abort_flag; ++gg) {
        const int step = gg / ngroup;
        for (int kc = 0; kc < nkl; ++kc) {
          const int gh = gg * nkl + kc, hs = gh % kDraftUStages;
          if (!mbar_wait(bar_uempty + 8 * hs, ((gh / kDraftUStages) & 1) ^ 1, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(bar_ufull + 8 * hs, kDraftUBytes);
          tma_load_3d(base + plan.u(hs), &tm_u3, bar_ufull + 8 * hs, kc * kDraftKChunk, step, r0, pol_h);
          tma_load_3d(base + plan.u(hs) + kDraftUBytes / 2, &tm_u3, bar_ufull + 8 * hs, kc * kDraftKChunk + 64, step, r0,
                      pol_h);
          ++hfilled;
        }
      }
      if (*abort_flag) {
        const uint64_t t0 = global_ns();
        for (int i = max(0, hfilled - kDraftUStages); i < hfilled; ++i)
          while (!mbar_try_wait(bar_ufull + 8 * (i % kDraftUStages), (i / kDraftUStages) & 1) &&
                 global_ns() - t0 < kWaitLimitNs) {
          }
      }
    }
    __syncwarp();
  } else if (kLm && warp == kCopyWarp) {
    // no U to copy: the MMA issuer waits for the epilogue's drain itself
  } else if (warp == kUWarp) {
    // ---------------------------------------------------------- U producer (all positions, lane 0)
    if (lane == 0) {
      const uint64_t pol_u = policy_evict_first();
      int ufilled = 0;
      for (int it = 0; it < total_tiles; ++it) {
        const int step = it / ntile;
        const int v0 = (t_begin + tile_of(step, it - step * ntile, ntile)) * kTileN;
        const int su = it % kDraftUStages;
        if (!mbar_wait(bar_uempty + 8 * su, ((it / kDraftUStages) & 1) ^ 1, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        // rows past R and columns past V are zero-filled
        mbar_arrive_expect_tx(bar_ufull + 8 * su, kDraftUBytes);
        if (u_fast_tile(p, v0)) {
          tma_load_5d(base + plan.u(su), &tm_u5, bar_ufull + 8 * su, 0, 0, v0 / 32, r0 / 8, step, pol_u);
        } else {
          tma_load_3d(base + plan.u(su), &tm_u3, bar_ufull + 8 * su, v0, step, r0, pol_u);
          tma_load_3d(base + plan.u(su) + 16384, &tm_u3, bar_ufull + 8 * su, v0 + 32, step, r0, pol_u);
        }
        ++ufilled;
      }
      if (*abort_flag) {
        const uint64_t t0 = global_ns();
        for (int i = max(0, ufilled - kDraftUStages); i < ufilled; ++i)
          while (!mbar_try_wait(bar_ufull + 8 * (i % kDraftUStages), (i / kDraftUStages) & 1) &&
                 global_ns() - t0 < kWaitLimitNs) {
          }
      }
    }
    __syncwarp();
  } else if (warp == kCopyWarp) {
    // ---------------------------------------------------------- U copier (all positions, lane 0)
    // Each tile's U goes from its ring stage into its accumulator pair once the
    // epilogue has drained that pair's previous use; the commit after a tile
    // frees its stage, the one after a pair's last tile lets the MMA in.
    if (lane == 0) {
      int issued = 0;
      for (int gp = 0; gp < npair * p.gamma; ++gp) {
        const int step = gp / npair, j = gp - step * npair, pa = gp % kDraftAccPairs;
        if (!mbar_wait(bar_tempty + 8 * pa, ((gp / kDraftAccPairs) & 1) ^ 1, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after_sync();
        const int ntp = 2 * j + 1 < ntile ? 2 : 1;
        bool ok = true;
        for (int t = 0; t < ntp; ++t) {
          const int it = step * ntile + 2 * j + t;
          const int su = it % kDraftUStages;
          if (!mbar_wait(bar_ufull + 8 * su, (it / kDraftUStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const int v0 = (t_begin + tile_of(step, 2 * j + t, ntile)) * kTileN;
          copy_u_tile(base + plan.u(su), tmem_base + static_cast<uint32_t>(pa * 2 * kTileN + t * kTileN),
                      u_fast_tile(p, v0));
          umma_commit(bar_uempty + 8 * su);
          issued = 1;
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        umma_commit(bar_ucopied + 8 * pa);
        if (j == 0) DRAFT_TRACE(p, step, kEvCopyFirst);
        if (j == 2) DRAFT_TRACE(p, step, kEvCopyThird);
      }
      if (issued) {
        // every copy this thread issued is complete before tensor memory is freed
        umma_commit(bar_cdrain);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(bar_cdrain, 0) && global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- UMMA issuer
    const uint32_t idesc_pair = idesc_bf16_f32(kMTile, 2 * kTileN, false, true);
    const uint32_t idesc_one = idesc_bf16_f32(kMTile, kTileN, false, true);
    int issued = 0;  // any MMA issued
    if constexpr (kLm) {
      // group m's LM part: the accumulators of its one or two pairs start from
      // h . W_lm (A = h rows in a U stage, K-major SW128: K-steps 32 bytes
      // apart in each 64-element box, shared by both pairs)
      auto lm_group = [&](int step, int m) -> bool {
        const int j0 = kGroup * m, nb = min(kGroup, npair - j0);
        uint32_t dacc[kGroup], idsc[kGroup];
#pragma unroll
        for (int b = 0; b < kGroup; ++b) {
          if (b >= nb) break;
          const int gp = step * npair + j0 + b, pa = gp % kDraftAccPairs;
          if (!mbar_wait(bar_tempty + 8 * pa, ((gp / kDraftAccPairs) & 1) ^ 1, abort_flag)) return false;
          idsc[b] = 2 * (j0 + b) + 1 < ntile ? idesc_pair : idesc_one;
          dacc[b] = tmem_base + static_cast<uint32_t>(pa * 2 * kTileN);
        }
        tc_fence_after_sync();
        for (int kc = 0; kc < nkl; ++kc) {
          const int gh = (step * ngroup + m) * nkl + kc, hs = gh % kDraftUStages;
          if (!mbar_wait(bar_ufull + 8 * hs, (gh / kDraftUStages) & 1, abort_flag)) return false;
          int sw[kGroup];
#pragma unroll
          for (int b = 0; b < kGroup; ++b) {
            if (b >= nb) break;
            const int g = (step * npair + j0) * nkw + kc * nb + b;
            sw[b] = g % kDraftWStages;
            if (!mbar_wait(bar_wfull + 8 * sw[b], static_cast<uint32_t>(g / kDraftWStages) & 1u, abort_flag))
              return false;
          }
          tc_fence_after_sync();
          const uint32_t a0 = base + plan.u(hs);
#pragma unroll
          for (int b = 0; b < kGroup; ++b) {
            if (b >= nb) break;
            const uint64_t bdesc = smem_desc_sw128(base + plan.w(sw[b]), kDraftWBox, 1024);
#pragma unroll
            for (int q4 = 0; q4 < kDraftKChunk / 16; ++q4)
              umma_bf16(dacc[b], smem_desc_sw128(a0 + (q4 >> 2) * (kDraftUBytes / 2) + (q4 & 3) * 32, 16, 1024),
                        bdesc + static_cast<uint64_t>(q4 * 128), idsc[b], (kc | q4) != 0 ? 1u : 0u);
          }
#pragma unroll
          for (int b = 0; b < kGroup; ++b) {
            if (b >= nb) break;
            umma_commit(bar_wempty + 8 * sw[b]);
          }
          umma_commit(bar_uempty + 8 * hs);
          issued = 1;
        }
        return true;
      };
      // member b of group m: its bias part (A = W1 rows in tensor memory), then the pair is done
      auto bias_member = [&](int step, int m, int b) -> bool {
        const int j0 = kGroup * m, nb = min(kGroup, npair - j0), j = j0 + b;
        const int gp = step * npair + j, pa = gp % kDraftAccPairs;
        const uint32_t idesc = 2 * j + 1 < ntile ? idesc_pair : idesc_one;
        const uint32_t d = tmem_base + static_cast<uint32_t>(pa * 2 * kTileN);
        for (int kw = 0; kw < nkc; ++kw) {
          const int g = (step * npair + j0) * nkw + nkl * nb + b * nkc + kw, sw = g % kDraftWStages;
          if (!mbar_wait(bar_wfull + 8 * sw, static_cast<uint32_t>(g / kDraftWStages) & 1u, abort_flag)) return false;
          tc_fence_after_sync();
          const int ks0 = kw * (kc_rows / 16), nks = min(kc_rows, p.rank - kw * kc_rows) / 16;
          const uint64_t desc0 = smem_desc_sw128(base + plan.w(sw), w_box, 1024);
#pragma unroll
          for (int q4 = 0; q4 < kDraftKChunk / 16; ++q4)
            if (q4 < nks) umma_bf16_ts(d, tmem_a + (ks0 + q4) * 8, desc0 + static_cast<uint64_t>(q4 * 128), idesc, 1u);
          umma_commit(bar_wempty + 8 * sw);
          issued = 1;
        }
        umma_commit(bar_tfull + 8 * pa);
        return true;
      };
      for (int step = 0; step < p.gamma; ++step) {
        // the first group's LM part needs no A operand: it runs while the
        // previous position's samplers are at work
        if (lane == 0 && !*abort_flag && !lm_group(step, 0)) *abort_flag = 1;
        __syncwarp();
        named_barrier(2, kEpiThreads + 32);  // this position's A operand is in tensor memory
        tc_fence_after_sync();
        if (lane == 0 && !*abort_flag) {
          for (int m = 0; m < ngroup; ++m) {
            bool ok = m == 0 || lm_group(step, m);
            const int nb = min(kGroup, npair - kGroup * m);
            for (int b = 0; b < nb && ok; ++b) ok = bias_member(step, m, b);
            if (!ok) {
              *abort_flag = 1;
              break;
            }
          }
        }
        __syncwarp();
      }
    } else
    for (int step = 0; step < p.gamma; ++step) {
      named_barrier(2, kEpiThreads + 32);  // this position's A operand is in tensor memory
      tc_fence_after_sync();
      if (lane == 0 && !*abort_flag) {
        bool ok = true;
        for (int j = 0; j < npair && ok; ++j) {
          const int gp = step * npair + j, pa = gp % kDraftAccPairs;
          // the pair's U is in its accumulator (the copier waited for the drain)
          if (!mbar_wait(bar_ucopied + 8 * pa, (gp / kDraftAccPairs) & 1, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after_sync();
          const uint32_t idesc = 2 * j + 1 < ntile ? idesc_pair : idesc_one;
          const uint32_t d = tmem_base + static_cast<uint32_t>(pa * 2 * kTileN);
          for (int kc = 0; kc < nkc; ++kc) {
            const int g = gp * nkc + kc;
            const int sw = g % kDraftWStages;
            if (!mbar_wait(bar_wfull + 8 * sw, static_cast<uint32_t>(g / kDraftWStages) & 1u, abort_flag)) {
              *abort_flag = 1;
              ok = false;
              break;
            }
            tc_fence_after_sync();
            // K-steps of 16 rank rows in this chunk; N-direction atom stride
            // (LBO) = one box: the pair's second tile
            const int ks0 = kc * (kc_rows / 16), nks = min(kc_rows, p.rank - kc * kc_rows) / 16;
            const uint64_t desc0 = smem_desc_sw128(base + plan.w(sw), w_box, 1024);
#pragma unroll
            for (int q4 = 0; q4 < kDraftKChunk / 16; ++q4)
              if (q4 < nks)  // + q4 * 2048 bytes: 16 rows of 128 bytes
                umma_bf16_ts(d, tmem_a + (ks0 + q4) * 8, desc0 + static_cast<uint64_t>(q4 * 128), idesc, 1u);  // onto U
            umma_commit(bar_wempty + 8 * sw);
            issued = 1;
          }
          if (ok) umma_commit(bar_tfull + 8 * pa);
        }
      }
      __syncwarp();
    }
    if (lane == 0 && *abort_flag && issued > 0) {
      // every MMA this thread issued is complete before tensor memory is freed
      umma_commit(bar_drain);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(bar_drain, 0) && global_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue + sampler warps 2..9
    const int q = warp & 3;         // tensor-memory lane quarter of this warp
    const int h = (warp - 2) >> 2;  // 32-column half of each tile; half of A's columns
    const int row = q * 32 + lane;
    const int r = r0 + row;
    const bool valid = row < rows_valid;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int half_u4 = p.rank / 16;  // uint4 (8 bf16) per half of a W1 row
    SampleSmem ssm;
    ssm.slot = reinterpret_cast<SampleSlot*>(gbase + plan.slots);
    ssm.part = reinterpret_cast<float*>(gbase + plan.part);
    ssm.wts = reinterpret_cast<float*>(gbase + plan.wts);
    ssm.ev = reinterpret_cast<float*>(gbase + plan.ev);
    ssm.slab = gbase + plan.slab;
    ssm.slab_s = base + plan.slab;
    ssm.bar = bar_slab;
    uint32_t slab_phase = 0;  // slab copies this CTA has waited for

    for (int step = 0; step < p.gamma; ++step) {
      // ---- gather: W1[x_{step-1}] of this row, K elements [h*rank/2, (h+1)*rank/2),
      // once every token of this M-tile's previous position is published (one
      // poller per CTA).  Every abort decision is warp-uniform: tensor-memory
      // loads and stores are warp-collective.
      if (step > 0) {
        if (threadIdx.x == 64 && !*abort_flag &&
            !wait_at_least(p.ready + 16 * mtile, static_cast<uint32_t>(rows_valid * step), p.abort))
          *abort_flag = 1;
        if (threadIdx.x == 64) DRAFT_TRACE(p, step, kEvReadySeen);
        named_barrier(4, kEpiThreads);
      }
      if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
        uint32_t a[64];  // all loads first, then the tensor-memory stores
        {
          // the staged W1 rows of this M-tile's previous tokens (the anchors at
          // position 0, staged by the prologue; later, written by other CTAs:
          // through L2)
          const uint4* src = p.abuf + ((((static_cast<size_t>(mtile) * 4 + q) * 2 + h) * 16) << 5) + lane;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            uint4 wv = make_uint4(0, 0, 0, 0);
            if (valid && k < half_u4) wv = __ldcg(src + (k << 5));
            a[4 * k] = wv.x; a[4 * k + 1] = wv.y; a[4 * k + 2] = wv.z; a[4 * k + 3] = wv.w;
          }
        }
        const uint32_t dst = tmem_a + lane_off + static_cast<uint32_t>(h * 4 * half_u4);
        const uint32_t(&a0)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&a[0]);
        const uint32_t(&a1)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&a[32]);
        if (half_u4 >= 8) {
          tmem_st_32x32(dst, a0);
          if (half_u4 == 16) tmem_st_32x32(dst + 32, a1);
          else if (half_u4 == 12) tmem_st_32x16(dst + 32, a1);
        } else {
          tmem_st_32x16(dst, a0);  // rank 64
        }
        tmem_wait_st();
      }
      tc_fence_before_sync();
      named_barrier(2, kEpiThreads + 32);
      if (threadIdx.x == 64) DRAFT_TRACE(p, step, kEvAReady);

      // ---- tiles
      float runM = -INFINITY, runS = 0.f;  // running (max, sum exp2) of this warp's half of the chunk
      int runIdx = 0;                      // greedy: running argmax
      if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
        // one pair of tiles per iteration: both accumulators are loaded
        // together and the two tiles' arithmetic is interleaved
        for (int j = 0; j < npair; ++j) {
          const int i0 = 2 * j;
          const bool two = i0 + 1 < ntile;
          const int gp = step * npair + j, pa = gp % kDraftAccPairs;
          if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8 * pa, (gp / kDraftAccPairs) & 1, abort_flag))) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after_sync();
          if (j == 0 && threadIdx.x == 64) DRAFT_TRACE(p, step, kEvFirstAcc);
          uint32_t a0[32], a1[32];
          const uint32_t tacc = tmem_base + lane_off + static_cast<uint32_t>(2 * pa * kTileN + h * kSubN);
          tmem_ld_32x32_nowait(tacc, a0);
          tmem_ld_32x32_nowait(tacc + kTileN, a1);  // the second tile (not used when the pair has one)
          tmem_wait_ld_tied(a0);
          tmem_wait_ld_tied(a1);
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty + 8 * pa);
          // z = U + bias: the accumulators started from U
          float z0[32], z1[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            z0[k] = __uint_as_float(a0[k]);
            z1[k] = __uint_as_float(a1[k]);
          }

          // z = bias + U of 32 columns of each tile; columns past V only in the
          // last tile, and none at all for a missing second tile
          const int ti0 = tile_of(step, i0, ntile);
          const int ti1 = two ? tile_of(step, i0 + 1, ntile) : ti0;
          const int v00 = (t_begin + ti0) * kTileN + h * kSubN;
          const int v01 = (t_begin + ti1) * kTileN + h * kSubN;
          const int ncol0 = min(kSubN, p.V - v00);
          const int ncol1 = two ? min(kSubN, p.V - v01) : 0;
          if (ncol0 < kSubN) {
#pragma unroll
            for (int k = 0; k < 32; ++k) z0[k] = k < ncol0 ? z0[k] : -INFINITY;
          }
          if (ncol1 < kSubN) {
#pragma unroll
            for (int k = 0; k < 32; ++k) z1[k] = k < ncol1 ? z1[k] : -INFINITY;
          }
          if constexpr (kGreedy) {
            int k0, k1;
            const float mx0 = tree_argmax32(z0, &k0);
            const float mx1 = tree_argmax32(z1, &k1);
            const int ix0 = v00 + k0, ix1 = v01 + k1;
            if (mx0 > runM || (mx0 == runM && ix0 < runIdx)) { runM = mx0; runIdx = ix0; }
            if (two && (mx1 > runM || (mx1 == runM && ix1 < runIdx))) { runM = mx1; runIdx = ix1; }
          } else {
            // y = z * log2(e)/T; partial (o, sum 2^(y - o)) with o the tagged
            // maximum (fine_ref); an all-empty sub-tile gives sum 0
            const uint32_t ftag = static_cast<uint32_t>(step + 1);
            const float o0 = fine_ref(tree_max32(z0) * p.scale, ftag), o1 = fine_ref(tree_max32(z1) * p.scale, ftag);
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              z0[k] = ex2(fmaf(z0[k], p.scale, -o0));
              z1[k] = ex2(fmaf(z1[k], p.scale, -o1));
            }
            const float sm0 = tree_sum32(z0), sm1 = tree_sum32(z1);
            const size_t f0 = static_cast<size_t>(2 * (t_begin + ti0) + h) * p.R_pad + r;
            const size_t f1 = static_cast<size_t>(2 * (t_begin + ti1) + h) * p.R_pad + r;
            if (valid) st_relaxed_gpu_u64(p.fine + f0, fine_word(o0, sm0));
            if (valid && two) st_relaxed_gpu_u64(p.fine + f1, fine_word(o1, sm1));
            merge_partial(o0, sm0, runM, runS);
            merge_partial(o1, sm1, runM, runS);
          }
        }
      }
      if (threadIdx.x == 64) DRAFT_TRACE(p, step, kEvTilesDone);
      // ---- combine the two column halves of this CTA's chunk
      if (h == 1) s_half[row] = kGreedy ? make_float2(runM, __int_as_float(runIdx)) : make_float2(runM, runS);
      named_barrier(1, kEpiThreads);
      if (h == 0 && valid && !*abort_flag) {
        // publish the row's chunk entry: one relaxed store (its tag is all a
        // reader checks)
        const float2 o = s_half[row];
        unsigned long long ent;
        if constexpr (kGreedy) {
          const int oi = __float_as_int(o.y);
          if (o.x > runM || (o.x == runM && oi < runIdx)) { runM = o.x; runIdx = oi; }
          ent = chunk_entry(runM, static_cast<uint32_t>(step + 1), static_cast<uint32_t>(runIdx));
        } else {
          const float Mx = fmaxf(runM, o.x);
          float S = 0.f;
          if (Mx > -INFINITY) {
            if (runM > -INFINITY) S += runS * ex2(runM - Mx);
            if (o.x > -INFINITY) S += o.y * ex2(o.x - Mx);
          }
          // a NaN sum stays NaN in L, so that the sampler reports the row
          const float L = Mx > -INFINITY ? Mx + __log2f(S) : -INFINITY;
          ent = chunk_entry(L, static_cast<uint32_t>(step + 1), 0u);
        }
        st_relaxed_gpu_u64(p.centry + static_cast<size_t>(r) * p.n_chunks + chunk, ent);
      }
      if (threadIdx.x == 64) DRAFT_TRACE(p, step, kEvEntry);

      // ---- sample this CTA's requests once every chunk of their M-tile is done
      if constexpr (kGreedy) {
        // one warp per request
        for (int rr = blockIdx.x + gridDim.x * (warp - 2); rr < p.R; rr += gridDim.x * (kEpiThreads / 32)) {
          if (__any_sync(0xffffffffu, *abort_flag != 0) || !sample_greedy(p, rr, step)) {
            *abort_flag = 1;
            break;
          }
        }
      } else {
        // all 8 epilogue warps on each of this CTA's requests in turn
        for (int rr = blockIdx.x; rr < p.R; rr += gridDim.x) {
          const int rc = sample_cta<kLm>(p, &tm_slab, &tm_lmslab, rr, step, warp - 2, ssm, slab_phase, abort_flag);
          if (rc < 0) {
            *abort_flag = 1;
            break;
          }
          slab_phase += static_cast<uint32_t>(rc);
        }
      }
    }
  }
  if (*abort_flag && threadIdx.x == 0) report(p.status, DSPARK_STATUS_TIMEOUT);
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) DRAFT_TRACE(p, 0, kEvEnd);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kDraftTmemCols);
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

// W2 [rank, V] bf16, box 64 columns x min(128, rank) rows with 128-byte
// swizzle: one K-chunk of one tile of the draft's W2 ring (the MN-major SW128
// operand layout of the UMMA).
static int encode_w2_kchunk_map(CUtensorMap* tm, const uint16_t* W2, int V, int rank) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(rank)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileN), static_cast<cuuint32_t>(std::min(kDraftKChunk, rank))};
  cuuint32_t estr[2] = {1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W2), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// W2 [rank, V] bf16 again, box 32 x rank without swizzle: the sampler's copy
// of the 32 columns of one sub-tile ([rank][32], 64-byte rows).
int encode_w2_slab_map(CUtensorMap* tm, const uint16_t* W2, int V, int rank) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(rank)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kSubN), static_cast<cuuint32_t>(rank)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W2), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// U [R, gamma, V] fp32 as a 5-D tensor for the fast tile layout (R % 8 == 0):
// (32 columns, 8 rows of a row group, 32-column block, row group, position),
// box {32, 8, 2, 16, 1} with 128-byte swizzle: one 64-column tile of 128 rows
// per load, each row's 256 bytes fetched together, half h of row group g at
// byte g * 2048 + h * 1024.  Only whole tiles are loaded through it.
static int encode_u_fast_map(CUtensorMap* tm, const float* U, int R, int gamma, int V) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  const cuuint64_t row = static_cast<cuuint64_t>(V) * 4 * gamma;  // bytes between requests
  cuuint64_t dims[5] = {32, 8, static_cast<cuuint64_t>(V / 32), static_cast<cuuint64_t>(R / 8),
                        static_cast<cuuint64_t>(gamma)};
  cuuint64_t strides[4] = {row, 128, 8 * row, static_cast<cuuint64_t>(V) * 4};
  cuuint32_t box[5] = {32, 8, 2, static_cast<cuuint32_t>(kMTile / 8), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float*>(U), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// U [R, gamma, V] fp32 as a 3-D tensor (x = vocabulary, y = position,
// z = request), box {32, 1, 128} with 128-byte swizzle: one 32-column half of
// a tile (the general layout), columns past V and rows past R zero-filled.
static int encode_u_half_map(CUtensorMap* tm, const float* U, int R, int gamma, int V) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(gamma), static_cast<cuuint64_t>(R)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(V) * 4, static_cast<cuuint64_t>(V) * 4 * gamma};
  cuuint32_t box[3] = {32, 1, static_cast<cuuint32_t>(kMTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(U), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? DSPARK_OK : DSPARK_ERR_CUDA;
}

#ifdef DSPARK_DRAFT_TRACE
static unsigned long long* g_trace = nullptr;
static size_t g_trace_bytes = 0;
#endif

int encode_u_rows_map(CUtensorMap* tm, const float* U, int R, int gamma, int V) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(R) * static_cast<cuuint64_t>(gamma)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileN), 1};
  cuuint32_t estr[2] = {1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(U), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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

// h [R, gamma, d] bf16 as a 3-D tensor (d, position, request), box
// {64, 1, 128} with 128-byte swizzle: 64 hidden elements of one position for
// the 128 rows of an M-tile, the K-major SW128 layout of the UMMA A operand.
static int encode_h_map(CUtensorMap* tm, const uint16_t* h, int R, int gamma, int d) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(gamma), static_cast<cuuint64_t>(R)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(gamma) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kMTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(h), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// W_lm [d, V] bf16, box 32 columns x 256 rows without swizzle: one chunk of
// the 32 columns the sampler recomputes ([256][32], 64-byte rows; rows past d
// zero-filled).
static int encode_lm_slab_map(CUtensorMap* tm, const uint16_t* W_lm, int V, int d) {
  auto fn = get_encode_fn();
  if (!fn) return DSPARK_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(d)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kSubN), 256};
  cuuint32_t estr[2] = {1, 1};
  const CUresult rc = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W_lm), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// The draft with U given (U != null) or formed by the fused LM head from h
// and W_lm (U == null, d > 0).
static int launch_draft(const float* U, const uint16_t* h, const uint16_t* W_lm, int d, const uint16_t* W1,
                        const uint16_t* W2, const int32_t* anchors, int R, int gamma, int V, int rank,
                        float temperature, uint64_t seed, uint32_t round, int32_t* tokens, float* pd_tok, float* logZ,
                        void* workspace, cudaStream_t stream) {
  const bool lm = U == nullptr;
  const WorkspaceLayout L = workspace_layout(R, gamma, V);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DraftArgs a = {};
  a.U = U; a.W1 = W1; a.W2 = W2; a.anchors = anchors;
  a.h = h; a.d = lm ? d : 0;
  a.tokens = tokens; a.pd_tok = pd_tok; a.logZ = logZ;
  a.centry = reinterpret_cast<unsigned long long*>(ws + L.coarse);
  a.fine = reinterpret_cast<unsigned long long*>(ws + L.fine);
  a.status = reinterpret_cast<int32_t*>(ws + L.status);
  a.R = R;
  a.n_mtiles = ceil_div(R, kMTile);
  a.ready = reinterpret_cast<uint32_t*>(ws + L.dsync) + 16 * a.n_mtiles;
  a.abort = a.ready + 16 * a.n_mtiles;
  a.abuf = reinterpret_cast<uint4*>(ws + L.abuf);
#ifdef DSPARK_DRAFT_TRACE
  a.trace = nullptr;
#endif
  a.R_pad = a.n_mtiles * kMTile;
  a.gamma = gamma; a.V = V; a.rank = rank;
  a.n_tiles = ceil_div(V, kTileN);
  a.n_chunks = vocab_chunks(a.n_tiles, a.n_mtiles);
  const bool greedy = temperature == 0.0f;
  a.scale = greedy ? 1.0f : static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  a.seed = seed; a.round = round;
  // the sampler holds a row's chunk partials, and the sub-tile partials of
  // one chunk, in registers
  if (a.n_chunks > kMaxSampleChunks || 2 * ceil_div(a.n_tiles, a.n_chunks) > kMaxSampleChunks || V > kMaxDraftV)
    return DSPARK_ERR_UNSUPPORTED_SHAPE;

  CUtensorMap tm_w2, tm_u5, tm_u3, tm_slab, tm_lmslab;
  std::memset(&tm_u5, 0, sizeof(tm_u5));  // not used unless R % 8 == 0 or with the LM head
  std::memset(&tm_lmslab, 0, sizeof(tm_lmslab));  // used with the LM head only
  if (encode_w2_kchunk_map(&tm_w2, W2, V, rank) != DSPARK_OK || encode_w2_slab_map(&tm_slab, W2, V, rank) != DSPARK_OK)
    return DSPARK_ERR_CUDA;
  if (lm) {
    if (encode_w2_kchunk_map(&tm_u5, W_lm, V, d) != DSPARK_OK || encode_h_map(&tm_u3, h, R, gamma, d) != DSPARK_OK ||
        encode_lm_slab_map(&tm_lmslab, W_lm, V, d) != DSPARK_OK)
      return DSPARK_ERR_CUDA;
  } else if (encode_u_half_map(&tm_u3, U, R, gamma, V) != DSPARK_OK ||
             ((R & 7) == 0 && encode_u_fast_map(&tm_u5, U, R, gamma, V) != DSPARK_OK)) {
    return DSPARK_ERR_CUDA;
  }

  const DraftSmem plan = draft_smem_plan(rank);
  const int max_smem = static_cast<int>(draft_smem_plan(256).total);
  auto kernel = lm ? (greedy ? k_markov_draft<true, true> : k_markov_draft<false, true>)
                  : (greedy ? k_markov_draft<true, false> : k_markov_draft<false, false>);
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  // the chunk entries and the sub-tile partials (no tag matches), the ready
  // counters and the abort word start at zero on every call
#ifdef DSPARK_DRAFT_TRACE
  if (g_trace && g_trace_bytes >= static_cast<size_t>(gamma) * a.n_chunks * a.n_mtiles * kTraceEvents * 8) {
    a.trace = g_trace;
    if (cudaMemsetAsync(g_trace, 0, g_trace_bytes, stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  }
#endif
  {
    const size_t coarse_b = static_cast<size_t>(a.R_pad) * a.n_chunks * 8;
    const size_t fine_b = greedy ? 0 : static_cast<size_t>(2 * a.n_tiles) * a.R_pad * 8;
    k_draft_prologue<<<sm_count(), 256, 0, stream>>>(a, reinterpret_cast<uint4*>(ws + L.coarse), coarse_b / 16,
                                                      reinterpret_cast<uint4*>(ws + L.dsync), (L.dsync_bytes + 15) / 16,
                                                      reinterpret_cast<uint4*>(ws + L.fine), fine_b / 16);
    if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks * a.n_mtiles);
  cfg.blockDim = dim3(kDraftKThreads);
  cfg.dynamicSmemBytes = plan.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: the grid barriers rely on it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tm_w2, tm_u5, tm_u3, tm_slab, tm_lmslab, a) == cudaSuccess ? DSPARK_OK
                                                                                         : DSPARK_ERR_CUDA;
}

int launch_markov_draft(const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* anchors, int R,
                        int gamma, int V, int rank, float temperature, uint64_t seed, uint32_t round,
                        int32_t* tokens, float* pd_tok, float* logZ, void* workspace, cudaStream_t stream) {
  return launch_draft(U, nullptr, nullptr, 0, W1, W2, anchors, R, gamma, V, rank, temperature, seed, round, tokens,
                      pd_tok, logZ, workspace, stream);
}

int launch_markov_draft_lmhead(const uint16_t* h, const uint16_t* W_lm, int d, const uint16_t* W1, const uint16_t* W2,
                               const int32_t* anchors, int R, int gamma, int V, int rank, float temperature,
                               uint64_t seed, uint32_t round, int32_t* tokens, float* pd_tok, float* logZ,
                               void* workspace, cudaStream_t stream) {
  return launch_draft(nullptr, h, W_lm, d, W1, W2, anchors, R, gamma, V, rank, temperature, seed, round, tokens,
                      pd_tok, logZ, workspace, stream);
}

}  // namespace dspark

#ifdef DSPARK_DRAFT_TRACE
// Traced build only: the device buffer the next draft calls stamp their phase
// times into ([gamma][n_ctas][kTraceEvents] uint64; too small = no tracing).
extern "C" int dspark_draft_trace_buffer(void* buf, size_t bytes) {
  dspark::g_trace = static_cast<unsigned long long*>(buf);
  dspark::g_trace_bytes = buf ? bytes : 0;
  return DSPARK_OK;
}
#endif
