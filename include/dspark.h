/*
 * dspark.h — C ABI of libdspark.so: the data-parallel hot path of one DSpark
 * speculative-decoding round on one GB300 (sm_103a).
 *
 * A round (pages: "DSpark", rainlin-net; "投机解码的新做法：整块草稿、按负载验证与
 * PD 分离"; "DSpark: Speculative decodingを活用したLLM推論の高速化"):
 *   1. dspark_markov_draft  — sequential Markov-head draft over gamma positions
 *                             ("DSpark" §2.2 eq. p_k, §2.3 eq. B = W1 W2).
 *   2. dspark_confidence    — c_k = sigma(w^T [h_k ; W1[x_{k-1}]]) (§3.1) and the
 *                             survival products a_j = prod_{i<=j} c_i (§1.1).
 *   3. dspark_schedule      — hardware-aware prefix scheduler maximising
 *                             Theta = tau * SPS(B) (§4.1), early stop (§4.2) or
 *                             lagged-budget Top-K (§4.3).
 *   4. dspark_verify        — standard rejection-sampling verification against
 *                             the target logits (introduction; §2.2).
 *
 * Conventions shared by every entry point:
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; row-major,
 *    contiguous, no padding.  The library never allocates, frees or
 *    synchronises; each call only enqueues kernels on `stream` (a
 *    cudaStream_t passed as void*, NULL = legacy default stream) and can be
 *    captured into a CUDA graph.
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - Scratch memory: `workspace` of at least dspark_workspace_size(...) bytes,
 *    256-byte aligned, owned by the caller and reusable across calls on the
 *    same stream.  Its first int32 is the device status word (DSPARK_STATUS_*
 *    bits, OR-ed by kernels); dspark_clear_status() zeroes it.  Read it after
 *    the stream has synchronised.
 *  - Return value: DSPARK_OK, or a negative DSPARK_ERR_* code, in which case
 *    nothing was enqueued (argument errors) or a launch failed (_CUDA).
 *  - Uniforms: Philox4x64-10 (Salmon et al., SC'11), key = (seed, 0),
 *    counter = (round, request, position, purpose), u = (word0 >> 40) * 2^-24;
 *    purpose 0 draft sample, 1 accept test, 2 residual / bonus sample.
 *  - temperature T > 0 samples from softmax(logits / T); T == 0 is greedy
 *    (argmax, lowest index on ties).
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSPARK_OK 0
#define DSPARK_ERR_INVALID_ARG (-1)       /* null pointer, negative size, bad temperature, short workspace, misalignment */
#define DSPARK_ERR_UNSUPPORTED_SHAPE (-2) /* V % 8 != 0, rank not in {64,128,192,256}, gamma > 64,
                                            R*gamma > 8192 (schedule), V > 2^24 (draft), R > 32768 (verify) */
#define DSPARK_ERR_CUDA (-3)              /* a kernel launch or CUDA runtime call failed */
#define DSPARK_ERR_STATIC_SCRATCH_TOO_SMALL (-4) /* dspark_markov_draft_noalloc: shape needs more than
                                                    DSPARK_NOALLOC_SCRATCH_BYTES of scratch */

/* bits of the device status word (first int32 of the workspace) */
#define DSPARK_STATUS_NONFINITE 1  /* a softmax row had a non-finite max or normaliser */
#define DSPARK_STATUS_BAD_TOKEN 2  /* a token / anchor outside [0, V) was read (clamped to 0) */
#define DSPARK_STATUS_TIMEOUT 4    /* a bounded device wait gave up; outputs are not valid */
#define DSPARK_STATUS_BAD_LENGTH 8 /* a verify length outside [0, gamma] was read (clamped) */

/* Scheduler modes ("DSpark" §4.2-4.3; "スケジューラの実運用適用"). */
#define DSPARK_MODE_EARLY_STOP 0 /* stop at the first b with Theta(b+1) <= Theta(b) */
#define DSPARK_MODE_TOP_K 1      /* admit the top min(budget_K, R*gamma) pairs */
#define DSPARK_MODE_FIXED 2      /* verify every drafted position */

/* Bytes of scratch memory the draft, schedule and verify calls need for these
 * sizes (any temperature).  Returns 0 for invalid sizes. */
size_t dspark_workspace_size(int R, int gamma, int V, int rank, int d);

/* Enqueue a zeroing of the workspace status word. */
int dspark_clear_status(void *workspace, void *stream);

/* Self-test of the device-side timeout path.  Enqueues one kernel in which a
 * thread waits, through the same bounded mbarrier wait the pipelined kernels
 * use on their rings, for a phase that nothing ever completes.  When the wait
 * gives up (after 2 s) the kernel ORs DSPARK_STATUS_TIMEOUT into the
 * workspace status word and returns; nothing faults, and the context stays
 * usable.  workspace: any 256-byte-aligned device buffer whose first int32 is
 * the status word.  Returns DSPARK_ERR_INVALID_ARG for a null or misaligned
 * workspace, DSPARK_ERR_CUDA if the launch fails. */
int dspark_selftest_bounded_wait(void *workspace, void *stream);

/*
 * Markov-head sequential draft ("DSpark" §2.2 eq. p_k and §2.3; the loop of
 * §6.2).  For each request r and position j = 0..gamma-1, with x_{-1} = anchor:
 *     z_j(v)  = (U[r,j,v] + W1[x_{j-1}] . W2[:,v]) / T
 *     x_j     = first v with sum_{u<=v} softmax(z_j)(u) > u_j   (T > 0)
 *             = argmax_v fp32(U[r,j,v] + bias(v))               (T == 0)
 * and records p_d(x_j) = softmax(z_j)(x_j) and log Z_j = logsumexp(z_j)
 * (T == 0: p_d = 1 and log Z = the maximal logit).
 *   U        fp32 [R, gamma, V]   base logits of the parallel backbone (16-byte aligned)
 *   W1       bf16 [V, rank]       Markov embedding (16-byte aligned)
 *   W2       bf16 [rank, V]       Markov projection (16-byte aligned)
 *   anchors  int32 [R]            x_0 of each request (the anchor token)
 *   tokens   int32 [R, gamma]     out: drafted tokens
 *   pd_tok   fp32 [R, gamma]      out: p_d(x_j)
 *   logZ     fp32 [R, gamma]      out: log Z_j (natural log, of z_j = logits / T)
 * Sizes: R >= 0, 1 <= gamma <= 64, 8 <= V <= 2^24 with V % 8 == 0, rank in {64,128,192,256}.
 * R == 0 enqueues nothing.  Enqueues a prologue kernel (zeroes the
 * workspace's synchronisation words and partials, stages the anchors' W1 rows)
 * and one cooperative kernel that keeps every CTA resident for all gamma
 * positions (one CTA per SM; it fails to launch, with DSPARK_ERR_CUDA, when R
 * needs more than one M-tile of 128 rows per SM).
 * The kernel's cross-CTA waits are bounded: a wait that gives up sets
 * DSPARK_STATUS_TIMEOUT and the outputs are then not valid.
 */
int dspark_markov_draft(const float *U, const uint16_t *W1, const uint16_t *W2,
                        const int32_t *anchors, int R, int gamma, int V, int rank,
                        float temperature, uint64_t seed, uint32_t round, int32_t *tokens,
                        float *pd_tok, float *logZ, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * The same draft with the LM head fused in: the pre-LM-head hidden states h
 * are given instead of the logits U, and U = h . W_lm is formed tile by tile
 * inside the draft (hidden-state communication: "DSpark: Speculative
 * decodingを活用した…", "実サービス配備 › 拡張可能な学習 › 隠れ状態通信" ships the
 * hidden state rather than V-wide logits and runs the LM head where the
 * tokens are drawn).  For each request r and position j:
 *     z_j(v) = (h[r,j,:] . W_lm[:,v] + W1[x_{j-1}] . W2[:,v]) / T
 * and the rest exactly as dspark_markov_draft (same outputs, same sampling,
 * same Philox draws).  Both dot products accumulate in one fp32 sum of bf16
 * products (tensor cores), so U is never rounded to fp32 on its own.
 *   h        bf16 [R, gamma, d]   pre-LM-head hidden states (16-byte aligned)
 *   W_lm     bf16 [d, V]          LM-head weight (16-byte aligned)
 *   W1, W2, anchors, tokens, pd_tok, logZ, workspace   as for dspark_markov_draft
 * Sizes: as dspark_markov_draft, and d % 128 == 0, d <= 65536.
 * Cost: W_lm is read once per position (gamma * d * V * 2 bytes a call), so at
 * batch sizes where R * gamma * V * 4 < gamma * d * V * 2 (R < d / 2) reading a
 * materialised U through dspark_markov_draft moves fewer bytes.
 */
int dspark_markov_draft_lmhead(const uint16_t *h, const uint16_t *W_lm, const uint16_t *W1,
                               const uint16_t *W2, const int32_t *anchors, int R, int gamma,
                               int V, int rank, int d, float temperature, uint64_t seed,
                               uint32_t round, int32_t *tokens, float *pd_tok, float *logZ,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * Confidence head and survival products ("DSpark" §3.1 eq. c_k; §1.1 eq. a_j):
 *     c[r,j] = sigma( sum_i w[i] h[r,j,i] + sum_i w[d+i] W1[x_{j-1}, i] ),  x_{-1} = anchor
 *     a[r,j] = fp32(a[r,j-1] * c[r,j]),  a[r,-1] = 1  (left to right)
 * No bias term; w = [w_h (d) ; w_e (rank)] follows the concatenation [h ; W1[x]].
 * Sequential temperature scaling ("DSpark" §3.2, STS): when sts_temperature is
 * given, the logit of position j is divided by t_j before the sigmoid,
 *     c[r,j] = sigma( logit[r,j] / t_j ),
 * with the t_j fitted offline, position after position, by a grid search that
 * minimises the calibration error of a[., j] (python: sts.fit_sts).
 *   h        bf16 [R, gamma, d]   backbone hidden states
 *   W1       bf16 [V, rank]
 *   w        fp32 [d + rank]
 *   sts_temperature fp32 [gamma]  device, or NULL for no scaling; a t_j that is not a
 *                                 finite positive number is taken as 1 and raises
 *                                 DSPARK_STATUS_NONFINITE
 *   anchors  int32 [R], tokens int32 [R, gamma] (only columns 0..gamma-2 are read)
 *   c, a     fp32 [R, gamma]      out
 * Sizes: R >= 0, 1 <= gamma <= 64, d >= 1, rank >= 1.
 */
int dspark_confidence(const uint16_t *h, const uint16_t *W1, const float *w,
                      const float *sts_temperature, const int32_t *anchors, const int32_t *tokens, int R, int gamma, int d,
                      int rank, int V, float *c, float *a, void *workspace, size_t workspace_bytes,
                      void *stream);

/*
 * Hardware-aware prefix scheduler ("DSpark" §4.1-4.3; "投机解码的新做法",
 * section "按负载决定验证多少").  Sorts all (r, j) by a[r,j] descending (ties:
 * j ascending, then r ascending), forms S_b = sum of the top b values in Q.40
 * fixed point, and scores every budget b = 0..R*gamma as
 *     Theta(b) = (R + S_b * 2^-40) * sps[R + b]        (fp64; B = R + b tokens)
 * then picks b* by `mode` and sets lens[r] = #{admitted pairs of request r}
 * (always a prefix of each request because a is non-increasing in j).
 *   a        fp32 [R, gamma]      survival products (non-negative)
 *   sps      fp64 [sps_len]       steps per second at batch B, indexed by B; sps_len >= R*(1+gamma)+1
 *   budget_K                      DSPARK_MODE_TOP_K: the budget chosen two rounds earlier
 *   lens     int32 [R]            out: verify length per request
 *   total_b  int32 [1]            out: b*
 *   argmax_b int32 [1]            out: global argmax_b Theta(b) (lowest b on ties) — keep it
 *                                 as the Top-K budget for round t+2
 *   theta    fp64 [1]             out: Theta(b*)
 * Sizes: R >= 1, 1 <= gamma <= 64, R * gamma <= 8192.  One CTA; no host round trip.
 */
int dspark_schedule(const float *a, int R, int gamma, const double *sps, int sps_len, int mode,
                    int budget_K, int32_t *lens, int32_t *total_b, int32_t *argmax_b,
                    double *theta, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Rejection-sampling verification (standard speculative verification:
 * "DSpark" introduction and §2.2; "DSpark: Speculative decodingを活用した…",
 * "問題定義").  For request r and j = 0..lens[r]-1:
 *     accept x_j  iff  u_acc(r,j) < p_t(x_j) / p_d(x_j)     (T > 0)
 *                 iff  x_j == argmax T[r,j,:]                (T == 0)
 * with p_t = softmax(T[r,j,:] / T) and p_d the draft's own probability.  At the
 * first rejection n the next token is drawn from max(0, p_t - p_d) renormalised
 * (from p_t if that mass is zero), where p_d's row is recomputed from U, W1, W2
 * and the stored log Z; if all lens[r] drafts are accepted, a bonus token is
 * drawn from target row lens[r].  Greedy: next = argmax of row n.
 *   T        fp32 [R, gamma+1, V] target logits (row gamma = bonus row for lens = gamma)
 *   U, W1, W2, anchors            as for dspark_markov_draft
 *   tokens, pd_tok, logZ          the draft's outputs
 *   lens     int32 [R]            verify lengths (from dspark_schedule)
 *   n_accept int32 [R]            out: accepted drafts
 *   next_token int32 [R]          out: correction or bonus token
 *   c_star   fp32 [R, gamma]      optional out (NULL: not computed, no extra work): the
 *                                 analytic acceptance ("DSpark" §3.1, eq. c_k*)
 *                                     c*[r,j] = 1 - 1/2 || p_d - p_t ||_1
 *                                 of every position j <= lens[r] (j < gamma), with p_d the
 *                                 draft distribution at j (conditioned on x_{j-1}) and p_t
 *                                 that of target row j; NaN for j > lens[r].  T == 0: both
 *                                 are point masses, c* = 1 if x_j == argmax T[r,j,:], else 0.
 *                                 With T > 0 the residual pass then covers every such row
 *                                 (it re-reads their U and T rows) instead of the rejected
 *                                 rows only.
 * Only rows 0..lens[r] of each request are read.
 * Sizes: as dspark_markov_draft, and R <= 32768.
 */
int dspark_verify(const float *T, const float *U, const uint16_t *W1, const uint16_t *W2,
                  const int32_t *anchors, const int32_t *tokens, const float *pd_tok,
                  const float *logZ, const int32_t *lens, int R, int gamma, int V, int rank,
                  float temperature, uint64_t seed, uint32_t round, int32_t *n_accept,
                  int32_t *next_token, float *c_star, void *workspace, size_t workspace_bytes,
                  void *stream);

/*
 * dspark_load_verified_rows — bring into device memory, from page-locked host
 * memory, exactly the target rows that dspark_verify reads: rows 0..lens[r]
 * of each request r, the prefix the scheduler admitted for verification
 * ("DSpark" §4.1-4.2: only the admitted positions are verified).  The pages
 * have no counterpart: this entry point exists for callers whose target
 * logits arrive in host memory.  lens is read on the device, so the ragged
 * copy needs no device-to-host read of the lengths and no synchronisation;
 * the SMs read the host memory over the host link (mapped memory), which
 * leaves the copy engines free for other copies running at the same time.
 *   T_host  fp32 [R, gamma+1, V]  HOST pointer: page-locked memory mapped into the
 *                                 device's address space (cudaHostAlloc, cudaMallocHost
 *                                 or cudaHostRegister on a device with unified
 *                                 addressing); 16-byte aligned; owned by the caller
 *   lens    int32 [R]             device; a length outside [0, gamma] is clamped and
 *                                 sets DSPARK_STATUS_BAD_LENGTH
 *   T       fp32 [R, gamma+1, V]  out, device: rows 0..lens[r] of request r are
 *                                 written, all other rows are left as they were
 *   workspace                     any 256-byte-aligned device buffer whose first int32
 *                                 is the status word
 * Sizes: R >= 0, 1 <= gamma <= 64, V >= 8 with V % 8 == 0.  R == 0 enqueues
 * nothing.  Returns DSPARK_ERR_INVALID_ARG, enqueuing nothing, when T_host is
 * not page-locked mapped host memory (pageable or device memory).  One kernel.
 */
int dspark_load_verified_rows(const float *T_host, const int32_t *lens, int R, int gamma, int V,
                              float *T, void *workspace, void *stream);

/*
 * dspark_markov_draft_noalloc — the Markov-head draft of dspark_markov_draft
 * without a caller workspace.  The pages have no counterpart: this entry point
 * exists for callers that cannot obtain device memory where they draft, such
 * as an engine recording its decode step into a CUDA graph (cudaMalloc is not
 * allowed while capture is open), a serving loop that bans allocator calls
 * because cudaMalloc / cudaFree can synchronise the device, or a plug-in whose
 * host program owns all device memory.
 *
 * Same inputs, outputs, sizes and results as dspark_markov_draft.  Scratch
 * (status word and softmax partials) lives in one file-scope device array of
 * DSPARK_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU loading the library
 * keeps until the process exits.
 *   status   int32 [1] or NULL   out: this call's DSPARK_STATUS_* bits (device
 *                                memory; copied there at the end of the call)
 * Returns DSPARK_ERR_STATIC_SCRATCH_TOO_SMALL, enqueuing nothing, when the shape
 * needs more scratch than the array holds: the draft needs 256 B + R_pad * 8 KiB
 * + R_pad * 16 * ceil(V / 64) bytes with R_pad = R rounded up to 128, e.g.
 * 5.6 MiB at R = 128, V = 151936 and 9.9 MiB at R = 256, V = 129280.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture begins.  All calls on a device share the
 * array and it keeps the previous call's contents: each call zeroes the status
 * word first and rewrites every partial it reads, but calls whose kernels
 * overlap on the GPU (unordered streams) race on it.  Allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.
 */
#define DSPARK_NOALLOC_SCRATCH_BYTES (16u << 20)
int dspark_markov_draft_noalloc(const float *U, const uint16_t *W1, const uint16_t *W2,
                                const int32_t *anchors, int R, int gamma, int V, int rank,
                                float temperature, uint64_t seed, uint32_t round, int32_t *tokens,
                                float *pd_tok, float *logZ, int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
