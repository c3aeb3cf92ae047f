/*
 * specsel.h -- C ABI of libspecsel.so: the selection step of one
 * speculative-decoding round on one NVIDIA GB300 (sm_103a).
 *
 * Two operations, from "A drafter inside the artifact" (Ignis DFlash2 page):
 *
 *   top-k   section "How it works", third paragraph: for each draft column,
 *           keep the k largest bf16 logits, largest first, ties going to
 *           the smaller row (token) id.  One launch streams the logits
 *           once: every CTA (or warp) of a full-GPU grid takes an equal
 *           slice of the flat run of columns, filters 16-byte vectors against
 *           a certified running k-th value, and the unit that completes a
 *           split column merges the published lists (spec_set_kernel).
 *
 *   verify  section "How it works", first paragraph: the target scores
 *           each lane's anchor and drafts in one pass; a lane keeps the
 *           drafts up to the first one the target disagrees with, and adds
 *           one token of the target's own choosing after them.  With greedy
 *           decoding ("Speculative decoding, measured on my M4 Max",
 *           section 1) the target's choice at a position is its argmax.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - bf16 values travel as uint16_t bit patterns.  Values compare as
 *    numbers: -0 and +0 tie, +-Inf are ordinary values.  NaN is outside the
 *    contract; the result for a column holding NaN is unspecified (but the
 *    call still returns and touches only its own outputs).
 *  - All data pointers are DEVICE pointers owned by the caller, except in
 *    spec_round_host.  The library keeps no reference after return.
 *  - Work is enqueued asynchronously on the calling thread's current stream
 *    (spec_set_stream; default: the legacy default stream 0).  Results are
 *    valid once that stream reaches the enqueued work.
 *  - Return value: SPEC_OK (0) or a negative SPEC_ERR_* code; argument
 *    errors are found on the host before anything is enqueued, and nothing
 *    is written.  spec_last_error() gives a message for the calling thread.
 *  - cols == 0 / lanes == 0 is a no-op that returns SPEC_OK.
 *  - Scratch: the library owns one scratch area per device (per-column
 *    tickets and partial lists, a few MB at most).  It grows on demand with
 *    cudaMalloc outside stream capture; inside a capture a call that needs
 *    more than spec_reserve set aside fails with SPEC_ERR_ALLOC.  An area
 *    that a larger one replaces stays allocated until spec_release, so
 *    launches in flight and CUDA graphs captured earlier keep valid scratch.  Calls that
 *    may run concurrently on the GPU (different streams, or different host
 *    threads) share this scratch and race: issue them on one stream.
 *  - Outputs must not alias inputs.
 */
#ifndef SPECSEL_H
#define SPECSEL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int spec_status;

#define SPEC_OK 0
#define SPEC_ERR_ARG (-1)    /* bad argument (null pointer, size, alignment, k, gamma) */
#define SPEC_ERR_ALLOC (-2)  /* scratch could not be obtained (incl. during capture) */
#define SPEC_ERR_CUDA (-3)   /* a CUDA runtime error; spec_last_error() has its text */

/* Vocabulary of the drafter's and target's output head: 248,046 tokens
   (same page, "How it works", third paragraph). spec_verify assumes it. */
#define SPEC_VOCAB 248046
/* Largest k: 64.  Largest gamma (drafts per lane): 15, the draft width of a
   block size of 16 ("Apathy-Qwen3.8-27B-DFlash-drafter-v2" model card: the
   usable draft width is one less than the block size, and the drafter's
   loader rejects a wider gamma). */
#define SPEC_MAX_K 64
#define SPEC_MAX_GAMMA 15

/* Per-column exact top-k.
 *   logits    bf16 [cols][V], row-major, contiguous, 2-byte aligned.  Column
 *             c starts at logits + c*V (any 16-byte phase is accepted).
 *   cols      number of draft columns, >= 0.
 *   V         vocabulary size, 1 <= V <= 2^31-1.
 *   k         1 <= k <= min(V, 64).
 *   out_vals  bf16 [cols][k]: the selected values, largest first; each is
 *             the selected element's own bit pattern.
 *   out_ids   int32 [cols][k]: their ids in [0, V); equal values appear in
 *             ascending id order.
 * Errors: SPEC_ERR_ARG for a null pointer with cols > 0, V < 1, k out of
 * range, or a misaligned pointer; SPEC_ERR_ALLOC; SPEC_ERR_CUDA. */
spec_status spec_topk(const uint16_t *logits, int64_t cols, int64_t V, int32_t k,
                      uint16_t *out_vals, int32_t *out_ids);

/* Shortlist top-k ("How it works", second paragraph: an optional drafter
 * head whose output covers only 131,072 of the commonest token ids).  As
 * spec_topk over [cols][V] shortlist logits, where local id i stands for
 * vocabulary id id_map[i]:
 *   id_map    int32 [V], device, injective (distinct entries), values >= 0.
 *   out_ids   vocabulary ids id_map[i]; ties go to the smaller VOCABULARY id.
 * Duplicate entries in id_map are outside the contract. */
spec_status spec_topk_mapped(const uint16_t *logits, int64_t cols, int64_t V, int32_t k,
                             const int32_t *id_map, uint16_t *out_vals, int32_t *out_ids);

/* Greedy verify over V = SPEC_VOCAB.
 *   target_logits  bf16 [lanes][gamma+1][V], contiguous.  Column j of a lane
 *                  is the target's next-token logits after the anchor and
 *                  the first j drafts (j = 0 is the anchor's own).
 *   drafts         int32 [lanes][gamma]: draft i is the token proposed for
 *                  the position target column i predicts.  Ids outside
 *                  [0, V) are not errors; they never match.
 *   lanes >= 0, 1 <= gamma <= 15.
 *   out_accept_len int32 [lanes]: a = the longest prefix with
 *                  drafts[l][i] == argmax(target column i), 0 <= a <= gamma.
 *   out_commit_ids int32 [lanes][gamma+1]: argmax of columns 0..a (the a
 *                  accepted drafts, then the bonus token), -1 after.
 *   The argmax breaks ties toward the smaller id.  Target logits are read
 *   once; argmax and prefix match happen in the same launch. */
spec_status spec_verify(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                        int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids);

/* spec_verify with an explicit vocabulary size V (1 <= V <= 2^31-1). */
spec_status spec_verify_v(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                          int32_t gamma, int64_t V, int32_t *out_accept_len,
                          int32_t *out_commit_ids);

/* Sampled verify with one-hot drafts (speculative sampling; "A drafter
 * inside the artifact", Ignis DFlash2 page, "The numbers": sampled
 * acceptance at T = 1.0, top_p 0.95, top_k 20).  Per target column the
 * target's distribution q is computed in float64 from the column's top_k
 * logits (largest first, ties to the smaller id), in this order:
 * z_t = v_t / temperature; e_t = exp(z_t - z_0); p_t = e_t / sum(e);
 * the nucleus is the shortest prefix whose running sum of p reaches top_p;
 * q_t = p_t / (that sum).  Position j < gamma accepts draft j when
 * uniforms[l][j][0] < q_j(draft j) (0 outside the nucleus).  The first
 * rejected position commits a draw from q_j without the draft: the first
 * nucleus token (draft skipped, list order) whose running q exceeds
 * uniforms[l][j][1] times the total q without the draft.  A lane that accepts
 * all gamma drafts commits a draw from q_gamma with uniforms[l][gamma][1].
 *   uniforms  double [lanes][gamma+1][2], each in [0, 1), caller-owned device
 *             memory (random numbers are inputs: no generator inside).
 *   temperature > 0, 0 < top_p <= 1, 1 <= top_k <= min(V, 64).
 *   out_accept_len, out_commit_ids as for spec_verify: the accepted drafts,
 *   then the draw, then -1.
 * With top_k = 1 this is exactly spec_verify_v.  One launch; target logits
 * are read once.  A column whose best value is +-Inf has no softmax: such
 * columns (like NaN) are outside this call's contract. */
spec_status spec_verify_sampled(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                                int32_t gamma, int64_t V, double temperature, double top_p,
                                int32_t top_k, const double *uniforms, int32_t *out_accept_len,
                                int32_t *out_commit_ids);

/* spec_round with sampled verify: spec_topk over the draft columns and
 * spec_verify_sampled over the target columns in ONE launch, same V. */
spec_status spec_round_sampled(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k,
                               uint16_t *out_vals, int32_t *out_ids,
                               const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                               int32_t gamma, double temperature, double top_p, int32_t top_k,
                               const double *uniforms, int32_t *out_accept_len,
                               int32_t *out_commit_ids);

/* One whole selection step in ONE kernel launch: spec_topk over the draft
 * columns and spec_verify_v over the target columns, same vocabulary V.
 * Results are identical to the two separate calls.  Either part may be
 * empty (cols == 0 or lanes == 0). */
spec_status spec_round(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k,
                       uint16_t *out_vals, int32_t *out_ids,
                       const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                       int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids);

/* Speculative-decoding counters ("A drafter inside the artifact", Ignis
 * DFlash2 page, section "See it, control it", Metrics: rounds, drafted and
 * accepted tokens, and the per-position drafted/accepted pair), kept in
 * DEVICE memory and only ever added to.  Per verified lane of a round:
 *   rounds += 1;  drafted_tokens += gamma;  accepted_tokens += a;
 *   position_drafted[i] += 1 and position_accepted[i] += (a > i)
 * for i < gamma, where a is the lane's accept length.  So the per-position
 * counts sum to the totals, and tokens committed per round are
 * (accepted_tokens + rounds) / rounds (the bonus token is not a draft). */
typedef struct {
    uint64_t rounds;
    uint64_t drafted_tokens;
    uint64_t accepted_tokens;
    uint64_t position_drafted[SPEC_MAX_GAMMA];
    uint64_t position_accepted[SPEC_MAX_GAMMA];
} spec_counters;

/* spec_round, also adding the round's verify outcome to *counters (a device
 * pointer to a zero-initialised or earlier-used spec_counters, 8-byte
 * aligned; NULL: no counting, exactly spec_round).  The counts are device
 * atomics in the same launch; concurrent calls may share one block. */
spec_status spec_round_counted(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k,
                               uint16_t *out_vals, int32_t *out_ids,
                               const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                               int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids,
                               spec_counters *counters);

/* spec_round for callers holding HOST buffers: every pointer is a host
 * pointer (pinned memory copies fastest).  The call copies the inputs to
 * library-owned device staging memory, runs spec_round, copies the outputs
 * back and waits for the stream, so outputs are valid on return.  Staging
 * grows with cudaMalloc as needed (not capturable); an area a larger one
 * replaces stays allocated until spec_release.  Host calls from several
 * threads are serialised inside the library (each holds it until its stream
 * has drained), so they never share the staging area while it is in use. */
spec_status spec_round_host(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k,
                            uint16_t *out_vals, int32_t *out_ids,
                            const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                            int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids);

/* spec_round without any allocation, for callers that cannot let a library
 * call cudaMalloc: an inference engine that serves every byte of device memory
 * from its own pool, a serving loop that cannot afford the device-wide
 * synchronisation of cudaFree, or a host under a fixed memory budget.  The
 * pages describe no such entry point; it is an addition of this library.
 *
 * Same arguments, results and errors as spec_round (all device pointers, the
 * calling thread's stream), except:
 *   - its scratch is one fixed device array inside the library (about 1.1
 *     MB), which every GPU that loads the library keeps until the process
 *     exits; nothing is ever allocated or freed (no cudaMalloc, no cudaFree);
 *   - sizes are limited: cols + lanes*(gamma+1) <= SPEC_NOALLOC_MAX_COLS and
 *     lanes <= SPEC_NOALLOC_MAX_LANES; larger calls return SPEC_ERR_ARG with
 *     a message naming the limit;
 *   - the array holds a fixed number of published partial lists, so a round
 *     with a large k may be spread over fewer streaming units than spec_round
 *     would use (same results, possibly slower: at k = 64 at most 992 units);
 *   - the first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture;
 *   - every call shares the one array and starts by clearing its tickets on
 *     the stream, so calls that overlap on the GPU (different streams, or
 *     different host threads) race and must not be issued that way. */
#define SPEC_NOALLOC_MAX_COLS 8192
#define SPEC_NOALLOC_MAX_LANES 512
spec_status spec_round_noalloc(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k,
                               uint16_t *out_vals, int32_t *out_ids,
                               const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                               int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids);

/* ---- The Q4 shortlist head ("A drafter inside the artifact", Ignis DFlash2
 * page, section "How it works", second paragraph: an opt-in 4-bit head over
 * the 131,072 most frequent tokens, about 356 MB, in place of the drafter's
 * full output head).  The page gives the bit width, the row count and the
 * size; the layout below is the reading taken (with a hidden width d of 5,120
 * it gives 131,072 x (2,560 + 160) bytes = 356.5 MB):
 *   weights  uint8 [rows][d/2]: byte j of a row holds weight 2j in its low
 *            nibble and weight 2j+1 in its high nibble; a nibble n stands for
 *            the integer n - 8;
 *   scales   fp16 bit patterns [rows][d/64]: scale b multiplies weights
 *            64b .. 64b+63 of its row.
 * The logit of row i for a hidden state h (bf16, length d) is
 *   sum_b scale[i][b] * sum_{j in block b} (n_ij - 8) * h_j,
 * summed in fp32 (each 64-weight block's products on the tensor cores, then
 * scaled and added) and rounded once to bf16, to nearest even.  It differs
 * from the exact value by at most half a bf16 unit plus 2^-16 times
 * sum_j |scale (n_ij - 8) h_j| (the bound the tests hold it to).
 * rows: a positive multiple of 16 below 2^31; d: a multiple of 64, at most 6,144. */

/* Reorder a head into the layout the logits kernel streams (once, at load):
 *   weights, scales  the head as above (device memory, caller-owned);
 *   wpack            device, rows*d/2 bytes, 16-byte aligned (the same size as weights);
 *   spack            device, rows*(d/64)*2 bytes, 4-byte aligned (the same size as scales).
 * Enqueued on the calling thread's stream; SPEC_ERR_ARG for bad sizes, null or
 * misaligned pointers. */
spec_status spec_shortlist_pack(const uint8_t *weights, const uint16_t *scales, int64_t rows, int64_t d,
                                void *wpack, void *spack);

/* The head's logits: hidden bf16 [cols][d] (16-byte aligned) -> out_logits
 * bf16 [cols][rows] (row i of column c at c*rows + i).  wpack/spack from
 * spec_shortlist_pack.  One launch per 16 hidden states, each streaming the
 * packed head once.  cols == 0 is a no-op. */
spec_status spec_shortlist_logits(const uint16_t *hidden, int64_t cols, int64_t d, const void *wpack,
                                  const void *spack, int64_t rows, uint16_t *out_logits);

/* The shortlist proposal of each hidden state: its logits (as
 * spec_shortlist_logits, into the caller's logits buffer [cols][rows], which
 * the call uses as its workspace and leaves filled), then spec_topk_mapped
 * over them with id_map [rows] (local row -> vocabulary id, injective): the k
 * largest, ties to the smaller vocabulary id, out_ids vocabulary ids.
 * 1 <= k <= min(rows, 64).  The top-k is bit-exact on the logits it leaves. */
spec_status spec_shortlist_topk(const uint16_t *hidden, int64_t cols, int64_t d, const void *wpack,
                                const void *spack, int64_t rows, const int32_t *id_map, int32_t k,
                                uint16_t *logits, uint16_t *out_vals, int32_t *out_ids);

/* Which streaming kernel runs a round.  All compute the same results (every
 * output is the unique exact answer); they differ only in speed:
 *   SPEC_KERNEL_GROUPMAX -- two phases in one launch.  The stream keeps only
 *                       the maximum of each thread's group of 64 logits
 *                       (a 2-byte key); per column, the k-th largest of
 *                       those maxima bounds the top-k, and only the few
 *                       groups that reach it are read again and ranked.
 *                       One-pass mode (rounds of at most 4,096 -- or 8,192
 *                       -- 16-byte vectors a CTA with every column on at
 *                       least one CTA): each CTA keeps its slice of one
 *                       column in registers and selects from them; a
 *                       column's CTAs publish their lists (greedy verify:
 *                       one argmax each) and the last to arrive merges --
 *                       through the shared memory of a thread-block
 *                       cluster of eight CTAs a column where that fills
 *                       the GPU (about 15 to 19 columns).
 *                       Columns in clusters (fewer columns, too many
 *                       logits for one pass): each column one cluster of
 *                       2 to 8 CTAs, each streaming part of it with its
 *                       keys in shared memory, the parts' lists merged in
 *                       the cluster's first CTA.
 *                       Column mode (at least 3/4 as many columns as SMs,
 *                       columns of 32,768 to ~393,000 logits): each CTA
 *                       owns whole columns and keeps their keys in shared
 *                       memory; from 1.5 columns per SM on, four of its
 *                       warps finish one column while twelve stream the
 *                       next.  Slice mode (otherwise, V >= 4096): CTAs own
 *                       equal slices and meet per column through tickets,
 *                       with scratch of about 2 bytes per 8-64 logits (the
 *                       CTA kernel runs instead inside a graph capture that
 *                       the scratch does not yet cover -- one call of the
 *                       same sizes before capturing makes room).
 *   SPEC_KERNEL_CTA  -- the CTAs of a full-GPU grid each stream a contiguous
 *                       slice in 60 KiB chunks; per column one threshold per
 *                       CTA (the k-th best the CTA has seen), kept by a
 *                       merging warp.
 *   SPEC_KERNEL_WARP -- every warp streams its own slice with its own ring,
 *                       buffer and threshold; no coordination inside the
 *                       stream.
 *   SPEC_KERNEL_AUTO -- (default) GROUPMAX in one-pass mode where it fits,
 *                       else in column mode at any size; else, up to 6 MiB
 *                       of logits per SM, GROUPMAX in slice mode (or CTA
 *                       where it cannot run); else WARP.
 * The choice is process-wide; SPEC_ERR_ARG for any other value. */
#define SPEC_KERNEL_AUTO 0
#define SPEC_KERNEL_WARP 1
#define SPEC_KERNEL_CTA 2
#define SPEC_KERNEL_GROUPMAX 3
spec_status spec_set_kernel(int32_t which);
int32_t spec_get_kernel(void);

/* The streaming kernel (SPEC_KERNEL_WARP, _CTA or _GROUPMAX) of the round
 * the calling thread launched last (spec_round and the entry points built on
 * it); SPEC_KERNEL_AUTO before the first.  Host-side bookkeeping only. */
int32_t spec_last_kernel(void);

/* Set the stream (a cudaStream_t, may be NULL for the legacy default stream)
 * that the calling thread's subsequent calls enqueue on.  Thread-local. */
spec_status spec_set_stream(void *stream);
void *spec_get_stream(void);

/* Make sure the current device's scratch covers calls up to these sizes
 * (so that later calls need no allocation, e.g. inside a CUDA graph
 * capture).  max_cols counts draft columns, max_lanes/max_gamma the verify
 * part; max_k is the largest k -- or sampled-verify top_k -- to come.
 * Growing allocates a new area (cudaMalloc + cudaMemset); the old one is
 * kept for what already uses it. */
spec_status spec_reserve(int64_t max_cols, int32_t max_k, int64_t max_lanes, int32_t max_gamma);

/* Free the scratch (current and replaced areas) and staging of the current
 * device, after synchronising it.  CUDA graphs that captured calls of this
 * library must not be replayed afterwards.  Later calls allocate again. */
spec_status spec_release(void);

/* Diagnostic of the bounded waits every kernel uses on its copy pipeline:
 * launches (on the calling thread's stream) one thread that waits on an
 * mbarrier nothing arrives on, for at most limit_ns (1 us .. 1 s), then
 * waits on it once more.  The first wait gives up and raises the flag that
 * spec_device_status reports; the second returns at once (a CTA whose wait
 * gave up waits no more).  out4: device uint64[4] = {first wait succeeded
 * (0), its ns, second wait succeeded (0), its ns}.  No fault, no hang. */
spec_status spec_selftest_wait_timeout(int64_t limit_ns, uint64_t *out4);

/* Text of the last error raised on the calling thread ("" if none). */
const char *spec_last_error(void);

/* Waits for the calling thread's stream, then reports whether any kernel
 * of the library gave up a bounded wait on its copy pipeline since the last
 * call (SPEC_ERR_CUDA, and the flag is cleared) or not (SPEC_OK).  Every
 * wait in the kernels is bounded, so a broken pipeline ends the kernel with
 * invalid results and this flag set, instead of hanging the GPU. */
spec_status spec_device_status(void);

/* Number of kernel launches this process made through the library (all
 * devices, all threads).  One per spec_topk / spec_verify / spec_round. */
int64_t spec_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECSEL_H */
