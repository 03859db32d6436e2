/*
 * specverify.h - C ABI of the GB300 (sm_103a) speculative-decoding verify sampler.
 *
 * Four calls make up the hot path of one DSpark verify step:
 *   dspark_markov_bias     - the Markov head's low-rank previous-token logit bias
 *                            (dspark_markov_walk: the same bias with the draft tokens sampled
 *                            slot by slot)
 *   spec_verify_tokenwise  - token-by-token speculative sampling
 *   spec_verify_block      - block verification
 *   adaptive_pick_k        - confidence head + the controller that picks how many drafts to verify
 * Sources (web pages, cited by title and section):
 *   [P1] "MTP, DSpark and Block Verification, Explained: Six Tokens per Step" (al-engr.com)
 *   [P2] "MTP Heads and Confidence Heads: Linking Three Self-Drafting Routes into One Chain"
 *        (naphjohn.github.io)
 *   [P3] "Teaching the Speculator What a Draft Costs" (al-engr.com)
 *
 * Conventions shared by every call
 *   - Every tensor argument is a DEVICE pointer to caller-owned memory, row-major and dense.
 *     The library never allocates, never frees and never keeps a pointer after the call
 *     returns.  It keeps no state between calls.  Two handles are the exceptions, each
 *     owning what it creates until its destroy call: the adaptive pipeline (a CUDA graph
 *     that keeps the device pointers it was created with) and the online cost curve (host
 *     memory, CUDA events and two pinned buffers).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and never synchronises the host.  Outputs are valid once the stream reaches
 *     the end of the call's work.  Calls on the same stream are ordered.
 *   - Logit and weight dtypes are SPEC_DTYPE_F32 (float) or SPEC_DTYPE_BF16 (bfloat16).
 *     Arithmetic is float32 per element; per-stream scalars are double-float (two float32s,
 *     about 48 significant bits).
 *   - Return value: SPEC_OK, or a negative SPEC_ERR_* for an error the host can see from the
 *     arguments alone (nothing is launched then), or SPEC_ERR_CUDA when a launch failed.
 *     spec_last_error() gives a one-line description of the last error in this host thread.
 *   - Errors that depend on device data never trap the GPU: the verify calls write a
 *     per-stream status code (SPEC_ST_*) and that stream emits nothing.
 *   - Greedy rows: a stream whose temperature is exactly 0 takes the greedy branch in both
 *     verify calls ([P1] §4 "Greedy is a different code path").
 *   - Random numbers: Philox4x32-10 (Salmon et al., SC'11), key = (seed lo, seed hi),
 *     counter = (slot, stream, step lo, step hi).  Output word 0 is the acceptance uniform
 *     of draft slot `slot` (u_slot for the token-wise rule, eta_{slot+1} for block
 *     verification); word 1 is the sampling uniform used when the step ends at `slot`; word 2
 *     is the draft-side uniform of slot `slot` (dspark_markov_walk).
 *     U(x) = ((x >> 8) + 0.5) * 2^-24.  Same (seed, step) => bit-identical outputs.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPECVERIFY_VERSION 1

/* dtypes */
#define SPEC_DTYPE_F32 0
#define SPEC_DTYPE_BF16 1

/* host-visible return codes */
#define SPEC_OK 0
#define SPEC_ERR_ARG (-1)      /* NULL pointer or invalid enum value */
#define SPEC_ERR_DTYPE (-2)    /* unsupported dtype combination */
#define SPEC_ERR_SHAPE (-3)    /* size out of the supported range */
#define SPEC_ERR_CUDA (-4)     /* a CUDA runtime call or launch failed */
#define SPEC_ERR_DEVICE (-5)   /* the current device cannot run these kernels */
#define SPEC_ERR_WORKSPACE (-6) /* workspace missing, too small or misaligned */

/* per-stream status codes written by the verify calls (device data errors) */
#define SPEC_ST_OK 0
#define SPEC_ST_BAD_TEMPERATURE 1 /* T is NaN, infinite, negative, or positive but below FLT_MIN */
#define SPEC_ST_BAD_TOKEN 2       /* a draft token of the stream lies outside [0, V) */
#define SPEC_ST_BAD_ROW 3         /* a read logit row holds NaN or +inf, or has no finite entry */
#define SPEC_ST_ZERO_DRAFT_PROB 4 /* T > 0 and q_i(x_i) = 0 (the draft logit at x_i is -inf) */
#define SPEC_ST_BAD_OFFSETS 5     /* cu_drafts[0] != 0, or the count of stream b or of an
                                     earlier stream is negative or above kmax */
#define SPEC_ST_TIMEOUT 6         /* a bounded device wait gave up, or the workspace was not zero-filled */
#define SPEC_ST_NUMERIC 7         /* the distribution to draw from has zero or non-finite mass */

/* limits */
#define SPEC_MAX_KMAX 32          /* drafts per stream */
#define SPEC_MAX_V 16777216       /* vocabulary size */

/* columns of the optional diag output (one row per target row) */
#define SPEC_DIAG_COLS 8
#define SPEC_DIAG_PX 0     /* p_i(x_i) */
#define SPEC_DIAG_QX 1     /* q_i(x_i) */
#define SPEC_DIAG_W 2      /* block: clipped running product w_i (w_0 = 1) */
#define SPEC_DIAG_H 3      /* block: threshold h_i, where it was evaluated */
#define SPEC_DIAG_R 4      /* residual mass r_i, where it was computed */
#define SPEC_DIAG_LOGZP 5  /* natural log of sum_v exp(l^p_i[v] / T) */
#define SPEC_DIAG_LOGZQ 6  /* natural log of sum_v exp(l^q_i[v] / T) */
#define SPEC_DIAG_RHO 7    /* rho_i = p_i(x_i) / q_i(x_i) */

/*
 * dspark_markov_bias - the Markov head's previous-token logit bias.
 * [P2] §6 "Why the Markov Head Helps": B = W1 @ W2 (default rank 256), added to the current
 * draft logits from the previous token; [P1] §3 "The Markov fix-up" and Figure 2: each
 * slot's logits are biased by the token sampled one slot earlier (slot 0: the anchor).
 *
 *   out[r, v] = draft[r, v] + sum_{j < rank} W1[prev[r], j] * W2[j, v]     (float32)
 *
 * draft_logits [rows, V] (draft_dtype), prev_tokens [rows] int32, W1 [V, rank] and
 * W2 [rank, V] (w_dtype), out_logits [rows, V] float32.  out may alias draft_logits only
 * when draft_dtype is F32 (in place).  A row whose prev token lies outside [0, V) is written
 * as all NaN (a later verify call reports it as SPEC_ST_BAD_ROW).
 * Errors: SPEC_ERR_ARG (NULL pointer), SPEC_ERR_DTYPE, SPEC_ERR_SHAPE (rows < 0, V < 1,
 * V > SPEC_MAX_V, rank < 1 or rank > 1024, or an alias with a bf16 input).
 * rows == 0 launches nothing.
 */
int dspark_markov_bias(const void* draft_logits, int32_t draft_dtype, int32_t rows, int32_t V,
                       const int32_t* prev_tokens, const void* W1, const void* W2,
                       int32_t w_dtype, int32_t rank, float* out_logits, void* stream);

/*
 * dspark_markov_walk - the draft-side Markov walk: bias slot i by the token sampled at slot
 * i - 1, then sample t_i, left to right ([P1] §3 "The Markov fix-up" and Figure 2; [P2] §6):
 *
 *   l~_i = l_i + W1[t_{i-1}] @ W2   (t_{-1} = anchor[b]),   t_i ~ softmax(l~_i / T_b)
 *
 * The draw is the verify calls' inverse CDF with the draft-side uniform: word 2 of the Philox
 * output for (slot i, stream b, step) under `seed` (the verify uses words 0 and 1 of the same
 * counter, so the two draws are independent); T_b = 0 takes the argmax (lowest index).
 * draft_logits [B, N, V] (draft_dtype) are the drafter's unbiased slot logits; W1 [V, rank],
 * W2 [rank, V] (w_dtype); anchor [B] int32; temperature [B] float.  Outputs: out_tokens
 * [B, N] int32 (the draft tokens; -1 from a slot a stream could not sample on), out_logits
 * [B, N, V] float32 (the biased rows: the draft logits a verify call takes), status [B]:
 * SPEC_ST_OK, BAD_TEMPERATURE, BAD_TOKEN (anchor outside [0, V)), BAD_ROW (a biased row with
 * NaN, +inf or no finite entry; the stream stops there), TIMEOUT (a bounded grid wait gave up).
 * workspace: dspark_markov_walk_workspace_bytes(B) bytes of device scratch, 16-byte aligned,
 * any contents (the call clears what it needs).  One cooperative launch: N slots for every
 * group of four streams (one stream alone: a group of one), one grid-wide barrier per slot.
 * Errors: SPEC_ERR_ARG (NULL pointer), SPEC_ERR_DTYPE, SPEC_ERR_SHAPE (B < 0, N outside
 * [0, SPEC_MAX_KMAX], V outside [1, SPEC_MAX_V], rank outside [1, 1024]), SPEC_ERR_WORKSPACE,
 * SPEC_ERR_CUDA.  B == 0 launches nothing.
 */
int dspark_markov_walk(const void* draft_logits, int32_t draft_dtype, int32_t B, int32_t N, int32_t V,
                       const int32_t* anchor, const void* W1, const void* W2, int32_t w_dtype, int32_t rank,
                       const float* temperature, uint64_t seed, uint64_t step, int32_t* out_tokens,
                       float* out_logits, int32_t* status, void* workspace, size_t workspace_bytes,
                       void* stream);
size_t dspark_markov_walk_workspace_bytes(int32_t B);

/*
 * Arguments shared by both verify calls.  B streams; stream b has
 * N_b = cu_drafts[b+1] - cu_drafts[b] drafts (0 <= N_b <= kmax), packed from row 0
 * (cu_drafts[0] = 0).  From the first stream that breaks this on, every stream reports
 * SPEC_ST_BAD_OFFSETS, since its rows no longer have a defined position.
 *   draft row of (b, i)  = cu_drafts[b] + i          (i < N_b)
 *   target row of (b, i) = cu_drafts[b] + b + i      (i <= N_b; i = N_b is the bonus slot)
 * Inputs (device): cu_drafts [B+1] int32; draft_logits [cu[B], V]; target_logits
 * [cu[B] + B, V]; draft_tokens [cu[B]] int32; temperature [B] float (0 = greedy).
 * Outputs (device, fully written for every stream): accepted_len [B] int32 (tau);
 * out_tokens [B, kmax+1] int32 = x_0 .. x_{tau-1}, then the target's token, then -1;
 * n_emitted [B] int32 = tau + 1 (0 when status != 0); status [B] int32 (SPEC_ST_*).
 * diag is optional (NULL = not written): float [cu[B] + B, SPEC_DIAG_COLS], NaN where a
 * value was not computed.
 * workspace: device scratch of at least spec_verify_workspace_bytes(B, kmax) bytes, zero-filled
 * once before its first use (each call leaves it in a valid state for the next); calls that
 * share a workspace must be ordered (same stream).
 * Rows read: T > 0 reads all 2 N_b + 1 rows of the stream; T = 0 reads the N_b + 1 target
 * rows only.  Status precedence: BAD_OFFSETS, BAD_TEMPERATURE, BAD_TOKEN, BAD_ROW,
 * ZERO_DRAFT_PROB, NUMERIC.
 * The caller must make the arrays at least as long as cu_drafts[B] implies; the kernels
 * read cu_drafts on the device and cannot check buffer lengths.
 */
typedef struct {
    int32_t B;
    int32_t V;
    int32_t kmax;
    const int32_t* cu_drafts;
    const void* draft_logits;
    int32_t draft_dtype;
    const void* target_logits;
    int32_t target_dtype;
    const int32_t* draft_tokens;
    const float* temperature;
    uint64_t seed;
    uint64_t step;
    int32_t* accepted_len;
    int32_t* out_tokens;
    int32_t* n_emitted;
    int32_t* status;
    float* diag;
    void* workspace;
    size_t workspace_bytes;
} spec_verify_args;

/*
 * spec_verify_workspace_bytes - device workspace a verify call over B streams with up to
 * kmax drafts each needs (16-byte aligned, caller-allocated; 0 for B = 0 and for invalid
 * arguments): 256 + 1536 B (2 kmax + 1) + 2048 B (kmax + 1) bytes.  It holds the claim tickets
 * of the two persistent kernels, per row the statistics partials and a counter of the pieces
 * published, the per-slot and per-stream scalars that one kernel of the call hands to the
 * next, and the residual sweep's work list.  Zero-fill it once before the first call; every
 * call returns its tickets and counters to zero (also when a bounded wait gave up), so the
 * workspace may then be reused by later calls on the same stream, for any B and kmax that fit.
 */
size_t spec_verify_workspace_bytes(int32_t B, int32_t kmax);

/*
 * spec_verify_tokenwise - token-by-token speculative sampling.
 * [P1] §4 "Token by token" (Leviathan et al. 2023): walk the drafts in order and accept x_i
 * while u_i <= min(1, p_i(x_i) / q_i(x_i)); at the first rejection j emit a token drawn
 * from max(0, p_j - q_j) (normalised) and stop; if all N drafts pass emit the bonus drawn
 * from p_N.  p_i = softmax(target_i / T), q_i = softmax(draft_i / T).  Draws are inverse
 * CDF: the smallest v with C(v) >= U * R (ascending vocabulary order).
 * Errors: SPEC_ERR_ARG, SPEC_ERR_DTYPE, SPEC_ERR_SHAPE (B < 0, V < 1, V > SPEC_MAX_V,
 * kmax < 0 or kmax > SPEC_MAX_KMAX), SPEC_ERR_WORKSPACE, SPEC_ERR_CUDA.  B == 0 launches
 * nothing.
 */
int spec_verify_tokenwise(const spec_verify_args* args, void* stream);

/*
 * spec_verify_block - block verification.
 * [P1] §4 "Block verification" (Sun et al. 2024) and Figure 3: with the clipped running
 * product w_0 = 1, w_{i+1} = min(1, w_i p_i(x_i) / q_i(x_i)), the residual mass
 * r_i = sum_v max(0, w_i p_i(v) - q_i(v)) and the threshold h_i = r_i / (r_i + 1 - w_i)
 * (i < N; h_N = w_N; 0/0 reads as 1), the accepted length is tau = the last i >= 1 with
 * eta_i <= h_i (0 if none); emit x_0 .. x_{tau-1} and a token drawn from
 * max(0, w_tau p_tau - q_tau) (tau < N) or from p_N (tau = N).
 * Errors: as spec_verify_tokenwise.
 */
int spec_verify_block(const spec_verify_args* args, void* stream);

/*
 * spec_verify_tokenwise_reduced / spec_verify_block_reduced - the same verify calls with the
 * draft rows over a reduced draft vocabulary.
 * [P1] §3 "The Markov fix-up": the drafter scores a reduced vocabulary and scatters those
 * logits into target-vocabulary columns, so the draft distribution is zero outside it.  The
 * verify is, by definition, the dense verify of the scattered rows: draft logit of target
 * column v = draft_logits[row, t2d[v]] when 0 <= t2d[v] < K, and -inf otherwise.
 * args->draft_logits is [cu_drafts[B], K] (draft_dtype); everything else as in the dense
 * calls (draft tokens are target-vocabulary ids; one outside the draft vocabulary gives
 * SPEC_ST_ZERO_DRAFT_PROB at T > 0).  t2d [V] int32 (device): the inverse of the map from draft
 * ids to target columns - every draft id in [0, K) must appear exactly once (the call does
 * not check this; with a duplicate or a missing id the result is that of the column-wise
 * definition above, which is then no distribution scattered from the draft rows).  Only the
 * target rows are read in full: the draft rows are read once (K logits each) and gathered
 * through t2d where the residual is summed.  The workspace is that of the dense calls.
 * Errors: those of the dense calls, SPEC_ERR_ARG (t2d NULL), SPEC_ERR_SHAPE (K outside [1, V]).
 */
int spec_verify_tokenwise_reduced(const spec_verify_args* args, const int32_t* t2d, int32_t K, void* stream);
int spec_verify_block_reduced(const spec_verify_args* args, const int32_t* t2d, int32_t K, void* stream);

/*
 * spec_verify_block_static - spec_verify_block without a caller workspace: the workspace is a
 * fixed device array of 16 MiB (16,777,216 bytes) that the library reserves when it is loaded,
 * so the call allocates no memory at all.  It is for callers that cannot allocate device memory
 * where they verify (an allocator that is not theirs to touch, a memory budget fixed at
 * start-up).  It is an engineering variant of the block verification above; the pages that
 * define the method have no counterpart to it.
 * args->workspace and args->workspace_bytes are ignored.  Capacity: a batch whose
 * spec_verify_workspace_bytes(B, kmax) exceeds the array (e.g. B = 512 at kmax = 16) returns
 * SPEC_ERR_WORKSPACE and launches nothing; B = 256 at kmax = 15 (15.6 MiB) fits.  The argument
 * checks of spec_verify_block come first, so a bad shape or dtype gets the same code as there.
 * The array starts zero-filled like every device variable, and every call leaves it so.
 * Every call on a device shares it: calls that can overlap in time (different streams or host
 * threads) race on it, so the caller must order them.  The first call on each device looks the
 * array's address up (cudaGetSymbolAddress) and keeps it for the life of the process: make
 * that first call outside any stream capture, and do not use this call across a reset of the
 * device's context (cudaDeviceReset), after which the kept address is no longer valid.
 * Errors: as spec_verify_block, plus SPEC_ERR_WORKSPACE for a batch above the capacity.
 */
int spec_verify_block_static(const spec_verify_args* args, void* stream);

/*
 * spec_verify_launch_info - the launch configuration a verify call with these arguments
 * would use (no launch, no device data read; only the scalar fields and the two logit
 * pointers' alignment are examined).  cluster_size: CTAs that one stream's decision and draw
 * use (1: one CTA per stream); resident_clusters: CTAs of the persistent residual-sweep grid
 * (all resident at once); elems_per_load: 8 when the rows take the 16-byte vector path, 1
 * otherwise.
 * Errors: as spec_verify_tokenwise (without the NULL checks of the tensor pointers), and
 * SPEC_ERR_ARG when an output pointer is NULL.
 */
int spec_verify_launch_info(const spec_verify_args* args, int32_t* cluster_size,
                            int32_t* resident_clusters, int32_t* elems_per_load);

/*
 * adaptive_pick_k - confidence head and adaptive verification.
 * [P2] §7 "Only Then Comes the Confidence Head": c_k = sigmoid(h_k . w + bias);
 * §9 "Why It Is Called Prefix Survival Probability": a_j = c_1 ... c_j;
 * [P1] §6: a stream that verifies n drafts expects E_n = 1 + a_1 + ... + a_n tokens;
 * [P3] "The controller, and the table it reads from": pick the count with the best
 * expected tokens per millisecond, the cost read from verify_ms[num_tokens].
 *   mode 0 (per stream): k_b = argmax_{n in 0..kmax} E_n / verify_ms[n + 1], ties -> smaller n.
 *   mode 1 (batch, greedy in descending a - figure text after [P2] §9): order every (b, j)
 *     by (a desc, b asc, j asc), m* = argmax_m (B + a-sum of the first m) / verify_ms[B + m]
 *     (ties -> smaller m), k_b = the number of stream b's entries among the first m*.
 * hidden [B, kmax, H] and w [H] in `dtype`; verify_ms [n_max + 1] float (index = tokens in
 * the verify pass; index 0 unused).  Outputs: c_out [B, kmax] float, a_out [B, kmax] float,
 * k_out [B] int32, cu_drafts_out [B + 1] int32 (exclusive prefix sum of k).
 * Errors: SPEC_ERR_ARG (NULL pointer, mode not 0/1), SPEC_ERR_DTYPE, SPEC_ERR_SHAPE
 * (B < 1, kmax < 1 or > SPEC_MAX_KMAX, H < 1, n_max < kmax + 1 in mode 0 or
 * n_max < B * (kmax + 1) in mode 1, B * kmax > 4096 in mode 1), SPEC_ERR_CUDA.
 */
int adaptive_pick_k(const void* hidden, const void* w, int32_t dtype, float bias, int32_t B,
                    int32_t kmax, int32_t H, const float* verify_ms, int32_t n_max,
                    int32_t mode, float* c_out, float* a_out, int32_t* k_out,
                    int32_t* cu_drafts_out, void* stream);

/*
 * spec_accept_counters - per-position acceptance counts of a batch's verify results.
 * [P1] §6 "The arithmetic you need before tuning k": a_p, the share of steps whose p-th
 * draft was accepted, and tokens per step = 1 + sum_p a_p (the emitted tokens tau + 1).
 * Adds to counts [2 kmax + 1] (uint64, device, accumulated over calls; zero it to start):
 *   counts[0]        += streams with status SPEC_ST_OK (the steps);
 *   counts[p]        += OK streams with accepted_len >= p, p = 1..kmax (accepted at p);
 *   counts[kmax + p] += OK streams that verified at least p drafts (offered at p).
 * a_p = counts[p] / counts[0]; the marginal rate a_p / a_{p-1}; tokens per step
 * 1 + sum_p a_p.  accepted_len, status [B] and cu_drafts [B + 1] as written / read by a
 * verify call.  Errors: SPEC_ERR_ARG (NULL pointer), SPEC_ERR_SHAPE (B < 0, kmax outside
 * [0, SPEC_MAX_KMAX]), SPEC_ERR_CUDA.  B == 0 launches nothing.
 */
int spec_accept_counters(const int32_t* accepted_len, const int32_t* status, const int32_t* cu_drafts,
                         int32_t B, int32_t kmax, uint64_t* counts, void* stream);

/*
 * The adaptive verify step as one CUDA graph: adaptive_pick_k (confidence head, prefix
 * survival, k_b per stream and the offsets cu_drafts_out) -> the verify of each stream's
 * first k_b drafts -> spec_accept_counters -> *step += 1.  [P1] §3 "The Markov fix-up" (the
 * sampling runs inside the same CUDA graph as the draft pass) and "Two cliffs, not one" (one
 * graph per batch size); [P3] "The controller, and the table it reads from" (the controller
 * picks how many drafts each stream verifies).
 * Layout: the drafter fills all kmax slots of every stream and the target scores all of
 * them, so draft_logits is [B, kmax, V] (row b kmax + i), target_logits [B, kmax + 1, V]
 * (row b (kmax + 1) + i, i <= k_b, row b (kmax + 1) + k_b is the bonus slot of the k_b
 * verified drafts), draft_tokens [B, kmax]; a stream verifies its first k_b drafts.
 * The Philox step of each launch is read from the device word *step (uint64), which the
 * graph increments at its end; every other argument is fixed at creation (device pointers
 * must stay valid while the pipeline lives; outputs as in adaptive_pick_k and the verify
 * calls, diag [B (kmax + 1), SPEC_DIAG_COLS] in the dense target-row order; accept_counts may
 * be NULL).  The workspace (spec_verify_workspace_bytes(B, kmax), zero-filled once) belongs
 * to the pipeline while it lives; launches of one pipeline must be ordered (one stream).
 */
typedef struct {
    /* confidence head and controller (see adaptive_pick_k) */
    const void* hidden;        /* [B, kmax, H] */
    const void* w;             /* [H] */
    int32_t head_dtype;
    float bias;
    int32_t H;
    const float* verify_ms;    /* [n_max + 1] */
    int32_t n_max;
    int32_t mode;              /* 0 per stream, 1 batch-greedy */
    /* verification */
    int32_t rule;              /* 0 token-wise, 1 block */
    int32_t B, V, kmax;
    const void* draft_logits;  /* [B, kmax, V] */
    int32_t draft_dtype;
    const void* target_logits; /* [B, kmax + 1, V] */
    int32_t target_dtype;
    const int32_t* draft_tokens;   /* [B, kmax] */
    const float* temperature;      /* [B] */
    uint64_t seed;
    uint64_t* step;            /* device, 1 word: this launch's step; incremented by the graph */
    /* outputs */
    float* c_out;              /* [B, kmax] */
    float* a_out;              /* [B, kmax] */
    int32_t* k_out;            /* [B] */
    int32_t* cu_drafts_out;    /* [B + 1] */
    int32_t* accepted_len;     /* [B] */
    int32_t* out_tokens;       /* [B, kmax + 1] */
    int32_t* n_emitted;        /* [B] */
    int32_t* status;           /* [B] */
    float* diag;               /* optional */
    uint64_t* accept_counts;   /* optional [2 kmax + 1], accumulated */
    void* workspace;
    size_t workspace_bytes;
} spec_pipeline_args;

/* Capture the graph (nothing runs yet).  *pipeline receives an opaque handle.  Errors: those
 * of adaptive_pick_k and the verify calls, SPEC_ERR_ARG (NULL pointer, rule not 0/1). */
int spec_pipeline_create(const spec_pipeline_args* args, void** pipeline);
/* Run one step: one graph launch on `stream`. */
int spec_pipeline_launch(void* pipeline, void* stream);
/* Release the graph (NULL is accepted). */
int spec_pipeline_destroy(void* pipeline);

/*
 * The online verify-cost curve (host code; the table adaptive_pick_k reads).
 * [P3] "What we changed": a pair of CUDA events is recorded around every real verification
 * step; the elapsed time is read later without making the host wait, and filed under the
 * step's token count (the tokens in the verify pass); every rebuild_every observations the
 * table is rebuilt from the boot curve with the median of the last `window` observations of
 * every count that has at least min_samples of them laid on top ([P3] "Reproduce": window
 * 32, min samples 3, rebuild every 32).  The median of an even number of samples is the
 * mean of the two middle ones.  A curve belongs to one host thread at a time.
 *
 * spec_cost_curve_create: boot_ms [n_max + 1] host floats (copied; index = token count).
 *   Returns an opaque handle, or NULL (spec_last_error says why: boot_ms NULL, n_max < 1,
 *   window < 1, min_samples outside [1, window], rebuild_every < 1).  Touches no device.
 * spec_cost_curve_begin / spec_cost_curve_end: bracket one verification step on `stream`
 *   (a stream that is not being captured: SPEC_ERR_ARG otherwise).  The step's token count is
 *   num_tokens, plus *device_count when device_count is not NULL (e.g. cu_drafts_out[B] of
 *   adaptive_pick_k, with num_tokens = B for the bonus rows); that int32 is stored into mapped
 *   pinned memory by a one-thread kernel launched after the end event, outside the timed
 *   region.  When 64 steps are
 *   still pending the step goes unobserved (counted as dropped).  Unmatched begin/end:
 *   SPEC_ERR_ARG.
 * spec_cost_curve_poll: folds every completed step, oldest first, into the windows; never
 *   waits (a step still running stays pending).  Steps whose count falls outside [0, n_max]
 *   are dropped.
 * spec_cost_curve_observe: files one observation directly (host clocks, tests); touches no
 *   device.
 * spec_cost_curve_table: out [n_max + 1] host floats = the table as last rebuilt (the boot
 *   curve until the first rebuild); counters [4] (may be NULL) = observations filed, rebuilds,
 *   dropped, steps pending.  Touches no device.
 * spec_cost_curve_upload: when the table changed since the last upload, queues its copy into
 *   device_table [n_max + 1] floats on `stream` from one of two pinned buffers (a buffer whose
 *   previous copy is still in flight is not overwritten: the upload is then deferred to the
 *   next call).  A graph that reads device_table (spec_pipeline_create's verify_ms) sees the
 *   new table from its next launch on that stream.
 * spec_cost_curve_destroy: waits for the curve's own pending copies, then frees it (NULL ok).
 */
void* spec_cost_curve_create(const float* boot_ms, int32_t n_max, int32_t window, int32_t min_samples,
                             int32_t rebuild_every);
int spec_cost_curve_begin(void* curve, void* stream);
int spec_cost_curve_end(void* curve, int32_t num_tokens, const int32_t* device_count, void* stream);
int spec_cost_curve_poll(void* curve);
int spec_cost_curve_observe(void* curve, int32_t num_tokens, float ms);
int spec_cost_curve_table(void* curve, float* out, int64_t* counters);
int spec_cost_curve_upload(void* curve, float* device_table, void* stream);
void spec_cost_curve_destroy(void* curve);

/*
 * spec_philox_uniforms - the verify calls' uniforms, exposed for checking.
 * out [n_streams, n_slots, 2] double: (acceptance uniform, sampling uniform) of every
 * (stream, slot) for the given seed and step, exactly as the verify kernels draw them.
 * Errors: SPEC_ERR_ARG (NULL out), SPEC_ERR_SHAPE (a negative count), SPEC_ERR_CUDA.
 */
int spec_philox_uniforms(uint64_t seed, uint64_t step, int32_t n_streams, int32_t n_slots,
                         double* out, void* stream);

/* One-line description of the last error returned in the calling host thread ("" if none). */
const char* spec_last_error(void);

/* SPECVERIFY_VERSION of the loaded library. */
int32_t spec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
