/*
 * uno.h -- C ABI of the Uno draft+verify hot path (libuno.so, sm_103a).
 *
 * Two operations make up one decoding step of a diffusion-augmented LLM:
 *
 *   1. the gated-LoRA linear projection
 *          y = x.W_AR^T + g_row * (alpha/rank) * (x.A^T).B^T
 *      where draft rows (gate 1) use the AR weights plus the diffusion
 *      adapter and verification rows (gate 0) use the AR weights only
 *      ("Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
 *      aifromscratch.in explainer, section "Two Decoupled Weight Sets":
 *      the adapters have rank 128 and alpha 256 and are coupled through a
 *      gate);
 *
 *   2. the block verifier of the Psi-Spec linear sampler: rejection sampling
 *      of a drafted block against the AR distribution that accepts the
 *      drafts up to the first rejection and leaves the emitted tokens
 *      distributed exactly as the AR model's
 *      (same page, section "The Psi-Spec Sampler"; "Uno Uses Discrete
 *      Diffusion to Accelerate LLMs Without Loss", cctest.ai, section
 *      "What 'lossless' means here").
 *
 * A third entry point draws the drafted block itself (a single token at each
 * position, the linear sampler's drafting half).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory owned by the caller, except
 *     where an argument says otherwise.  The library allocates no device or
 *     host memory on the compute path and keeps no per-call state.  (It
 *     caches the driver entry point used to encode TMA descriptors and the
 *     per-device SM count and kernel attributes; these caches assume that
 *     the process does not call cudaDeviceReset and then use the library
 *     again.)
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call is asynchronous and stream-ordered; the library never
 *     synchronises.  Workspace must not be shared by calls that may overlap
 *     on the GPU.
 *   - Host-detectable errors (null pointers, bad sizes, misalignment, small
 *     workspace) return a negative uno_status before anything is enqueued.
 *     A CUDA launch error returns UNO_ERR_CUDA.  Errors the GPU detects in
 *     the data (a draft id outside [0,V), a NaN or +inf logit) are reported
 *     per sequence in `status` (see UNO_SEQ_*), never by trapping.
 *   - Row-major layouts; "[a,b]" means a rows of b contiguous elements.
 *   - Sizes are int64_t; a size of 0 where allowed is a no-op returning
 *     UNO_OK.
 *   - Device pointers must be 16-byte aligned.
 */
#ifndef UNO_H_
#define UNO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *uno_stream_t;

typedef enum {
    UNO_OK = 0,
    UNO_ERR_ARG = -1,         /* null pointer, negative or unsupported size */
    UNO_ERR_ALIGN = -2,       /* pointer or row stride not 16-byte aligned  */
    UNO_ERR_UNSUPPORTED = -3, /* dtype or shape outside what is built       */
    UNO_ERR_WORKSPACE = -4,   /* ws_bytes smaller than the query returned   */
    UNO_ERR_CUDA = -5         /* a CUDA runtime/driver call failed          */
} uno_status;

typedef enum {
    UNO_F32 = 0,  /* float32 inputs and output (inputs rounded to bf16 for the
                     tensor cores, fp32 accumulation, fp32 output)          */
    UNO_BF16 = 1  /* bfloat16 inputs and output, fp32 accumulation         */
} uno_dtype;

/* Per-sequence (or per-row) status written by the device. */
enum {
    UNO_SEQ_OK = 0,
    UNO_SEQ_BAD_DRAFT = 1, /* a draft id outside [0, V)                     */
    UNO_SEQ_NONFINITE = 2  /* a NaN or +inf logit, or a row that is all -inf */
};

/* ---------------------------------------------------------------------------
 * Gated-LoRA linear projection
 *   y[m,n] = sum_k x[m,k] W[n,k] + gate[m] * (alpha/rank) * sum_j T[m,j] B[n,j]
 *   T[m,j] = sum_k x[m,k] A[j,k]
 * ("Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
 *  aifromscratch.in, "Two Decoupled Weight Sets".)
 *
 *   x    [M, d_in]      activations (dtype)
 *   W    [d_out, d_in]  theta_AR, nn.Linear layout (dtype)
 *   A    [rank, d_in]   theta_Delta down-projection (dtype)
 *   B    [d_out, rank]  theta_Delta up-projection (dtype)
 *   gate [M]            uint8 per row: 1 = draft row, 0 = verification row
 *                       (any other value is used as the multiplier itself)
 *   y    [M, d_out]     output (dtype); must not alias any input
 *   workspace           device scratch of at least
 *                       uno_gated_lora_linear_workspace(...) bytes, 256-byte
 *                       aligned; contents on entry are ignored.
 * Arithmetic: bf16 operands on the tcgen05 tensor cores, fp32 accumulation
 * in tensor memory.  (x.A^T) is scaled by gate*alpha/rank in fp32 and
 * rounded to bf16 before the up-projection, which runs as extra K-blocks of
 * the same accumulator as x.W^T.  Gate-0 rows therefore equal the plain
 * x.W^T of the same kernel bit for bit.  Deterministic: the same inputs
 * give the same bits on every call.
 * Requirements: M >= 0, d_in >= 1, d_out >= 1, rank in [0, 256], d_in,
 * d_out and rank multiples of 8; alpha finite.  rank == 0 gives x.W^T.
 * Residency: the kernel is persistent (one CTA per SM) and some CTAs wait,
 * with a 2-second limit, for partial sums that other CTAs of the same launch
 * publish (of output tiles and, for up to 64 rows, of the adapter input
 * x.A^T, which the CTAs compute by splitting d_in).  Large M (more than 128
 * rows, with little padding of 256-row tiles) runs as clusters of two CTAs
 * that share each 256-row tile through the pair MMA, no more clusters than
 * the runtime reports resident; their output tiles wait, with the same limit,
 * for the adapter-input tiles of the same launch.  When other work keeps SMs from this launch (another
 * stream's long kernel, an MPS or green-context SM limit) such a wait can run
 * out; the CTA then skips its output tile and sets bit 0 of the device error
 * word.  y is therefore defined only when uno_device_error() reads 0 after
 * the call; a caller that shares the GPU should check it.
 * The workspace query returns the bytes for the device current at the time
 * of the call; use the same device for the compute call.
 * ------------------------------------------------------------------------- */
size_t uno_gated_lora_linear_workspace(int64_t M, int64_t d_in, int64_t d_out,
                                       int64_t rank, int dtype);

int uno_gated_lora_linear(const void *x, const void *W, const void *A,
                          const void *B, const uint8_t *gate, int64_t M,
                          int64_t d_in, int64_t d_out, int64_t rank,
                          float alpha, int dtype, void *y, void *workspace,
                          size_t ws_bytes, uno_stream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped gated-LoRA projections: up to UNO_MAX_LORA_PROBLEMS projections
 * that share the row count M (for instance the q/k/v/o/gate/up/down
 * projections of one transformer layer, each with its own input, weights,
 * adapter and gate) computed by ONE persistent kernel launch.  Each problem
 * follows exactly the definition of uno_gated_lora_linear above, with the
 * same error bound.  The schedule splits the concatenated K loops of all
 * problems evenly over the SMs (so small projections leave no SM idle); a
 * K loop cut between two CTAs is summed in a fixed order, so results are
 * deterministic for a given group, but a problem computed alone may be cut
 * elsewhere and differ in the last bits.  uno_gated_lora_linear is this
 * call with n = 1.
 *   problems  HOST array of n descriptors (device pointers inside)
 *   M         rows of every x, gate and y
 *   workspace at least uno_gated_lora_linear_batched_workspace(...) bytes,
 *             256-byte aligned, contents ignored on entry.
 * Requirements: 1 <= n <= UNO_MAX_LORA_PROBLEMS; per problem as above.
 * ------------------------------------------------------------------------- */
#define UNO_MAX_LORA_PROBLEMS 8

typedef struct {
    const void *x;       /* [M, d_in]      activations (dtype)                */
    const void *W;       /* [d_out, d_in]  theta_AR (dtype)                   */
    const void *A;       /* [rank, d_in]   theta_Delta down-projection (dtype)*/
    const void *B;       /* [d_out, rank]  theta_Delta up-projection (dtype)  */
    const uint8_t *gate; /* [M]            1 = draft row, 0 = verification row */
    void *y;             /* [M, d_out]     output (dtype)                     */
    int64_t d_in;
    int64_t d_out;
    int64_t rank;
    float alpha;
} uno_lora_problem;

/* Diagnostic, host only (no GPU, no CUDA call): builds the schedule that
 * uno_gated_lora_linear_batched would use on a GPU with `sms` SMs and checks
 * its invariants -- the grid fits one CTA per SM, every section's K-blocks
 * are partitioned over the CTAs in order, a split T tile's finisher takes no
 * other work (decode order) or a split T tile's pieces are whole CTA ranges
 * in consecutive CTAs (token-rows order), the adapter's d_in chunks cover every adapted problem with at
 * most one chunk per CTA, a pair-order launch has an even grid and 256-row
 * tiles with the adapter-input tiles first, the workspace regions fit.  Returns 0 when all hold, a positive
 * invariant number otherwise, or UNO_ERR_ARG / UNO_ERR_UNSUPPORTED for
 * arguments the projection itself would refuse (pointers are not read). */
int uno_lora_plan_check(int n, const uno_lora_problem *problems, int64_t M, int dtype, int sms);

size_t uno_gated_lora_linear_batched_workspace(int n, const uno_lora_problem *problems,
                                               int64_t M, int dtype);

int uno_gated_lora_linear_batched(int n, const uno_lora_problem *problems, int64_t M,
                                  int dtype, void *workspace, size_t ws_bytes,
                                  uno_stream_t stream);

/* ---------------------------------------------------------------------------
 * Block verifier (Psi-Spec linear sampler, verification half).
 * ("Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
 *  aifromscratch.in, "The Psi-Spec Sampler"; "Uno Uses Discrete Diffusion to
 *  Accelerate LLMs Without Loss", cctest.ai, "What 'lossless' means here".)
 *
 * For each sequence b, with p_i = softmax(p_logits[b,i,:]) and
 * q_i = softmax(q_logits[b,i,:]) (temperature 1):
 *   accept draft i iff u_accept[b,i] < min(1, p_i(x_i) / q_i(x_i)),
 *   n = length of the accepted prefix;
 *   if n < K: one token from max(0, p_n - q_n) normalised (p_n if that is
 *             all zero), drawn by the exponential race
 *             argmax_v r(v) / (-ln u_resample[b,v]);
 *   else if Kp == K+1: the bonus token from p_K by the same race;
 *   out_tokens[b,0..n-1] = drafts, out_tokens[b,n] = the drawn token,
 *   remaining entries -1; n_emitted[b] = n + (a token was drawn).
 *
 *   p_logits   [Bn, Kp, V] float32 AR logits, Kp == K or K+1
 *   q_logits   [Bn, K, V]  float32 draft logits
 *   draft      [Bn, K]     int32 drafted ids
 *   u_accept   [Bn, K]     float32 in [0,1)
 *   u_resample [Bn, V]     float32 in (0,1)
 *   n_accepted [Bn], out_tokens [Bn, K+1], n_emitted [Bn], status [Bn]
 *              int32 outputs; a sequence with status != 0 has n = 0,
 *              n_emitted = 0 and out_tokens all -1.
 *   workspace  at least uno_verify_block_workspace(Bn, K, Kp, V) bytes,
 *              256-byte aligned, contents ignored on entry.
 * Requirements: Bn >= 0, K >= 0, Kp in {K, K+1}, Kp >= 1, 1 <= V < 2^31.
 * Logit rows need not be 16-byte aligned (any V works).
 * ------------------------------------------------------------------------- */
size_t uno_verify_block_workspace(int64_t Bn, int64_t K, int64_t Kp, int64_t V);

int uno_verify_block(const float *p_logits, const float *q_logits,
                     const int32_t *draft, const float *u_accept,
                     const float *u_resample, int64_t Bn, int64_t K,
                     int64_t Kp, int64_t V, int32_t *n_accepted,
                     int32_t *out_tokens, int32_t *n_emitted, int32_t *status,
                     void *workspace, size_t ws_bytes, uno_stream_t stream);

/* ---------------------------------------------------------------------------
 * Block verifier with sampling variants: temperature and the resample draw.
 * (Same rule and passages as uno_verify_block; the pages sample at
 * temperature 1 and say only that the residual is resampled.)
 *   temperature  T > 0, finite: every distribution is taken at T,
 *                p_i = softmax(p_logits[b,i,:] / T), q_i likewise (the drafts
 *                are expected to come from q at the same T).  T == 1 with
 *                UNO_RESAMPLE_RACE gives exactly uno_verify_block's outputs.
 *   resample     UNO_RESAMPLE_RACE: the exponential race of uno_verify_block,
 *                u_resample [Bn, V] float32 in (0,1);
 *                UNO_RESAMPLE_INVERSE_CDF: one uniform per sequence,
 *                u_resample [Bn] float32 in [0,1); the token is the smallest v
 *                whose cumulative weight (vocabulary order) exceeds u * S,
 *                S the weights' sum; fp32 weights are summed exactly in
 *                integer units of 2^-46.  Its result agrees with an fp64
 *                evaluation except when u * S falls within rounding of a
 *                bucket edge.
 * Other arguments, outputs, workspace and requirements as uno_verify_block;
 * UNO_ERR_ARG for a temperature that is not finite and positive or an
 * unknown mode.
 * ------------------------------------------------------------------------- */
enum { UNO_RESAMPLE_RACE = 0, UNO_RESAMPLE_INVERSE_CDF = 1 };

int uno_verify_block_ex(const float *p_logits, const float *q_logits,
                        const int32_t *draft, const float *u_accept,
                        const float *u_resample, int64_t Bn, int64_t K,
                        int64_t Kp, int64_t V, float temperature, int resample,
                        int32_t *n_accepted, int32_t *out_tokens,
                        int32_t *n_emitted, int32_t *status, void *workspace,
                        size_t ws_bytes, uno_stream_t stream);

/* ---------------------------------------------------------------------------
 * Block verifier that allocates nothing (the paper has no counterpart: this is
 * a library convenience).  For callers that cannot provide device scratch --
 * e.g. an op embedded in another runtime that receives only its input and
 * output buffers, or a serving path whose memory belongs to a pool it may not
 * grow or where cudaMalloc is forbidden.  Same arguments, semantics and
 * outputs as uno_verify_block, minus the workspace: the scratch is a fixed
 * array of uno_verify_block_no_alloc_max_scratch() bytes (8 MiB) inside the
 * library, present on every GPU that loads it until the process exits.
 *   - Returns UNO_ERR_WORKSPACE, without launching anything, when the call
 *     needs more scratch than the array holds (uno_verify_block_workspace()
 *     of the same sizes is what it needs).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls share the array: calls that can overlap on the GPU (other
 *     streams, other threads) race on it; the caller must serialise them.
 *   - Calls no allocating routine (no cudaMalloc/cudaFree).
 * ------------------------------------------------------------------------- */
size_t uno_verify_block_no_alloc_max_scratch(void);

int uno_verify_block_no_alloc(const float *p_logits, const float *q_logits,
                              const int32_t *draft, const float *u_accept,
                              const float *u_resample, int64_t Bn, int64_t K,
                              int64_t Kp, int64_t V, int32_t *n_accepted,
                              int32_t *out_tokens, int32_t *n_emitted,
                              int32_t *status, uno_stream_t stream);

/* ---------------------------------------------------------------------------
 * LM head + block verifier: the verifying forward pass ends in the LM head,
 * logits = h . W^T, whose rows feed the block verifier ("Unlocking Lossless
 * Speedups in LLMs via Discrete Diffusion", aifromscratch.in, "The Psi-Spec
 * Sampler"; aiany.app summary, "Key Findings": one forward pass of the AR
 * model verifies the drafted block).  The result is uno_verify_block's on
 * p = the AR rows' logits and q = the draft rows' logits, with one LM head
 * W shared by both pathways (the adapter of the draft pathway sits in the
 * projections, not in the head).
 *
 *   h          [Bn*Kp + Bn*K, d] bf16 final hidden states: the AR rows of
 *              every sequence (row b*Kp + j), then the draft rows (row
 *              Bn*Kp + b*K + i)
 *   W          [V, d] bf16 LM head (nn.Linear layout)
 *   draft, u_accept, u_resample, outputs: as uno_verify_block
 *   mode       UNO_LM_PLAIN: the head GEMM stores every logit (fp32) and the
 *                block verifier reads them;
 *              UNO_LM_STATS_STORE: the GEMM's epilogue leaves each row's
 *                softmax statistics and drafted-token logit, the accept
 *                decisions use those, and only the resampled rows are read
 *                back from the stored logits;
 *              UNO_LM_STATS_RECOMPUTE: the epilogue leaves only the
 *                statistics (no logit reaches memory); the two rows per
 *                sequence that the resample needs are recomputed;
 *              UNO_LM_AUTO: PLAIN below 8 sequences, STATS_STORE from 8
 *                (the fastest on a B300; STATS_RECOMPUTE needs no logit
 *                buffer, the choice where workspace memory is short).
 *              All modes compute the same function (bf16 operands, fp32
 *              accumulation; they may differ in the last bits of a logit).
 *   workspace  at least uno_lm_head_verify_workspace(Bn, K, Kp, V, d, mode)
 *              bytes, 256-byte aligned, contents ignored on entry.
 * Requirements: as uno_verify_block, plus d >= 8 and V multiples of 8, and
 * h, W, u_resample 16-byte aligned.
 * ------------------------------------------------------------------------- */
enum { UNO_LM_AUTO = 0, UNO_LM_PLAIN = 1, UNO_LM_STATS_STORE = 2, UNO_LM_STATS_RECOMPUTE = 3 };

size_t uno_lm_head_verify_workspace(int64_t Bn, int64_t K, int64_t Kp, int64_t V,
                                    int64_t d, int mode);

int uno_lm_head_verify(const void *h, const void *W, const int32_t *draft,
                       const float *u_accept, const float *u_resample, int64_t Bn,
                       int64_t K, int64_t Kp, int64_t V, int64_t d, int mode,
                       int32_t *n_accepted, int32_t *out_tokens,
                       int32_t *n_emitted, int32_t *status, void *workspace,
                       size_t ws_bytes, uno_stream_t stream);

/* ---------------------------------------------------------------------------
 * Tree verifier (Psi-Spec tree sampler, verification half): several drafted
 * candidates per position, arranged in a prefix tree, verified so that the
 * emitted tokens keep the AR model's distribution ("Unlocking Lossless
 * Speedups in LLMs via Discrete Diffusion", aifromscratch.in, "The Psi-Spec
 * Sampler": the tree sampler takes the top K candidates at each position and
 * verifies them in a prefix tree, best at low batch sizes).
 *
 * Node 0 is the committed prefix; nodes 1..N are drafted tokens.  Every node
 * is a deterministic candidate, for which the lossless rule is, from the root:
 * with r = p_cur (softmax of logits[b,cur,:]) and S = 1, test the children of
 * cur in index order: accept child j (token x = token[b,j]) iff
 * u_accept[b,j] < r(x)/S; else S -= r(x), r(x) = 0 and test the next child.
 * An acceptance emits x and moves to j; when every child is rejected (or
 * there is none) one token is drawn from r (from p_cur should r be all zero)
 * by the exponential race argmax_v r(v) / (-ln u_resample[b,v]), and the walk
 * stops.  n_accepted = tokens accepted, n_emitted = n_accepted + 1.
 *
 *   logits     [Bn, N+1, V] float32: AR logits of the token after node j
 *   parent     [Bn, N+1]    int32: parent[b,0] = -1, 0 <= parent[b,j] < j
 *   token      [Bn, N+1]    int32: the token of node j (token[b,0] unused)
 *   u_accept   [Bn, N+1]    float32 in [0,1): u_accept[b,j] tests node j
 *   u_resample [Bn, V]      float32 in (0,1)
 *   n_accepted [Bn], path [Bn, N] (accepted node ids by depth, -1 padded;
 *   may be NULL when N = 0), out_tokens [Bn, N+1] (-1 padded), n_emitted
 *   [Bn], status [Bn] int32 outputs.  A malformed tree (parent or token out
 *   of range) gives UNO_SEQ_BAD_DRAFT; a NaN or +inf logit, or an all -inf
 *   row, at a node the walk reaches gives UNO_SEQ_NONFINITE; either way the
 *   sequence emits nothing (outputs -1, counts 0).
 *   workspace  at least uno_tree_verify_workspace(Bn, N, V) bytes, 256-byte
 *              aligned, contents ignored on entry.
 * Requirements: Bn >= 0, 0 <= N <= 255, 1 <= V < 2^31.
 * ------------------------------------------------------------------------- */
size_t uno_tree_verify_workspace(int64_t Bn, int64_t N, int64_t V);

int uno_tree_verify(const float *logits, const int32_t *parent,
                    const int32_t *token, const float *u_accept,
                    const float *u_resample, int64_t Bn, int64_t N, int64_t V,
                    int32_t *n_accepted, int32_t *path, int32_t *out_tokens,
                    int32_t *n_emitted, int32_t *status, void *workspace,
                    size_t ws_bytes, uno_stream_t stream);

/* ---------------------------------------------------------------------------
 * Draft sampling (Psi-Spec linear sampler, drafting half: a single token at
 * each position; "Unlocking Lossless Speedups in LLMs via Discrete Diffusion",
 * aifromscratch.in, "The Psi-Spec Sampler").
 *   tokens[r] = argmax_v softmax(logits[r,:])(v) / (-ln u[r,v])
 * which draws v with probability softmax(logits[r,:])(v).
 *   logits [R, V] float32, u [R, V] float32 in (0,1), tokens [R] int32,
 *   status [R] int32 (UNO_SEQ_NONFINITE rows get token -1).
 * Requirements: R >= 0, 1 <= V < 2^31.  No workspace.
 * ------------------------------------------------------------------------- */
int uno_draft_sample(const float *logits, const float *u, int64_t R, int64_t V,
                     int32_t *tokens, int32_t *status, uno_stream_t stream);

/* Device error word of this library on the current device (synchronous).
 * Bit 0 is set when a pipeline wait inside a projection kernel exceeded its
 * 2-second limit; that kernel unwound without writing its output tile.
 * reset != 0 clears the word.  Returns the word (>= 0) or UNO_ERR_CUDA. */
int uno_device_error(int reset);

/* Human-readable text for a uno_status code (static storage). */
const char *uno_status_string(int code);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int uno_version(void);

#ifdef __cplusplus
}
#endif

#endif /* UNO_H_ */
