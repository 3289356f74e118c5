/*
 * spec_verify.h - C ABI of the batched speculative-decoding verifier for GB300 (sm_103a).
 *
 * One call verifies one round for a batch of B requests. Request i proposed K_i draft tokens
 * (K_i may differ per request, and may be 0). The caller has run the target model over the
 * round and passes K_i+1 target logit rows for request i (positions 1..K_i+1) and the K_i
 * draft logit rows its drafter sampled the tokens from. The verifier applies the rule of
 * "SOTA-227: Decode with a draft model and an accept-reject rule" (section "What to do",
 * steps 3-4), which is Rule 2 of "Speculative Decoding Coordination Protocol (SDCP)"
 * (section "Acceptance Rules"):
 *   - p_j = softmax(z^target_j / T), q_j = softmax(z^draft_j / T) (SDCP "Session Model":
 *     temperature is applied first);
 *   - walking j = 1..K_i left to right, draft x_j is accepted when u_j <= p_j(x_j)/q_j(x_j);
 *   - at the first rejection the frontier token is drawn from max(p_j - q_j, 0) normalised,
 *     and the walk stops; if all K_i are accepted it is drawn from p_{K_i+1};
 *   - with T == 0 the greedy rule applies (SDCP Rule 1): x_j is accepted when it is the
 *     argmax of p_j (ties to the smallest id) and the frontier token is argmax p_{A+1}.
 * Every draw is an inverse-CDF lookup in ascending token order: the token chosen is the
 * smallest v whose inclusive prefix mass exceeds u * (total mass).
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated otherwise. The caller owns all memory;
 *     no entry point allocates, frees or synchronises. Work is enqueued on `stream` in order.
 *   - Host-detectable argument errors return SPEC_ERR_INVALID_ARG (or SPEC_ERR_UNSUPPORTED)
 *     before anything is enqueued. A failed launch returns SPEC_ERR_CUDA.
 *   - Errors in the data of one request (found on the device) are reported per request in
 *     req_status and never disturb the other requests of the batch (SDCP "Error Handling":
 *     sdcp-bad-proposal is per proposal).
 *   - Logit rows must start on 16-byte boundaries: both logits pointers 16-byte aligned and
 *     V * sizeof(logit) a multiple of 16 (true for V = 32000, 128256, 151936, 256000 ...).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = -1, /* a host-checkable argument is wrong; nothing was enqueued   */
    SPEC_ERR_WORKSPACE = -2,   /* workspace missing, too small or misaligned                  */
    SPEC_ERR_CUDA = -3,        /* a CUDA call or launch failed                                */
    SPEC_ERR_UNSUPPORTED = -4  /* valid request this build cannot serve (e.g. unaligned rows) */
} spec_status;

/* req_status bits. A request with any bit set emits nothing: accept_len = n_emitted = 0 and
 * all its out_tokens slots are -1. */
enum {
    SPEC_REQ_OK = 0,
    SPEC_REQ_BAD_PROPOSAL = 1, /* a draft token outside [0, V), or q(x) == 0 (draft logit -inf),
                                  found before any uniform is used (SDCP Rule 2)             */
    SPEC_REQ_BAD_LOGITS = 2,   /* a row of the request holds NaN or +inf, or no finite logit  */
    SPEC_REQ_BAD_SHAPE = 4,    /* K_i < 0, K_i > K_max, or row_off inconsistent               */
    SPEC_REQ_BAD_PARAM = 8,    /* temperature NaN, infinite or negative, or top_p NaN         */
    SPEC_REQ_BAD_BLOCKS = 16,  /* spec_compact: a committed position has no page             */
    SPEC_REQ_TIMEOUT = 32      /* a bounded wait inside the verifier gave up before the request's
                                  data was ready; the request emits nothing (an internal fault,
                                  never produced on a healthy device)                          */
};

/* ---- spec_verify ------------------------------------------------------------------------
 * Layout: target logits are T = sum_i (K_i+1) rows of V values; request i owns rows
 * row_off[i] .. row_off[i+1]-1, row row_off[i]+j holding position j+1. Draft logits are
 * T - B rows; request i owns rows row_off[i]-i .. row_off[i+1]-i-2. draft_tokens and the
 * per-draft outputs use the draft-row index; uniforms and out_tokens use the target-row index.
 */
typedef struct {
    int32_t B;                   /* requests, >= 1                                             */
    int32_t V;                   /* vocabulary size, >= 1                                      */
    int32_t K_max;               /* upper bound on every K_i, 0..64 (SDCP: m_max <= 64)         */
    int32_t total_rows;          /* T = row_off[B] = sum_i (K_i + 1), as known to the host      */
    spec_dtype dtype;            /* type of both logits tensors                                */
    const void *target_logits;   /* [T][V]                                                    */
    const void *draft_logits;    /* [T-B][V] (may be NULL when T == B)                          */
    const int32_t *row_off;      /* [B+1], row_off[0] = 0, K_i = row_off[i+1]-row_off[i]-1     */
    const int32_t *draft_tokens; /* [T-B] x_j, sampled by the drafter from q_j                  */
    const double *uniforms;      /* [T] in [0,1): slot row_off[i]+j, j < K_i, is the accept draw
                                    of draft j; slot row_off[i]+K_i is the frontier draw       */
    const float *temperature;    /* [B] per request, or NULL to use temperature_scalar         */
    float temperature_scalar;
    const int32_t *stop_token;   /* [B] or NULL: emission stops after this token (-1: none)     */
    const int32_t *max_new;      /* [B] or NULL: most tokens request i may still emit           */
    /* outputs */
    int32_t *accept_len;         /* [B] A_i, drafts accepted by the rule                        */
    int32_t *n_emitted;          /* [B] tokens emitted: A_i + 1 unless a stop token or max_new
                                    truncated the round (SDCP "Verification and Commit" step 7)
                                    (may be NULL)                                              */
    int32_t *out_tokens;         /* [T] slot row_off[i]+j: emitted token j, -1 past n_emitted   */
    int32_t *req_status;         /* [B] SPEC_REQ_* bits                                        */
    float *alpha_rows;           /* [T-B] sum_v min(p_j(v), q_j(v)) per draft row; NaN on every draft
                                    row of a request with status bits (may be NULL)             */
    double *alpha_sum;           /* device scalar: sum of alpha over draft rows of OK requests
                                    (may be NULL)                                              */
    int32_t *alpha_count;        /* device scalar: number of those rows (may be NULL)           */
    /* diagnostics (each may be NULL) */
    float *rho_rows;             /* [T-B] p_j(x_j)/q_j(x_j) (greedy: 1 accepted / 0 rejected)   */
    float *resid_rows;           /* [T-B] sum_v max(p_j - q_j, 0) where the kernel formed the
                                    residual (a request's first rejected position, the only
                                    one drawn from), else -1                                   */
    float *frontier_prob;        /* [B] probability of the frontier token in the law it was
                                    drawn from                                                 */
    float *frontier_margin;      /* [B] distance of u*Z to the nearer end of the frontier
                                    token's CDF interval, over Z                                */
    int32_t *fallback;           /* [B] 1 when the residual had zero mass and p was used        */
    /* profiling (each may be NULL): cudaEvent_t recorded on `stream` immediately before the
       verifier's first kernel (after the truncation kernel, when there is one) and after its
       last, so that a caller can time the verifier's kernels alone; stats_event_end is recorded
       right after the first (per-chunk statistics) kernel, so that with rows_event_begin it
       brackets that kernel alone. Recording it holds the next kernel back until the statistics
       kernel has finished (no early launch), which costs the call a few microseconds. */
    cudaEvent_t rows_event_begin;
    cudaEvent_t rows_event_end;
    cudaEvent_t stats_event_end;
    /* depth statistics ("M7.8 - Speculative Serving", sections 0x02D and 0x07B; each may be
       NULL): over the requests without status bits, depth j = 1..K_max (index j-1) was reached
       when K_i >= j and the first j-1 drafts were accepted, and accepted when A_i >= j. Written
       (not accumulated) by each call; the ratio is the censoring-aware acceptance rate. */
    int32_t *depth_reached;      /* [K_max]                                                    */
    int32_t *depth_accepted;     /* [K_max]                                                    */
    /* top-k / top-p (SDCP "Session Model": p is the target's distribution after temperature,
       top-k and top-p, in that order; q is not truncated). Tokens rank by logit, ties by
       ascending id. Each may be NULL (no truncation); ignored under the greedy rule (T == 0).
       The cut of each target row is computed by an extra kernel before the verifier's, and
       every other token is treated as probability zero: the accept ratio, alpha, the residual
       and both draws use the truncated, renormalised law. */
    const int32_t *top_k;        /* [B] keep the k highest-ranked tokens (k <= 0 or k >= V: all) */
    const float *top_p;          /* [B] then keep the shortest head whose mass, renormalised over
                                    the top-k set, reaches top_p (>= 1: all; <= 0: the first
                                    token; NaN: SPEC_REQ_BAD_PARAM)                            */
} spec_verify_args;

/* Bytes of device workspace spec_verify needs for a batch of total_rows target rows of V logits
 * of type dtype. The workspace must be 256-byte aligned; its contents need no preparation (the
 * first kernel of each call zeroes the counters the later ones use), so one workspace may serve
 * calls of any shape that fits its size. Calls that share a workspace must not overlap on the
 * GPU. */
size_t spec_verify_workspace_size(int32_t B, int32_t V, int32_t total_rows, spec_dtype dtype);

/* Verify one round. Enqueues four kernels on `stream` (five with top-k / top-p, whose cut of each
 * target row runs first) and returns without waiting: spec_stats_kernel reads every logit once
 * (a persistent grid), spec_decide_kernel decides every position and marks each request's
 * frontier, spec_pass2_kernel reads the pairs' rows again (mostly from L2) for alpha and the
 * frontier's residual, and spec_finish_kernel draws the frontier tokens and selects each
 * request's result; each kernel after the first is launched so that its CTAs may start as the one
 * before drains. */
spec_status spec_verify(const spec_verify_args *args, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/* spec_verify without a caller-supplied workspace, for callers that cannot allocate device
 * memory where they verify (a memory planner that owns all device memory, a callback inside
 * another runtime, a path where cudaMalloc's synchronisation is not acceptable). The pages have
 * no counterpart to this entry point: it is an interface convenience of this library.
 * Scratch comes from one fixed array of 16 MiB in the library's device memory, present on every
 * GPU that loads the library until exit (a workspace needs no preparation between calls).
 * Limits: total_rows <= 16384 target rows per call, and spec_verify_workspace_size() of the
 * call's shape at most 16 MiB (for example T = 16384 rows with V * sizeof(logit) <= 64 KB, or the
 * B = 512, V = 256000 bf16 batch); larger calls return SPEC_ERR_UNSUPPORTED before anything is
 * enqueued. The array's address is looked up on the first call on each device (make that call
 * before any stream capture). All calls share the array: calls that overlap on the GPU (other
 * streams, other threads) race on it and must be serialised by the caller. Arguments, outputs
 * and errors are otherwise those of spec_verify. */
spec_status spec_verify_noalloc(const spec_verify_args *args, cudaStream_t stream);

/* Which kernel reads the logits for a batch of this shape (B requests, total_rows target rows,
 * vocabulary V, dtype) on the current device, and its grid: *cluster CTAs per cluster (1) and
 * *clusters CTAs (the same number on every SM); either pointer may be NULL. Returns a static
 * string naming the kernel ("spec_stats_kernel"), or NULL when the shape is invalid (B <= 0, V <= 0,
 * total_rows < B, a row not a multiple of 16 bytes) or the device cannot host the kernel. A
 * diagnostic: it enqueues nothing and only queries the device. */
const char *spec_verify_plan(int32_t B, int32_t V, int32_t total_rows, spec_dtype dtype, int32_t *cluster,
                             int32_t *clusters);

/* ---- spec_compact ------------------------------------------------------------------------
 * Packs the ragged result of spec_verify ("M7.8 - Speculative Serving", section 0x03C): for
 * request i with prefix length P_i (target KV rows already committed), E_i accepted drafts
 * emitted and F_i = 1 when the frontier token was emitted:
 *   tokens  : packed at out_off[i] .. out_off[i+1]-1, positions P_i .. P_i+n_i-1;
 *   KV rows : the first E_i candidate rows of the round are committed: kv_src = the caller's
 *             cand_kv_rows[row_off[i]-i+j], kv_dst = block_table[i][(P_i+j)/page]*page +
 *             (P_i+j) % page, for j < E_i; the frontier has no KV row yet (section 0x08A);
 *   lengths : L_out = P_i+E_i+F_i, L_target = P_i+E_i, L_draft = P_i+min(E_i, K_i-1)
 *             (section 0x09, "EOS and length-limit stopping").
 * A request with a nonzero req_status, or whose committed positions fall outside its block
 * table (SPEC_REQ_BAD_BLOCKS), emits and commits nothing and keeps its lengths at P_i.
 */
typedef struct {
    int32_t B, page_size, max_blocks, total_rows;
    const int32_t *row_off;      /* [B+1] as for spec_verify                                    */
    const int32_t *accept_len;   /* [B] from spec_verify                                        */
    const int32_t *n_emitted;    /* [B] from spec_verify (NULL: accept_len + 1)                 */
    const int32_t *out_tokens;   /* [T] from spec_verify                                        */
    const int32_t *req_status;   /* [B] from spec_verify (NULL: all OK)                         */
    const int32_t *prefix_len;   /* [B] P_i                                                    */
    const int32_t *cand_kv_rows; /* [T-B] physical row holding draft j's candidate target KV    */
    const int32_t *block_table;  /* [B][max_blocks] page ids                                   */
    /* outputs; capacities: T tokens, T-B KV pairs */
    int32_t *out_off;            /* [B+1] exclusive prefix of n_i                               */
    int32_t *packed_tokens;      /* [T]                                                        */
    int32_t *packed_pos;         /* [T]                                                        */
    int32_t *kv_off;             /* [B+1] exclusive prefix of E_i                               */
    int32_t *kv_src;             /* [T-B]                                                      */
    int32_t *kv_dst;             /* [T-B]                                                      */
    int32_t *new_seq_len;        /* [B] L_out                                                  */
    int32_t *new_kv_len;         /* [B] L_target                                               */
    int32_t *new_draft_len;      /* [B] L_draft (may be NULL)                                   */
    int32_t *compact_status;     /* [B] req_status | SPEC_REQ_BAD_BLOCKS (may be NULL)           */
} spec_compact_args;

/* Enqueues one kernel on `stream`. Needs no workspace. The output arrays must not overlap the
 * input arrays (the kernel reads each request's inputs before it writes its packed outputs, in
 * any order across requests). */
spec_status spec_compact(const spec_compact_args *args, cudaStream_t stream);

/* ---- choosing gamma ---------------------------------------------------------------------
 * SOTA-227, "Why it is free rather than a trade": with acceptance rate alpha = E[min(p,q)]
 * and draft cost c relative to the target, drafting gamma tokens improves wall time by
 *     f(gamma) = (1 - alpha^(gamma+1)) / ((1 - alpha)(gamma*c + 1)),
 * f = (gamma+1)/(gamma*c+1) at alpha = 1, and gamma is chosen numerically.
 *
 * spec_gamma_objective evaluates f on the host (double precision).
 * spec_choose_gamma runs on the device: alpha = alpha_sum / alpha_count read from device
 * memory (as written by spec_verify), or alpha_prev when alpha_count == 0; it writes the
 * maximiser of f over [gamma_min, gamma_max] to *gamma_out (an exact tie goes to the smaller
 * gamma, as the controller of "M7.8 - Speculative Serving" section 0x07A breaks ties toward
 * smaller K) and the alpha it used to *alpha_out. All four pointers are device pointers. */
double spec_gamma_objective(double alpha, double c, int32_t gamma);

/* spec_choose_gamma with the per-depth rates in place of one alpha ("M7.8 - Speculative
 * Serving", section 0x07B): alpha_hat_j = n_accepted[j-1] / n_reached[j-1] (device arrays of
 * depth_max counts, as written by spec_verify); a depth nobody reached takes the pooled rate
 * sum(n_accepted) / sum(n_reached), and with nothing reached alpha_prev. E[A](gamma) =
 * sum_{j<=gamma} prod_{m<=j} alpha_hat_m; gamma maximises (1 + E[A]) / (gamma*c + 1) over
 * [gamma_min, gamma_max] (ties to the smaller). Writes *gamma_out and *ea_out = E[A] at that gamma
 * (device scalars). Runs on the device, one thread; SPEC_ERR_INVALID_ARG for a null output, a
 * negative depth_max (or null counts with depth_max > 0), gamma_min < 0, gamma_max < gamma_min or
 * > 4096, c < 0 or not finite, alpha_prev outside [0, 1]. */
spec_status spec_choose_gamma_depth(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                                    double alpha_prev, double c, int32_t gamma_min, int32_t gamma_max,
                                    int32_t *gamma_out, double *ea_out, cudaStream_t stream);

/* Host, double precision: the objective (1 + E[A](gamma)) / (gamma*c + 1) of
 * spec_choose_gamma_depth from HOST arrays of counts. */
double spec_depth_objective(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                            double alpha_prev, double c, int32_t gamma);
spec_status spec_choose_gamma(const double *alpha_sum, const int32_t *alpha_count,
                              double alpha_prev, double c, int32_t gamma_min, int32_t gamma_max,
                              int32_t *gamma_out, double *alpha_out, cudaStream_t stream);

/* ---- spec_verify_round ---------------------------------------------------------------------
 * One verification round, enqueued as one call: the same results, bit for bit, as
 *   spec_verify(args, workspace, workspace_bytes, stream);
 *   spec_compact(compact, stream);
 *   spec_choose_gamma(args->alpha_sum, args->alpha_count, alpha_prev, c, gamma_min, gamma_max,
 *                     gamma_out, alpha_out, stream);
 * with the compaction and the gamma choice run by the CTA of spec_verify's finishing kernel that
 * completes the batch, so that the round adds no launch. `compact` carries the compaction's own inputs and outputs as for
 * spec_compact; its accept_len / n_emitted / out_tokens / req_status are normally args'
 * outputs. Every argument is checked as by the three calls (plus compact->B == args->B and
 * compact->total_rows == args->total_rows; args->alpha_sum and args->alpha_count are required)
 * before anything is enqueued; errors are theirs. A convenience of this library: the pages
 * define the three steps, not their grouping. */
spec_status spec_verify_round(const spec_verify_args *args, void *workspace, size_t workspace_bytes,
                              const spec_compact_args *compact, double alpha_prev, double c, int32_t gamma_min,
                              int32_t gamma_max, int32_t *gamma_out, double *alpha_out, cudaStream_t stream);

/* Version string of the library build. */
const char *spec_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
