/*
 * Oracle for the batched speculative-decoding verifier: plain, slow, float64, host only.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load this code. It shares no source, header or helper with the CUDA library: the
 * structs below are this file's own, and nothing here includes the library's header.
 *
 * What it computes follows the pages:
 *   - "SOTA-227: Decode with a draft model and an accept-reject rule", section "What to do",
 *     steps 3 and 4: walk the draft left to right, accept x_i when r_i <= p_i(x)/q_i(x),
 *     at the first rejection resample from the normalised positive part of p - q and stop;
 *     if nothing was rejected, draw the extra token from p at position gamma + 1.
 *   - "Speculative Decoding Coordination Protocol (SDCP)", section "Acceptance Rules",
 *     Rule 2 (speculative sampling): the same rule, q(x) must be checked non-zero before any
 *     random draw; the accept draw and the extra-token draw are separate values.
 *   - SDCP, section "Session Model": p is the target's distribution after temperature, top-k
 *     and top-p, in that order (the draft's q is not truncated). Reading of the silent points:
 *     tokens are ranked by logit, ties by ascending token id; top-k keeps the first k; top-p
 *     then keeps the shortest head whose mass, renormalised over the top-k set, is >= top_p.
 *   - "M7.8 - Speculative Serving", section 0x03C (ragged acceptance) and 0x09 (draft,
 *     target and frontier cache transitions): L_out = P + A + 1, L_kv = P + A.
 *   - SOTA-227, section "Why it is free rather than a trade": alpha = E[min(p, q)] and the
 *     expected wall-time improvement (1 - alpha^(gamma+1)) / ((1 - alpha)(gamma*c + 1)).
 *
 * Parity status: every function here is pinned by CPU tests against values the pages print
 * (ledgers), closed forms, brute-force enumeration of the exact law on tiny vocabularies and a
 * chi-square test of the exactness theorem.
 */
#ifndef SPEC_ORACLE_H
#define SPEC_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* request status bits (a request with any bit set emits nothing) */
#define ORACLE_REQ_BAD_PROPOSAL 1 /* draft token outside [0,V) or q(x) == 0 (draft logit -inf) */
#define ORACLE_REQ_BAD_LOGITS   2 /* a row holds NaN or +inf, or has no finite logit          */
#define ORACLE_REQ_BAD_SHAPE    4 /* K_i < 0 or K_i > K_max                                  */
#define ORACLE_REQ_BAD_PARAM    8 /* temperature not finite or < 0, or top_p NaN            */
#define ORACLE_REQ_BAD_BLOCKS  16 /* compaction: a committed position has no page            */

typedef struct {
    int32_t B, V, K_max;
    int32_t dtype;              /* 0: float32 logits, 1: bfloat16 logits given as raw uint16 */
    const void *target;         /* [T][V], T = row_off[B]; request i owns rows row_off[i]..  */
    const void *draft;          /* [T-B][V]; request i owns rows row_off[i]-i ..             */
    const int32_t *row_off;     /* [B+1], K_i = row_off[i+1]-row_off[i]-1                    */
    const int32_t *draft_tokens;/* [T-B]                                                     */
    const double *uniforms;     /* [T]: slot j<K_i accept draw of draft j, slot K_i the draw
                                   of the extra token                                        */
    const float *temperature;   /* [B]; 0 selects the greedy rule                             */
    const int32_t *stop_token;  /* [B] or NULL: token that ends generation (-1: none)         */
    const int32_t *max_new;     /* [B] or NULL: output tokens still allowed (budget)          */
    const int32_t *top_k;       /* [B] or NULL: keep the k most probable tokens of p (k <= 0 or
                                   k >= V: all)                                                */
    const float *top_p;         /* [B] or NULL: then keep the shortest head of p, renormalised
                                   over the top-k set, whose mass reaches top_p (>= 1: all)    */
} oracle_batch;

typedef struct {
    int32_t *accept_len;        /* [B] A_i: accepted drafts actually emitted                  */
    int32_t *out_tokens;        /* [T] slot j of request i; -1 where nothing was emitted       */
    int32_t *n_emitted;         /* [B] tokens emitted this round (A_i + frontier flag)        */
    int32_t *req_status;        /* [B] status bits                                            */
    double *alpha;              /* [T-B] sum_v min(p_j(v), q_j(v)), every draft position      */
    double *rho;                /* [T-B] p_j(x_j) / q_j(x_j)                                  */
    double *resid_mass;         /* [T-B] sum_v max(p_j(v) - q_j(v), 0)                        */
    double *accept_margin;      /* [T-B] u_j - rho_j                                          */
    double *sample_margin;      /* [B] distance of u*Z to the nearer end of the chosen token's
                                   CDF interval, divided by Z (NaN when no draw was made)     */
    double *sample_prob;        /* [B] probability of the frontier token under the law it was
                                   drawn from                                                  */
    int32_t *fallback;          /* [B] 1 when the residual had zero mass and p was used        */
    double *trunc_margin;       /* [T] or NULL: distance of top_p to the nearer of the
                                   cumulative masses of the kept head and of the head one token
                                   shorter (when that has a token; NaN: no top-p cut)           */
    int32_t *trunc_keep;        /* [T] or NULL: tokens kept by top-k / top-p (V: all)          */
    /* Conditioning of the residual quantities (diagnostics for comparing a float32 kernel; they
     * take no part in any decision). A float32 p or q carries a relative error e, so
     * p(v) - q(v) carries up to e (p(v) + q(v)): */
    double *resid_scale;        /* [T-B] or NULL: sum over {v : p_j(v) > q_j(v)} of
                                   p_j(v) + q_j(v); resid_scale / resid_mass is the relative
                                   error bound of the residual mass per unit of e             */
    double *sample_cond;        /* [B] or NULL: the same bound for sample_prob. A residual draw
                                   of token x: (p(x) + q(x)) / (p(x) - q(x)) + resid_scale /
                                   resid_mass of its row; a draw from p, or a greedy pick: 1;
                                   NaN when no token was drawn                                 */
} oracle_result;

int oracle_verify(const oracle_batch *in, oracle_result *out);

/* The same result computed with up to n_threads threads (OpenMP, requests split across them;
 * each request is still computed by oracle_verify's own code, serially). Returns the number of
 * threads used (1 when the library was built without OpenMP), or a negative error code. For
 * timing the oracle on all of a host's cores. */
int oracle_verify_threads(const oracle_batch *in, oracle_result *out, int32_t n_threads);

typedef struct {
    int32_t B, page_size, max_blocks;
    const int32_t *row_off;      /* [B+1] as for oracle_verify                                 */
    const int32_t *accept_len;   /* [B]                                                        */
    const int32_t *n_emitted;    /* [B]                                                        */
    const int32_t *out_tokens;   /* [T]                                                        */
    const int32_t *req_status;   /* [B]                                                        */
    const int32_t *prefix_len;   /* [B] P_i, committed target KV length before the round       */
    const int32_t *cand_kv_rows; /* [T-B] physical row holding draft j's candidate target KV   */
    const int32_t *block_table;  /* [B][max_blocks] page ids                                  */
    int32_t *out_off;            /* [B+1]                                                      */
    int32_t *packed_tokens;      /* [sum emitted]                                              */
    int32_t *packed_pos;         /* [sum emitted]                                              */
    int32_t *kv_off;             /* [B+1]                                                      */
    int32_t *kv_src;             /* [sum A]                                                    */
    int32_t *kv_dst;             /* [sum A]                                                    */
    int32_t *new_seq_len;        /* [B] L_out                                                  */
    int32_t *new_kv_len;         /* [B] L_target                                               */
    int32_t *new_draft_len;      /* [B] L_draft                                                */
    int32_t *compact_status;     /* [B] req_status | ORACLE_REQ_BAD_BLOCKS                     */
} oracle_compact_args;

int oracle_compact(const oracle_compact_args *a);

double oracle_gamma_objective(double alpha, double c, int32_t gamma);

/* Depth statistics ("M7.8 - Speculative Serving", sections 0x02D and 0x07B): depth j = 1..depth_max
 * of request i (no status bits) was reached when K_i >= j and its first j-1 drafts were accepted
 * (A_i >= j-1), and accepted when A_i >= j. n_reached[j-1], n_accepted[j-1] count requests. */
void oracle_depth_counts(int32_t B, const int32_t *row_off, const int32_t *accept_len,
                         const int32_t *req_status, int32_t depth_max, int32_t *n_reached,
                         int32_t *n_accepted);
/* alpha_hat_j = n_accepted_j / n_reached_j (censoring-aware); a depth nobody reached takes the
 * pooled estimate over all depths, and with no depth reached at all alpha_prev. j = 1..n_out. */
void oracle_depth_alpha(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                        double alpha_prev, int32_t n_out, double *alpha_hat);
/* Expected accepted drafts with gamma drafts, E[A] = sum_{j<=gamma} prod_{m<=j} alpha_hat_m, and
 * the depth-aware objective (1 + E[A]) / (gamma*c + 1), which for a constant alpha_hat is
 * oracle_gamma_objective. */
double oracle_depth_expected_accept(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                                    double alpha_prev, int32_t gamma);
double oracle_depth_objective(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                              double alpha_prev, double c, int32_t gamma);
int32_t oracle_choose_gamma_depth(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                                  double alpha_prev, double c, int32_t gamma_min, int32_t gamma_max,
                                  double *ea_out);
int32_t oracle_choose_gamma(double alpha_sum, int32_t alpha_count, double alpha_prev, double c,
                            int32_t gamma_min, int32_t gamma_max, double *alpha_out);

#ifdef __cplusplus
}
#endif
#endif
