/*
 * Oracle for the batched speculative-decoding verifier (float64, host only).
 *
 * TEST INFRASTRUCTURE: see spec_oracle.h for the pages this follows and for who may call it.
 * The code is deliberately plain: every row is reduced in ascending token order in double
 * precision, with separate loops for each quantity, so that it can be checked against the
 * pages by eye. Nothing here is blocked, fused or reordered for speed.
 */
#include "spec_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- reading logits --------------------------------------------------------------- */

/* bfloat16 is the upper half of a binary32; widening it is exact. */
static double widen_bf16(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double logit_at(const void *base, int32_t dtype, int64_t row, int32_t V, int32_t v) {
    int64_t k = row * (int64_t)V + v;
    if (dtype == 1) return widen_bf16(((const uint16_t *)base)[k]);
    return (double)((const float *)base)[k];
}

/* ---- one row's distribution --------------------------------------------------------- */

/* The row's law p(v) = exp(z_v/T) / sum_w exp(z_w/T) (SDCP "Session Model": temperature
 * first), held as its log-normaliser: log p(v) = z_v/T - m - log S with m = max_w z_w/T and
 * S = sum_w exp(z_w/T - m). Greedy rows (T == 0) are the point mass at the smallest index
 * among the maxima. */
typedef struct {
    const void *base;
    int32_t dtype, V;
    int64_t row;
    double T;
    int greedy;
    int32_t argmax; /* smallest index attaining the maximum logit */
    double m, logS; /* only for T > 0; S over the kept tokens */
    int valid;      /* 0 when a logit is NaN or +inf or none is finite */
    /* top-k / top-p: token v is kept when (z_v, v) ranks no later than (z_cut, id_cut) in the
     * order "larger logit first, then smaller id"; without truncation every token is kept */
    int truncated;
    double z_cut;
    int32_t id_cut, keep;
    double cut_margin; /* top-p only: |top_p - nearer cumulative mass at the cut| */
} row_law;

static int row_kept(const row_law *L, double z, int32_t v) {
    if (!L->truncated) return 1;
    return z > L->z_cut || (z == L->z_cut && v <= L->id_cut);
}

/* Ranking of one row for the truncation: larger logit first, then smaller id. */
typedef struct {
    double z;
    int32_t v;
} ranked;

static int ranked_cmp(const void *a, const void *b) {
    const ranked *x = (const ranked *)a, *y = (const ranked *)b;
    if (x->z > y->z) return -1;
    if (x->z < y->z) return 1;
    return (x->v > y->v) - (x->v < y->v);
}

/* Top-k, then top-p (SDCP "Session Model", in that order) on the row's law at temperature T:
 * rank the tokens; keep the first n_k = k of them (all when k <= 0 or k >= V); renormalise p
 * over them; keep the first n_p whose cumulative mass reaches top_p (n_p >= 1; all when
 * top_p >= 1). Records the last kept token as the cut. */
static void row_truncate(row_law *L, int32_t top_k, double top_p) {
    const int32_t V = L->V;
    L->truncated = 0;
    L->keep = V;
    L->cut_margin = NAN;
    const int use_k = top_k > 0 && top_k < V, use_p = top_p < 1.0;
    if (!use_k && !use_p) return;
    ranked *r = (ranked *)malloc(sizeof(ranked) * (size_t)V);
    if (!r) return;
    for (int32_t v = 0; v < V; ++v) {
        r[v].z = logit_at(L->base, L->dtype, L->row, V, v);
        r[v].v = v;
    }
    qsort(r, (size_t)V, sizeof(ranked), ranked_cmp);
    int32_t n = use_k ? top_k : V;
    if (use_p) {
        /* masses of the top-k head, renormalised over it */
        double Sk = 0.0;
        for (int32_t j = 0; j < n; ++j) Sk += exp(r[j].z / L->T - L->m);
        double cum = 0.0, prev = 0.0;
        int32_t np = n;
        for (int32_t j = 0; j < n; ++j) {
            prev = cum;
            cum += exp(r[j].z / L->T - L->m) / Sk;
            if (cum >= top_p) {
                np = j + 1;
                break;
            }
        }
        /* the cut can move only between heads of one or more tokens: the empty head (mass 0)
         * never counts, so with n_p = 1 only the first token's mass is compared */
        const double d1 = fabs(cum - top_p), d0 = fabs(prev - top_p);
        L->cut_margin = (np >= 2 && d0 < d1) ? d0 : d1;
        n = np;
    }
    L->truncated = 1;
    L->keep = n;
    L->z_cut = r[n - 1].z;
    L->id_cut = r[n - 1].v;
    free(r);
}

static row_law row_law_make(const void *base, int32_t dtype, int64_t row, int32_t V, double T) {
    row_law L;
    L.base = base;
    L.dtype = dtype;
    L.V = V;
    L.row = row;
    L.T = T;
    L.greedy = (T == 0.0);
    L.argmax = -1;
    L.m = -INFINITY;
    L.logS = 0.0;
    L.valid = 1;
    L.truncated = 0;
    L.keep = V;
    L.cut_margin = NAN;

    double zmax = -INFINITY;
    for (int32_t v = 0; v < V; ++v) {
        double z = logit_at(base, dtype, row, V, v);
        if (isnan(z) || z == INFINITY) L.valid = 0;
        if (z > zmax) {
            zmax = z;
            L.argmax = v;
        }
    }
    if (zmax == -INFINITY) L.valid = 0;
    if (!L.valid || L.greedy) return L;

    double m = -INFINITY;
    for (int32_t v = 0; v < V; ++v) {
        double y = logit_at(base, dtype, row, V, v) / T;
        if (y > m) m = y;
    }
    double S = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        double y = logit_at(base, dtype, row, V, v) / T;
        S += exp(y - m);
    }
    L.m = m;
    L.logS = log(S);
    return L;
}

/* Renormalise a truncated law over its kept tokens. */
static void row_law_renormalise(row_law *L) {
    if (!L->truncated || L->greedy || !L->valid) return;
    double S = 0.0;
    for (int32_t v = 0; v < L->V; ++v) {
        double z = logit_at(L->base, L->dtype, L->row, L->V, v);
        if (row_kept(L, z, v)) S += exp(z / L->T - L->m);
    }
    L->logS = log(S);
}

static double row_prob(const row_law *L, int32_t v) {
    if (L->greedy) return v == L->argmax ? 1.0 : 0.0;
    double z = logit_at(L->base, L->dtype, L->row, L->V, v);
    if (!row_kept(L, z, v)) return 0.0;
    double y = z / L->T;
    return exp(y - L->m - L->logS);
}

/* ---- inverse-CDF draw --------------------------------------------------------------- */

/* Draw from the (unnormalised) weights w[0..V-1] with the uniform u: the smallest v whose
 * inclusive prefix sum C_v exceeds u*Z, Z = sum w, scanning ascending token ids. A token of
 * zero weight is never chosen. Returns -1 when Z == 0. */
static int32_t inverse_cdf(const double *w, int32_t V, double u, double *margin, double *prob) {
    double Z = 0.0;
    for (int32_t v = 0; v < V; ++v) Z += w[v];
    if (!(Z > 0.0)) return -1;
    double t = u * Z;
    double C = 0.0;
    int32_t last = -1;
    for (int32_t v = 0; v < V; ++v) {
        double C_prev = C;
        C += w[v];
        if (w[v] > 0.0) last = v;
        if (C > t && w[v] > 0.0) {
            double lo = t - C_prev, hi = C - t;
            *margin = (lo < hi ? lo : hi) / Z;
            *prob = w[v] / Z;
            return v;
        }
    }
    /* u*Z rounded up to Z: the last token of positive weight */
    *margin = 0.0;
    *prob = w[last] / Z;
    return last;
}

/* ---- the verifier ---------------------------------------------------------------------- */

/* Requests i0 .. i1-1 of the batch (each request is independent of the others). */
static int verify_requests(const oracle_batch *in, oracle_result *out, int32_t i0, int32_t i1) {
    const int32_t V = in->V;
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    row_law *Plaw = (row_law *)malloc(sizeof(row_law) * (size_t)(in->K_max + 1));
    row_law *Qlaw = (row_law *)malloc(sizeof(row_law) * (size_t)(in->K_max + 1));
    if (!w || !Plaw || !Qlaw) {
        free(w);
        free(Plaw);
        free(Qlaw);
        return -2;
    }

    for (int32_t i = i0; i < i1; ++i) {
        const int32_t r0 = in->row_off[i];
        const int32_t K = in->row_off[i + 1] - r0 - 1;
        const int32_t d0 = r0 - i; /* first draft row of request i */
        const double T = (double)in->temperature[i];
        int32_t status = 0;

        const int32_t tk = in->top_k ? in->top_k[i] : 0;
        const double tp = in->top_p ? (double)in->top_p[i] : 1.0;
        if (K < 0 || K > in->K_max) status |= ORACLE_REQ_BAD_SHAPE;
        if (!(T >= 0.0) || isinf(T) || isnan(tp)) status |= ORACLE_REQ_BAD_PARAM;
        if (K >= 0 && out->trunc_margin)
            for (int32_t j = 0; j <= K; ++j) out->trunc_margin[r0 + j] = NAN;
        if (K >= 0 && out->trunc_keep)
            for (int32_t j = 0; j <= K; ++j) out->trunc_keep[r0 + j] = V;

        out->accept_len[i] = 0;
        out->n_emitted[i] = 0;
        out->sample_margin[i] = NAN;
        out->sample_prob[i] = NAN;
        out->fallback[i] = 0;
        if (out->sample_cond) out->sample_cond[i] = NAN;
        if (status) {
            for (int32_t j = 0; j < in->row_off[i + 1] - r0; ++j) out->out_tokens[r0 + j] = -1;
            for (int32_t j = 0; j < K; ++j) {
                out->alpha[d0 + j] = NAN;
                out->rho[d0 + j] = NAN;
                out->resid_mass[d0 + j] = NAN;
                out->accept_margin[d0 + j] = NAN;
                if (out->resid_scale) out->resid_scale[d0 + j] = NAN;
            }
            out->req_status[i] = status;
            continue;
        }

        /* Preconditions, checked before any uniform is read (SDCP "Verification and
         * Commit" step 5, and Rule 2: a proposal whose q(x) is zero is rejected before any
         * random draw). */
        for (int32_t j = 0; j <= K; ++j) {
            Plaw[j] = row_law_make(in->target, in->dtype, r0 + j, V, T);
            if (!Plaw[j].valid) status |= ORACLE_REQ_BAD_LOGITS;
            if (Plaw[j].valid && !Plaw[j].greedy) {
                row_truncate(&Plaw[j], tk, tp);
                row_law_renormalise(&Plaw[j]);
                if (out->trunc_margin) out->trunc_margin[r0 + j] = Plaw[j].cut_margin;
                if (out->trunc_keep) out->trunc_keep[r0 + j] = Plaw[j].keep;
            }
        }
        for (int32_t j = 0; j < K; ++j) {
            Qlaw[j] = row_law_make(in->draft, in->dtype, d0 + j, V, T);
            if (!Qlaw[j].valid) status |= ORACLE_REQ_BAD_LOGITS;
            int32_t x = in->draft_tokens[d0 + j];
            if (x < 0 || x >= V) {
                status |= ORACLE_REQ_BAD_PROPOSAL;
            } else if (T > 0.0 && logit_at(in->draft, in->dtype, d0 + j, V, x) == -INFINITY) {
                status |= ORACLE_REQ_BAD_PROPOSAL; /* q(x) == 0 */
            }
        }
        out->req_status[i] = status;
        if (status) {
            for (int32_t j = 0; j <= K; ++j) out->out_tokens[r0 + j] = -1;
            for (int32_t j = 0; j < K; ++j) {
                out->alpha[d0 + j] = NAN;
                out->rho[d0 + j] = NAN;
                out->resid_mass[d0 + j] = NAN;
                out->accept_margin[d0 + j] = NAN;
                if (out->resid_scale) out->resid_scale[d0 + j] = NAN;
            }
            continue;
        }

        /* Per-position quantities, for every draft position (alpha = E[min(p,q)], SOTA-227
         * "Why it is free rather than a trade"). */
        for (int32_t j = 0; j < K; ++j) {
            const row_law P = Plaw[j], Q = Qlaw[j];
            int32_t x = in->draft_tokens[d0 + j];
            double a = 0.0, z = 0.0, zs = 0.0;
            for (int32_t v = 0; v < V; ++v) {
                double p = row_prob(&P, v), q = row_prob(&Q, v);
                a += (p < q ? p : q);
                z += (p - q > 0.0 ? p - q : 0.0);
                if (p > q) zs += p + q;
            }
            out->alpha[d0 + j] = a;
            out->resid_mass[d0 + j] = z;
            if (out->resid_scale) out->resid_scale[d0 + j] = zs;
            if (P.greedy) {
                /* Rule 1 has no ratio; report the accept test as 1/0. */
                out->rho[d0 + j] = (x == P.argmax) ? 1.0 : 0.0;
                out->accept_margin[d0 + j] = NAN;
            } else {
                const double zx = logit_at(in->target, in->dtype, r0 + j, V, x);
                double lp = zx / T - P.m - P.logS;
                double lq = logit_at(in->draft, in->dtype, d0 + j, V, x) / T - Q.m - Q.logS;
                /* p(x) = 0 where top-k / top-p removed x */
                double rho = row_kept(&P, zx, x) ? exp(lp - lq) : 0.0;
                out->rho[d0 + j] = rho;
                out->accept_margin[d0 + j] = in->uniforms[r0 + j] - rho;
            }
        }

        /* Walk the draft left to right (SOTA-227 "What to do", step 3; SDCP Rules 1 and 2). */
        const double u_extra = in->uniforms[r0 + K]; /* the extra token's own draw */
        int32_t A = K;
        int32_t frontier = -1;
        for (int32_t j = 0; j < K; ++j) {
            int32_t x = in->draft_tokens[d0 + j];
            double rho = out->rho[d0 + j];
            int accept;
            if (T == 0.0) {
                accept = (rho == 1.0);
            } else {
                /* accept when u <= p/q; a token the target gives zero probability is never
                 * accepted (this decides the u == 0 edge of "<=") */
                double u = in->uniforms[r0 + j];
                accept = (rho > 0.0) && (u <= rho);
            }
            out->out_tokens[r0 + j] = x;
            if (accept) continue;

            A = j;
            const row_law P = Plaw[j];
            if (T == 0.0) {
                frontier = P.argmax; /* Rule 1: the correction is argmax p at the rejection */
                out->sample_prob[i] = 1.0;
                if (out->sample_cond) out->sample_cond[i] = 1.0;
                break;
            }
            /* Rule 2 / step 3: resample from max(0, p - q), normalised. */
            const row_law Q = Qlaw[j];
            for (int32_t v = 0; v < V; ++v) {
                double diff = row_prob(&P, v) - row_prob(&Q, v);
                w[v] = diff > 0.0 ? diff : 0.0;
            }
            frontier = inverse_cdf(w, V, u_extra, &out->sample_margin[i], &out->sample_prob[i]);
            if (frontier < 0) {
                /* The residual has zero mass in double precision. Mathematically a rejection
                 * then has probability zero; draw from p instead and say so. */
                out->fallback[i] = 1;
                for (int32_t v = 0; v < V; ++v) w[v] = row_prob(&P, v);
                frontier = inverse_cdf(w, V, u_extra, &out->sample_margin[i],
                                       &out->sample_prob[i]);
                if (out->sample_cond) out->sample_cond[i] = 1.0;
            } else if (out->sample_cond) {
                const double px = row_prob(&P, frontier), qx = row_prob(&Q, frontier);
                double zs = 0.0, z = 0.0;
                for (int32_t v = 0; v < V; ++v) {
                    double p = row_prob(&P, v), q = row_prob(&Q, v);
                    if (p > q) {
                        zs += p + q;
                        z += p - q;
                    }
                }
                out->sample_cond[i] = (px + qx) / (px - qx) + zs / z;
            }
            break;
        }
        if (A == K) {
            /* Step 4: nothing rejected, the extra token comes from p at position K+1. */
            const row_law P = Plaw[K];
            if (T == 0.0) {
                frontier = P.argmax;
                out->sample_prob[i] = 1.0;
            } else {
                for (int32_t v = 0; v < V; ++v) w[v] = row_prob(&P, v);
                frontier = inverse_cdf(w, V, u_extra, &out->sample_margin[i],
                                       &out->sample_prob[i]);
            }
            if (out->sample_cond) out->sample_cond[i] = 1.0;
        }
        out->out_tokens[r0 + A] = frontier;
        for (int32_t j = A + 1; j <= K; ++j) out->out_tokens[r0 + j] = -1;
        out->accept_len[i] = A;

        /* Stopping (SDCP "Verification and Commit" step 7; M7.8 section 0x09 "EOS and
         * length-limit stopping"): keep tokens up to and including the first stop token and
         * no more than the remaining budget. */
        int32_t n = A + 1;
        if (in->max_new && in->max_new[i] < n) n = in->max_new[i] < 0 ? 0 : in->max_new[i];
        if (in->stop_token && in->stop_token[i] >= 0) {
            for (int32_t j = 0; j < n; ++j) {
                if (out->out_tokens[r0 + j] == in->stop_token[i]) {
                    n = j + 1;
                    break;
                }
            }
        }
        for (int32_t j = n; j <= A; ++j) out->out_tokens[r0 + j] = -1;
        out->n_emitted[i] = n;
    }
    free(w);
    free(Plaw);
    free(Qlaw);
    return 0;
}

int oracle_verify(const oracle_batch *in, oracle_result *out) {
    if (in->B < 0 || in->V <= 0) return -1;
    return verify_requests(in, out, 0, in->B);
}

int oracle_verify_threads(const oracle_batch *in, oracle_result *out, int32_t n_threads) {
    if (in->B < 0 || in->V <= 0 || n_threads < 1) return -1;
#ifdef _OPENMP
    int err = 0, used = 1;
#pragma omp parallel num_threads(n_threads) reduction(| : err)
    {
#pragma omp single
        used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 1)
        for (int32_t i = 0; i < in->B; ++i) err |= (verify_requests(in, out, i, i + 1) != 0);
    }
    return err ? -2 : used;
#else
    return verify_requests(in, out, 0, in->B) == 0 ? 1 : -2;
#endif
}

/* ---- compaction ---------------------------------------------------------------------- */

/* M7.8 section 0x03C: request i advances its output to L_out = P + A + 1 but commits only the
 * A candidate target-KV rows of its accepted drafts (L_kv = P + A); the frontier token keeps
 * no KV row. Section 0x09 with stopping: E accepted drafts emitted, F in {0,1} frontier
 * emitted, L_out = P + E + F, L_target = P + E, L_draft = P + min(E, K - 1). Committed KV row
 * j lands at logical position P + j, in page block_table[i][(P+j)/page] at offset
 * (P+j) mod page. */
int oracle_compact(const oracle_compact_args *a) {
    int32_t out_pos = 0, kv_pos = 0;
    for (int32_t i = 0; i < a->B; ++i) {
        const int32_t r0 = a->row_off[i];
        const int32_t K = a->row_off[i + 1] - r0 - 1;
        const int32_t d0 = r0 - i;
        const int32_t P = a->prefix_len[i];
        int32_t status = a->req_status[i];
        int32_t n = 0, E = 0;
        if (!status) {
            n = a->n_emitted[i];
            int32_t A = a->accept_len[i];
            E = n < A ? n : A;
            /* every committed position needs a page */
            if (E > 0) {
                int32_t last_page = (P + E - 1) / a->page_size;
                if (P < 0 || last_page >= a->max_blocks) status |= ORACLE_REQ_BAD_BLOCKS;
                for (int32_t j = 0; j < E && !status; ++j) {
                    int32_t blk = a->block_table[(int64_t)i * a->max_blocks + (P + j) / a->page_size];
                    if (blk < 0) status |= ORACLE_REQ_BAD_BLOCKS;
                }
            }
            if (status) n = E = 0;
        }
        a->compact_status[i] = status;
        a->out_off[i] = out_pos;
        a->kv_off[i] = kv_pos;
        for (int32_t j = 0; j < n; ++j) {
            a->packed_tokens[out_pos + j] = a->out_tokens[r0 + j];
            a->packed_pos[out_pos + j] = P + j;
        }
        for (int32_t j = 0; j < E; ++j) {
            int32_t pos = P + j;
            int32_t blk = a->block_table[(int64_t)i * a->max_blocks + pos / a->page_size];
            a->kv_src[kv_pos + j] = a->cand_kv_rows[d0 + j];
            a->kv_dst[kv_pos + j] = blk * a->page_size + pos % a->page_size;
        }
        out_pos += n;
        kv_pos += E;
        a->new_seq_len[i] = P + n;
        a->new_kv_len[i] = P + E;
        int32_t dk = (K - 1 < E) ? K - 1 : E;
        if (dk < 0) dk = 0;
        a->new_draft_len[i] = P + dk;
    }
    a->out_off[a->B] = out_pos;
    a->kv_off[a->B] = kv_pos;
    return 0;
}

/* ---- choosing gamma ---------------------------------------------------------------- */

/* SOTA-227: expected wall-time improvement of drafting gamma tokens at acceptance rate alpha
 * and relative draft cost c: (1 - alpha^(gamma+1)) / ((1 - alpha)(gamma*c + 1)). At
 * alpha == 1 the numerator's ratio is its limit gamma + 1 (SDCP "Drafting and Proposal"). */
double oracle_gamma_objective(double alpha, double c, int32_t gamma) {
    double committed;
    if (alpha == 1.0) {
        committed = (double)gamma + 1.0;
    } else {
        double ag = 1.0;
        for (int32_t k = 0; k < gamma + 1; ++k) ag *= alpha;
        committed = (1.0 - ag) / (1.0 - alpha);
    }
    return committed / ((double)gamma * c + 1.0);
}

/* gamma chosen numerically (SOTA-227): the maximiser over [gamma_min, gamma_max]; an exact
 * tie goes to the smaller gamma (M7.8 section 0x07A breaks ties toward smaller K). alpha is
 * the mean of the per-position acceptance rates; with no draft position measured the previous
 * estimate is kept. */
int32_t oracle_choose_gamma(double alpha_sum, int32_t alpha_count, double alpha_prev, double c,
                            int32_t gamma_min, int32_t gamma_max, double *alpha_out) {
    double alpha = alpha_count > 0 ? alpha_sum / (double)alpha_count : alpha_prev;
    if (alpha < 0.0) alpha = 0.0;
    if (alpha > 1.0) alpha = 1.0;
    if (alpha_out) *alpha_out = alpha;
    int32_t best = gamma_min;
    double best_f = oracle_gamma_objective(alpha, c, gamma_min);
    for (int32_t g = gamma_min + 1; g <= gamma_max; ++g) {
        double f = oracle_gamma_objective(alpha, c, g);
        if (f > best_f) {
            best_f = f;
            best = g;
        }
    }
    return best;
}

/* ---- depth statistics ("M7.8 - Speculative Serving", 0x02D "Estimation Bias And Censoring" and
 * 0x07B): a deeper position is observed only when every earlier draft was accepted, so its rate
 * divides by the requests that reached it, not by the rounds. */
void oracle_depth_counts(int32_t B, const int32_t *row_off, const int32_t *accept_len,
                         const int32_t *req_status, int32_t depth_max, int32_t *n_reached,
                         int32_t *n_accepted) {
    for (int32_t j = 0; j < depth_max; ++j) n_reached[j] = n_accepted[j] = 0;
    for (int32_t i = 0; i < B; ++i) {
        if (req_status[i] != 0) continue;
        const int32_t K = row_off[i + 1] - row_off[i] - 1, A = accept_len[i];
        for (int32_t j = 1; j <= depth_max; ++j) {
            if (K >= j && A >= j - 1) n_reached[j - 1] += 1;
            if (A >= j) n_accepted[j - 1] += 1;
        }
    }
}

void oracle_depth_alpha(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                        double alpha_prev, int32_t n_out, double *alpha_hat) {
    double sr = 0.0, sa = 0.0;
    for (int32_t j = 0; j < depth_max; ++j) {
        sr += (double)n_reached[j];
        sa += (double)n_accepted[j];
    }
    const double pooled = sr > 0.0 ? sa / sr : alpha_prev;
    for (int32_t j = 0; j < n_out; ++j) {
        const int32_t r = j < depth_max ? n_reached[j] : 0;
        alpha_hat[j] = r > 0 ? (double)n_accepted[j] / (double)r : pooled;
    }
}

double oracle_depth_expected_accept(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                                    double alpha_prev, int32_t gamma) {
    double ah[4096];
    if (gamma > 4096) gamma = 4096;
    oracle_depth_alpha(n_reached, n_accepted, depth_max, alpha_prev, gamma, ah);
    double ea = 0.0, prod = 1.0;
    for (int32_t j = 0; j < gamma; ++j) {
        prod *= ah[j];
        ea += prod;
    }
    return ea;
}

double oracle_depth_objective(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                              double alpha_prev, double c, int32_t gamma) {
    const double ea = oracle_depth_expected_accept(n_reached, n_accepted, depth_max, alpha_prev, gamma);
    return (1.0 + ea) / ((double)gamma * c + 1.0);
}

/* The same choice as oracle_choose_gamma (maximiser, ties to the smaller gamma) with E[A] from the
 * per-depth rates in place of the constant-alpha closed form. */
int32_t oracle_choose_gamma_depth(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                                  double alpha_prev, double c, int32_t gamma_min, int32_t gamma_max,
                                  double *ea_out) {
    int32_t best = gamma_min;
    double best_f = oracle_depth_objective(n_reached, n_accepted, depth_max, alpha_prev, c, gamma_min);
    for (int32_t g = gamma_min + 1; g <= gamma_max; ++g) {
        const double f = oracle_depth_objective(n_reached, n_accepted, depth_max, alpha_prev, c, g);
        if (f > best_f) {
            best_f = f;
            best = g;
        }
    }
    if (ea_out) *ea_out = oracle_depth_expected_accept(n_reached, n_accepted, depth_max, alpha_prev, best);
    return best;
}
