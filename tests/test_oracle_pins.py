"""Pins for the float64 oracle, against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself:
  * the exactness theorem (SOTA-227 "Why it is free rather than a trade"; SDCP Rule 2: the
    output has the target's distribution) by a chi-square test over 10^6 rounds;
  * the exact law of a round, enumerated by brute force over all draft sequences (V <= 8,
    K <= 3), which is first checked analytically against the theorem;
  * the accept threshold u <= p/q and the inverse-CDF boundaries, by sweeping the uniforms
    across values computed here from the definition;
  * the acceptance rate alpha = sum min(p, q) and the prefix law Pr(A >= j) = alpha^j
    (M7.8 section 0x02) by binomial / chi-square tests;
  * the gamma objective by exact rational arithmetic of the tail-sum form
    E[C] = 1 + alpha + ... + alpha^gamma (M7.8 section 0x02) and its limits;
  * the page's worked examples stored under tests/golden/.
"""
import itertools
import json
import os
from collections import Counter, defaultdict
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def law(z, T):
    """softmax(z / T) in float64 (the test's own statement of p and q). The temperature is
    a binary32 value at the interface, so it is rounded to one here as well."""
    y = np.asarray(z, np.float64) / float(np.float32(T))
    e = np.exp(y - y.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def trials(tz, dz, T, n, seed, u_override=None):
    """n independent rounds of one request with fixed rows; drafts sampled from q_j."""
    tz = np.asarray(tz, np.float32)
    dz = np.asarray(dz, np.float32)
    K, V = dz.shape
    rng = np.random.default_rng(seed)
    q = law(dz, T)
    cdf = np.cumsum(q, axis=1)
    ux = rng.random((n, K))
    x = np.empty((n, K), np.int32)
    for j in range(K):
        x[:, j] = np.minimum(np.searchsorted(cdf[j], ux[:, j], side="right"), V - 1)
    target = np.tile(tz, (n, 1))
    draft = np.tile(dz, (n, 1))
    row_off = np.arange(n + 1, dtype=np.int32) * (K + 1)
    u = rng.random(n * (K + 1)) if u_override is None else u_override
    out = oracle.verify(target, draft, row_off, x.reshape(-1), u, T)
    return out, x, row_off


def rows_example(V=6, K=3, seed=11, scale=1.3, noise=1.0):
    rng = np.random.default_rng(seed)
    tz = rng.normal(0, scale, size=(K + 1, V))
    dz = tz[:K] + rng.normal(0, noise, size=(K, V))
    return tz.astype(np.float32), dz.astype(np.float32)


# ---------------------------------------------------------------- exactness (chi-square)

@pytest.mark.parametrize("T", [1.0, 0.7])
def test_exactness_chi_square_each_depth(T):
    """Every emitted token, given its depth was reached, is distributed as p at that depth."""
    tz, dz = rows_example()
    K, V = dz.shape
    p = law(tz, T)
    n_total = 1_000_000
    counts = np.zeros((K + 1, V), np.int64)
    for part in range(4):
        out, x, row_off = trials(tz, dz, T, n_total // 4, seed=100 + part + int(10 * T))
        A = out["accept_len"]
        tok = out["out_tokens"].reshape(-1, K + 1)
        assert (out["req_status"] == 0).all()
        for d in range(K + 1):
            reached = A >= d
            counts[d] += np.bincount(tok[reached, d], minlength=V)
    for d in range(K + 1):
        n = counts[d].sum()
        assert n > 10_000
        chi2, pval = stats.chisquare(counts[d], n * p[d])
        assert pval > 1e-3, (d, chi2, pval, counts[d] / n, p[d])


def test_exactness_detects_planted_bias():
    """The chi-square test has power: a sampler that uses q in place of the residual fails."""
    tz, dz = rows_example()
    K, V = dz.shape
    p = law(tz, 1.0)
    q = law(dz, 1.0)
    # depth-0 law of a wrong rule: accept x ~ q with prob min(1,p/q), else resample from q
    a = np.minimum(p[0], q[0])
    wrong = a + (1.0 - a.sum()) * q[0]
    rng = np.random.default_rng(5)
    counts = rng.multinomial(250_000, wrong)
    assert stats.chisquare(counts, 250_000 * p[0]).pvalue < 1e-6


# ---------------------------------------------------------------- exact law by enumeration

def enumerate_law(p, q):
    """Law of the emitted sequence of one round, by summing over every draft sequence."""
    K, V = q.shape
    out = defaultdict(float)

    def walk(xs, j, prob, prefix):
        if j == K:
            for t in range(V):
                out[prefix + (t,)] += prob * p[K][t]
            return
        x = xs[j]
        acc = min(1.0, p[j][x] / q[j][x])
        if acc > 0:
            walk(xs, j + 1, prob * acc, prefix + (x,))
        r = np.maximum(p[j] - q[j], 0.0)
        Z = r.sum()
        if acc < 1 and Z > 0:
            for t in range(V):
                out[prefix + (t,)] += prob * (1 - acc) * r[t] / Z

    for xs in itertools.product(range(V), repeat=K):
        w = np.prod([q[j][xs[j]] for j in range(K)])
        walk(xs, 0, w, ())
    return out


@pytest.mark.parametrize("V,K,T,seed", [(4, 2, 1.0, 3), (5, 3, 0.8, 4), (8, 1, 1.5, 5),
                                        (3, 3, 1.0, 6)])
def test_enumerated_law_satisfies_theorem(V, K, T, seed):
    tz, dz = rows_example(V=V, K=K, seed=seed)
    p, q = law(tz, T), law(dz, T)
    L = enumerate_law(p, q)
    assert abs(sum(L.values()) - 1.0) < 1e-12
    for d in range(K + 1):
        reach = sum(v for s, v in L.items() if len(s) > d)
        marg = np.zeros(V)
        for s, v in L.items():
            if len(s) > d:
                marg[s[d]] += v
        np.testing.assert_allclose(marg / reach, p[d], atol=1e-12)
    # Pr(A >= j) = prod_{m <= j} alpha_m (M7.8 section 0x02B, context-free rows)
    alpha = np.minimum(p[:K], q).sum(axis=1)
    for j in range(1, K + 1):
        tail = sum(v for s, v in L.items() if len(s) - 1 >= j)
        assert abs(tail - np.prod(alpha[:j])) < 1e-12


@pytest.mark.parametrize("V,K,T,seed", [(4, 2, 1.0, 3), (5, 3, 0.8, 4), (3, 3, 1.0, 6)])
def test_oracle_matches_enumerated_law(V, K, T, seed):
    tz, dz = rows_example(V=V, K=K, seed=seed)
    L = enumerate_law(law(tz, T), law(dz, T))
    n = 300_000
    out, x, _ = trials(tz, dz, T, n, seed=seed + 1000)
    tok = out["out_tokens"].reshape(n, K + 1)
    A = out["accept_len"]
    seqs = Counter(tuple(tok[i, :A[i] + 1]) for i in range(n))
    assert set(seqs) <= set(L), set(seqs) - set(L)
    keys = sorted(L, key=lambda s: (len(s), s))
    exp = np.array([L[s] * n for s in keys])
    obs = np.array([seqs.get(s, 0) for s in keys], np.float64)
    big = exp >= 5
    obs_m = np.append(obs[big], obs[~big].sum())
    exp_m = np.append(exp[big], exp[~big].sum())
    if exp_m[-1] < 5:
        obs_m, exp_m = obs_m[:-1], exp_m[:-1]
        exp_m *= obs_m.sum() / exp_m.sum()
    assert stats.chisquare(obs_m, exp_m).pvalue > 1e-3


# ---------------------------------------------------------------- thresholds

def single(tz, dz, xs, u, T=1.0, **kw):
    tz = np.asarray(tz, np.float32)
    dz = np.asarray(dz, np.float32)
    K = dz.shape[0]
    return oracle.verify(tz, dz, np.array([0, K + 1]), np.asarray(xs), np.asarray(u), T, **kw)


def test_accept_threshold_is_p_over_q():
    tz, dz = rows_example(V=6, K=2, seed=21)
    p, q = law(tz, 1.0), law(dz, 1.0)
    x0 = int(np.argmax(q[0] - p[0]))  # p < q here, so rho < 1
    rho = p[0][x0] / q[0][x0]
    assert rho < 0.95
    o = single(tz, dz, [x0, 0], [rho * (1 - 1e-9), 0.5, 0.5])
    assert o["accept_len"][0] >= 1
    np.testing.assert_allclose(o["rho"][0], rho, rtol=1e-12)
    o = single(tz, dz, [x0, 0], [rho * (1 + 1e-9), 0.5, 0.5])
    assert o["accept_len"][0] == 0
    # p >= q: every uniform in [0,1) accepts
    x1 = int(np.argmax(p[0] - q[0]))
    o = single(tz, dz, [x1, 0], [1 - 2 ** -53, 0.5, 0.5])
    assert o["accept_len"][0] >= 1


def residual_boundaries(p, q):
    r = np.maximum(p - q, 0.0)
    C = np.cumsum(r) / r.sum()
    return r, C


def test_residual_draw_switches_at_cdf_boundaries():
    tz, dz = rows_example(V=7, K=2, seed=22)
    # make token 0 a zero-residual token (p_0 <= q_0 at position 0)
    dz[0, 0] = tz[0, 0] + 2.0
    p, q = law(tz, 1.0), law(dz, 1.0)
    r, C = residual_boundaries(p[0], q[0])
    assert r[0] == 0.0
    x0 = 0  # rho < 1 because p_0 < q_0; u = 1 - 2^-53 rejects
    positive = np.nonzero(r > 0)[0]
    o = single(tz, dz, [x0, 1], [1 - 2 ** -53, 0.5, 0.0])
    assert o["accept_len"][0] == 0
    assert o["out_tokens"][0] == positive[0]  # u = 0 -> first token of positive mass
    for k, tok in enumerate(positive[:-1]):
        nxt = positive[k + 1]
        lo = single(tz, dz, [x0, 1], [1 - 2 ** -53, 0.5, C[tok] - 1e-9])
        hi = single(tz, dz, [x0, 1], [1 - 2 ** -53, 0.5, C[tok] + 1e-9])
        assert lo["out_tokens"][0] == tok
        assert hi["out_tokens"][0] == nxt
    o = single(tz, dz, [x0, 1], [1 - 2 ** -53, 0.5, 1 - 2 ** -53])
    assert o["out_tokens"][0] == positive[-1]
    np.testing.assert_allclose(o["resid_mass"][0], r.sum(), rtol=1e-12)


def test_residual_conditioning_closed_forms():
    """The conditioning diagnostics on rows whose residual is known in closed form."""
    # p = (3/4, 1/4), q = (1/2, 1/2): draft token 1 has rho = 1/2, u = 0.9 rejects; the residual
    # is (1/4, 0), Z = 1/4, its support {0} carries p + q = 5/4; the drawn token 0 has
    # (p + q) / (p - q) = 5 and Z's own bound is (5/4) / (1/4) = 5.
    o = single([[np.log(3.0), 0.0], [0.0, 0.0]], [[0.0, 0.0]], [1], [0.9, 0.3])
    assert o["accept_len"][0] == 0 and o["out_tokens"][0] == 0
    np.testing.assert_allclose(o["resid_mass"][0], 0.25, rtol=1e-6)
    np.testing.assert_allclose(o["resid_scale"][0], 1.25, rtol=1e-6)
    np.testing.assert_allclose(o["sample_cond"][0], 10.0, rtol=1e-5)
    # disjoint supports: p = (1, 0), q = (0, 1); the residual is p itself, every bound is 1
    o = single([[0.0, -np.inf], [0.0, 0.0]], [[-np.inf, 0.0]], [1], [0.5, 0.7])
    assert o["accept_len"][0] == 0 and o["out_tokens"][0] == 0
    assert o["resid_mass"][0] == 1.0 and o["resid_scale"][0] == 1.0 and o["sample_cond"][0] == 2.0
    # identical rows: no residual at all (Z = 0, empty support); the bonus draw is from p
    tz, _ = rows_example(V=6, K=1, seed=25)
    o = single(tz, tz[:1], [2], [0.999, 0.4])
    assert o["accept_len"][0] == 1
    assert o["resid_mass"][0] == 0.0 and o["resid_scale"][0] == 0.0 and o["sample_cond"][0] == 1.0
    # greedy picks and bad requests
    o = single(tz, tz[:1] + 1.0, [int(np.argmax(tz[0])) ^ 1], [0.5, 0.5], T=0.0)
    assert o["accept_len"][0] == 0 and o["sample_cond"][0] == 1.0
    o = single(tz, tz[:1], [9], [0.5, 0.5])
    assert o["req_status"][0] == oracle.REQ_BAD_PROPOSAL
    assert np.isnan(o["sample_cond"][0]) and np.isnan(o["resid_scale"][0])


def test_resid_scale_is_the_positive_part_support_mass():
    tz, dz = rows_example(V=9, K=3, seed=26)
    p, q = law(tz, 0.8), law(dz, 0.8)
    o = single(tz, dz, [0, 1, 2], [0.1, 0.2, 0.3, 0.4], T=0.8)
    want = np.where(p[:3] > q, p[:3] + q, 0.0).sum(axis=1)
    np.testing.assert_allclose(o["resid_scale"], want, rtol=1e-12)
    # the bound is never below 1: the support's p + q is at least its p - q
    assert (o["resid_scale"] >= o["resid_mass"]).all()


def test_threaded_oracle_equals_serial():
    """The OpenMP split over requests changes nothing: every output, bit for bit."""
    tz, dz, row_off, toks, u, K = ragged_batch(40, 30, 5, seed=57)
    temp = np.linspace(0.0, 1.3, 40).astype(np.float32)
    dz[row_off[3] - 3] = np.nan if K[3] > 0 else dz[row_off[3] - 3]
    a = oracle.verify(tz, dz, row_off, toks, u, temp, top_k=7, top_p=0.8)
    b = oracle.verify(tz, dz, row_off, toks, u, temp, top_k=7, top_p=0.8, threads=4)
    assert b.pop("threads_used") >= 1
    assert a.keys() == b.keys()
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_bonus_draw_uses_last_target_row_and_sample_slot():
    tz, dz = rows_example(V=6, K=3, seed=23)
    p = law(tz, 0.9)
    C = np.cumsum(p[3])
    xs = [0, 1, 2]
    for tok in range(5):
        for delta, want in ((-1e-9, tok), (1e-9, tok + 1)):
            u = [0.0, 0.0, 0.0, C[tok] + delta]
            o = single(tz, dz, xs, u, T=0.9)
            assert o["accept_len"][0] == 3
            assert list(o["out_tokens"][:3]) == xs
            assert o["out_tokens"][3] == want
    # the accept draws do not move the extra token
    o1 = single(tz, dz, xs, [0.0, 0.0, 0.0, 0.42], T=0.9)
    o2 = single(tz, dz, xs, [1e-12, 1e-12, 1e-12, 0.42], T=0.9)
    assert o1["out_tokens"][3] == o2["out_tokens"][3]


def test_zero_target_probability_is_never_accepted():
    tz, dz = rows_example(V=5, K=1, seed=24)
    tz[0, 2] = -np.inf
    o = single(tz, dz, [2], [0.0, 0.3])
    assert o["accept_len"][0] == 0 and o["rho"][0] == 0.0
    assert o["out_tokens"][0] != 2


# ---------------------------------------------------------------- acceptance rate

def test_acceptance_rate_is_sum_min_p_q():
    tz, dz = rows_example(V=6, K=3, seed=31)
    T = 1.0
    p, q = law(tz, T), law(dz, T)
    alpha = np.minimum(p[:3], q).sum(axis=1)
    n = 400_000
    out, _, _ = trials(tz, dz, T, n, seed=77)
    np.testing.assert_allclose(out["alpha"][:3], alpha, rtol=1e-12)
    A = out["accept_len"]
    frac = (A >= 1).mean()
    assert abs(frac - alpha[0]) < 4 * np.sqrt(alpha[0] * (1 - alpha[0]) / n)
    EA = sum(np.prod(alpha[:j]) for j in range(1, 4))
    sd = A.std()
    assert abs(A.mean() - EA) < 4 * sd / np.sqrt(n)


def test_prefix_law_constant_alpha():
    """Identical rows at every depth: Pr(A = a) = alpha^a (1 - alpha), Pr(A = K) = alpha^K."""
    rng = np.random.default_rng(41)
    V, K = 6, 4
    t1 = rng.normal(0, 1, V)
    d1 = t1 + rng.normal(0, 0.8, V)
    tz = np.tile(t1, (K + 1, 1))
    dz = np.tile(d1, (K, 1))
    a = np.minimum(law(t1, 1.0), law(d1, 1.0)).sum()
    n = 300_000
    out, _, _ = trials(tz, dz, 1.0, n, seed=42)
    A = out["accept_len"]
    pmf = np.array([a ** k * (1 - a) for k in range(K)] + [a ** K])
    assert abs(pmf.sum() - 1) < 1e-12
    assert stats.chisquare(np.bincount(A, minlength=K + 1), n * pmf).pvalue > 1e-3
    EC = (1 - a ** (K + 1)) / (1 - a)
    n_emit = out["n_emitted"]
    assert abs(n_emit.mean() - EC) < 4 * n_emit.std() / np.sqrt(n)


# ---------------------------------------------------------------- greedy (Rule 1)

def test_sdcp_greedy_worked_round():
    g = json.load(open(os.path.join(GOLDEN, "sdcp_greedy_round.json")))
    V = 16
    M = len(g["drafts"])
    tz = np.zeros((M + 1, V), np.float32)
    for j, a in enumerate(g["target_argmax"]):
        tz[j, a] = 5.0
    # a tie at a smaller id than the argmax would break toward the smaller id: none here
    dz = np.zeros((M, V), np.float32)
    o = single(tz, dz, g["drafts"], np.zeros(M + 1), T=0.0)
    assert o["accept_len"][0] == g["accepted"]
    n = o["n_emitted"][0]
    assert list(o["out_tokens"][:n]) == g["emitted"]
    assert g["committed_before"] + n == g["committed_after"]


def test_greedy_ties_break_to_smallest_id():
    V = 8
    tz = np.zeros((2, V), np.float32)
    tz[0, [3, 5]] = 2.0
    tz[1, [1, 6]] = 1.0
    dz = np.zeros((1, V), np.float32)
    o = single(tz, dz, [5], [0.0, 0.0], T=0.0)
    assert o["accept_len"][0] == 0 and o["out_tokens"][0] == 3
    o = single(tz, dz, [3], [0.0, 0.0], T=0.0)
    assert o["accept_len"][0] == 1 and list(o["out_tokens"][:2]) == [3, 1]


# ---------------------------------------------------------------- invariants and status

def ragged_batch(B, V, Kmax, seed, dtype=np.float32):
    rng = np.random.default_rng(seed)
    K = rng.integers(0, Kmax + 1, size=B)
    row_off = np.concatenate([[0], np.cumsum(K + 1)]).astype(np.int32)
    T = int(row_off[-1])
    tz = rng.normal(0, 2, size=(T, V)).astype(np.float32)
    dz = np.empty((T - B, V), np.float32)
    toks = np.empty(T - B, np.int32)
    for i in range(B):
        for j in range(K[i]):
            d = row_off[i] - i + j
            dz[d] = tz[row_off[i] + j] + rng.normal(0, 1, V)
            toks[d] = rng.choice(V, p=law(dz[d], 1.0))
    u = rng.random(T)
    return tz, dz, row_off, toks, u, K


def test_round_invariants_ragged():
    tz, dz, row_off, toks, u, K = ragged_batch(64, 50, 7, seed=51)
    o = oracle.verify(tz, dz, row_off, toks, u, 1.0)
    assert (o["req_status"] == 0).all()
    for i in range(64):
        A = o["accept_len"][i]
        n = o["n_emitted"][i]
        assert 0 <= A <= K[i] and n == A + 1 and 1 <= n <= K[i] + 1
        seg = o["out_tokens"][row_off[i]:row_off[i + 1]]
        d0 = row_off[i] - i
        assert list(seg[:A]) == list(toks[d0:d0 + A])
        assert 0 <= seg[A] < 50
        assert (seg[A + 1:] == -1).all()
        for j in range(A):
            assert u[row_off[i] + j] <= o["rho"][d0 + j]
        if A < K[i]:
            assert u[row_off[i] + A] > o["rho"][d0 + A]
    assert np.isnan(o["sample_margin"]).sum() == 0
    assert ((o["alpha"] + o["resid_mass"]) - 1.0 < 1e-12).all()


def test_bf16_input_equals_widened_fp32():
    tz, dz, row_off, toks, u, _ = ragged_batch(16, 40, 4, seed=52)
    tb = (tz.view(np.uint32) >> 16).astype(np.uint16)
    db = (dz.view(np.uint32) >> 16).astype(np.uint16)
    tw = (tb.astype(np.uint32) << 16).view(np.float32)
    dw = (db.astype(np.uint32) << 16).view(np.float32)
    a = oracle.verify(tb, db, row_off, toks, u, 0.7)
    b = oracle.verify(tw, dw, row_off, toks, u, 0.7)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_bad_requests_emit_nothing_and_do_not_disturb_others():
    tz, dz, row_off, toks, u, K = ragged_batch(12, 30, 3, seed=53)
    ref = oracle.verify(tz, dz, row_off, toks, u, 1.0)
    K = np.diff(row_off) - 1
    withd = [i for i in range(12) if K[i] > 0]
    i_nan, i_tok, i_q0 = withd[0], withd[1], withd[2]
    tz2, dz2, toks2 = tz.copy(), dz.copy(), toks.copy()
    tz2[row_off[i_nan], 3] = np.nan
    toks2[row_off[i_tok] - i_tok] = 30
    x = toks2[row_off[i_q0] - i_q0]
    dz2[row_off[i_q0] - i_q0, x] = -np.inf
    temp = np.ones(12, np.float32)
    temp[withd[3]] = -1.0
    o = oracle.verify(tz2, dz2, row_off, toks2, u, temp)
    assert o["req_status"][i_nan] == oracle.REQ_BAD_LOGITS
    assert o["req_status"][i_tok] == oracle.REQ_BAD_PROPOSAL
    assert o["req_status"][i_q0] == oracle.REQ_BAD_PROPOSAL
    assert o["req_status"][withd[3]] == oracle.REQ_BAD_PARAM
    bad = {i_nan, i_tok, i_q0, withd[3]}
    for i in range(12):
        seg = o["out_tokens"][row_off[i]:row_off[i + 1]]
        if i in bad:
            assert o["n_emitted"][i] == 0 and (seg == -1).all()
        else:
            assert o["req_status"][i] == 0
            np.testing.assert_array_equal(seg, ref["out_tokens"][row_off[i]:row_off[i + 1]])
    o = oracle.verify(tz, dz, row_off, toks, u, 1.0, K_max=2)
    assert all(o["req_status"][i] == oracle.REQ_BAD_SHAPE for i in range(12) if K[i] > 2)


def test_stopping_truncates_after_stop_token_and_at_budget():
    tz, dz, row_off, toks, u, K = ragged_batch(20, 30, 5, seed=54)
    ref = oracle.verify(tz, dz, row_off, toks, u, 1.0)
    B = 20
    stop = np.full(B, -1, np.int32)
    budget = np.full(B, 100, np.int32)
    for i in range(B):
        n = ref["n_emitted"][i]
        seg = ref["out_tokens"][row_off[i]:row_off[i] + n]
        if i % 3 == 0 and n >= 2:
            stop[i] = seg[n // 2]
        if i % 3 == 1:
            budget[i] = max(0, n - 2)
    o = oracle.verify(tz, dz, row_off, toks, u, 1.0, stop_token=stop, max_new=budget)
    for i in range(B):
        n0 = ref["n_emitted"][i]
        seg0 = list(ref["out_tokens"][row_off[i]:row_off[i] + n0])
        want = seg0[:budget[i]]
        if stop[i] >= 0 and stop[i] in want:
            want = want[:want.index(stop[i]) + 1]
        n = o["n_emitted"][i]
        assert n == len(want)
        assert list(o["out_tokens"][row_off[i]:row_off[i] + n]) == want
        assert (o["out_tokens"][row_off[i] + n:row_off[i + 1]] == -1).all()
        assert o["accept_len"][i] == ref["accept_len"][i]


# ---------------------------------------------------------------- gamma objective

def committed_tail_sum(alpha: Fraction, gamma: int) -> Fraction:
    """E[committed] = 1 + alpha + ... + alpha^gamma (M7.8 section 0x02, tail-sum identity)."""
    return sum((alpha ** j for j in range(gamma + 1)), Fraction(0))


def test_gamma_objective_closed_forms():
    a = Fraction(7, 10)
    for g, want in zip(range(1, 5), ("1.7", "2.19", "2.533", "2.7731")):
        assert committed_tail_sum(a, g) == Fraction(want)
        assert abs(oracle.gamma_objective(0.7, 0.0, g) - float(Fraction(want))) < 1e-14
    for alpha in (0.0, 0.3, 0.99):
        assert oracle.gamma_objective(alpha, 0.37, 0) == 1.0
    # c -> 0, gamma -> infinity: 1 / (1 - alpha) (SOTA-227)
    assert abs(oracle.gamma_objective(0.7, 0.0, 400) - 1 / 0.3) < 1e-12
    # alpha = 1: gamma + 1 committed tokens (SDCP "Drafting and Proposal")
    assert oracle.gamma_objective(1.0, 0.25, 3) == 4 / 1.75
    for alpha, c, g in ((0.55, 0.1, 3), (0.9, 0.02, 7), (0.1, 0.5, 2)):
        f = committed_tail_sum(Fraction(alpha), g) / (g * Fraction(c) + 1)
        assert abs(oracle.gamma_objective(alpha, c, g) - float(f)) < 1e-14


def test_choose_gamma_argmax_near_tie_and_rules():
    a, c = Fraction(7, 10), Fraction(1, 20)
    f = {g: committed_tail_sum(a, g) / (g * c + 1) for g in range(0, 9)}
    best = max(f, key=lambda g: (f[g], -g))
    assert best == 6 and f[6] == Fraction(3058819, 1300000)
    assert 0 < f[6] - f[5] < Fraction(2, 10 ** 6)
    g, alpha = oracle.choose_gamma(0.7 * 40, 40, 0.1, 0.05)
    assert (g, round(alpha, 12)) == (6, 0.7)
    # exact tie everywhere (alpha = 1, c = 1): the smallest gamma wins
    assert oracle.choose_gamma(5.0, 5, 0.0, 1.0, 2, 8)[0] == 2
    # nothing measured: the previous alpha is kept
    assert oracle.choose_gamma(0.0, 0, 0.7, 0.05) == (6, 0.7)
    # alpha = 0: drafting never pays
    assert oracle.choose_gamma(0.0, 10, 0.5, 0.05)[0] == 0


# ---------------------------------------------------------------- compaction ledgers

def ledger_round(P, K, A, stop):
    """One request with K drafts whose first A are accepted, then compacted."""
    V = 32
    tz = np.zeros((K + 1, V), np.float32)
    dz = np.zeros((K, V), np.float32)
    xs = list(range(1, K + 1))
    u = np.zeros(K + 1)
    if A < K:
        u[A] = 1 - 2 ** -53  # q = p = uniform gives rho = 1: force rejection via zero p(x)
        tz[A, xs[A]] = -np.inf
    u[K] = 0.5
    stop_token = np.array([-1], np.int32)
    max_new = np.array([1000], np.int32)
    if stop == "max_new=4":
        max_new[0] = 4
    o = oracle.verify(tz, dz, np.array([0, K + 1]), np.array(xs), u, 1.0,
                      stop_token=stop_token, max_new=max_new)
    if stop == "eos_at_bonus":
        stop_token[0] = o["out_tokens"][A]
        o = oracle.verify(tz, dz, np.array([0, K + 1]), np.array(xs), u, 1.0,
                          stop_token=stop_token, max_new=max_new)
    assert o["accept_len"][0] == A
    page = 4
    nblk = 8
    block_table = (np.arange(nblk, dtype=np.int32)[::-1] + 10).reshape(1, nblk)
    cand = np.arange(K, dtype=np.int32) + 500
    c = oracle.compact(np.array([0, K + 1]), o["accept_len"], o["n_emitted"], o["out_tokens"],
                       o["req_status"], np.array([P]), cand, block_table, page)
    return o, c, block_table, page, cand


def test_m78_cache_ledgers():
    g = json.load(open(os.path.join(GOLDEN, "m78_cache_ledgers.json")))
    P, K = g["P"], g["K"]
    for case in g["cases"]:
        o, c, bt, page, cand = ledger_round(P, K, case["A"], case["stop"])
        assert c["new_seq_len"][0] == case["L_out"], case["name"]
        assert c["new_kv_len"][0] == case["L_target"], case["name"]
        assert c["new_draft_len"][0] == case["L_draft"], case["name"]
        n = c["out_off"][1]
        assert list(c["packed_pos"]) == list(range(P, P + n))
        E = c["kv_off"][1]
        assert list(c["kv_src"]) == list(cand[:E])
        want_dst = [bt[0, (P + j) // page] * page + (P + j) % page for j in range(E)]
        assert list(c["kv_dst"]) == want_dst


def test_compaction_batch_properties():
    tz, dz, row_off, toks, u, K = ragged_batch(40, 30, 6, seed=61)
    o = oracle.verify(tz, dz, row_off, toks, u, 1.0)
    B = 40
    rng = np.random.default_rng(62)
    P = rng.integers(0, 200, size=B).astype(np.int32)
    page = 16
    nblk = 32
    perm = rng.permutation(B * nblk).astype(np.int32).reshape(B, nblk)
    cand = rng.permutation(10_000)[: int(row_off[-1]) - B].astype(np.int32)
    c = oracle.compact(row_off, o["accept_len"], o["n_emitted"], o["out_tokens"],
                       o["req_status"], P, cand, perm, page)
    assert c["out_off"][-1] == o["n_emitted"].sum()
    assert c["kv_off"][-1] == o["accept_len"].sum()
    assert len(set(c["kv_dst"].tolist())) == len(c["kv_dst"])
    for i in range(B):
        s, e = c["out_off"][i], c["out_off"][i + 1]
        assert list(c["packed_pos"][s:e]) == list(range(P[i], P[i] + e - s))
        assert list(c["packed_tokens"][s:e]) == list(o["out_tokens"][row_off[i]:row_off[i] + e - s])
        assert c["new_seq_len"][i] == P[i] + o["accept_len"][i] + 1
        assert c["new_kv_len"][i] == P[i] + o["accept_len"][i]
        ks, ke = c["kv_off"][i], c["kv_off"][i + 1]
        for j in range(ke - ks):
            pos = P[i] + j
            assert c["kv_dst"][ks + j] // page == perm[i, pos // page]
            assert c["kv_dst"][ks + j] % page == pos % page
    # a request whose committed positions run past its block table commits nothing
    P2 = P.copy()
    P2[0] = nblk * page - 1
    c2 = oracle.compact(row_off, o["accept_len"], o["n_emitted"], o["out_tokens"],
                        o["req_status"], P2, cand, perm, page)
    if o["accept_len"][0] >= 2:
        assert c2["compact_status"][0] == oracle.REQ_BAD_BLOCKS
        assert c2["out_off"][1] == 0 and c2["new_seq_len"][0] == P2[0]
