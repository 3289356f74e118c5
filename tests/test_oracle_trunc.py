"""Pins for the oracle's top-k / top-p truncation of the target law.

SDCP, section "Session Model": p is the target model's next-token distribution after
temperature, top-k and top-p, in that order; the draft's q is not truncated. The readings of
what the page leaves open (ties rank by ascending token id; top-p keeps the shortest head whose
mass, renormalised over the top-k set, reaches top_p) are pinned here by:
  * reduction to a special case: top_k = 1 turns Rule 2 into Rule 1 (the greedy rule);
  * laws computed here by hand for small rows (the kept set, alpha, the residual mass, rho);
  * an example in which top-k-then-top-p and the reverse order keep different sets;
  * ties at the cut, broken by token id;
  * the exactness theorem for the truncated law, by a chi-square test.
"""
import numpy as np
import pytest
from scipy import stats

import oracle


def law(z, T):
    y = np.asarray(z, np.float64) / float(np.float32(T))
    e = np.exp(y - y.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def truncated(z, T, k, top_p):
    """The test's own statement of the truncated law: rank by (logit desc, id asc), keep k,
    renormalise, keep the shortest head reaching top_p, renormalise."""
    z = np.asarray(z, np.float32).astype(np.float64)
    V = z.shape[0]
    order = sorted(range(V), key=lambda v: (-z[v], v))
    n = k if 0 < k < V else V
    p = law(z, T)
    head = order[:n]
    if top_p < 1.0:
        pk = p[head] / p[head].sum()
        c = np.cumsum(pk)
        n = int(np.argmax(c >= top_p)) + 1
        head = head[:n]
    out = np.zeros(V)
    out[head] = p[head] / p[head].sum()
    return out


def one(tz, dz, xs, u, T, **kw):
    tz = np.asarray(tz, np.float32)
    dz = np.asarray(dz, np.float32)
    K = dz.shape[0]
    return oracle.verify(tz, dz, np.array([0, K + 1]), np.asarray(xs), np.asarray(u), T, **kw)


def test_hand_computed_top_p_law():
    """p = (0.5, 0.3, 0.15, 0.05), top_p = 0.75 keeps {0, 1} (0.5 < 0.75 <= 0.8): p' =
    (0.625, 0.375, 0, 0). Against q uniform: alpha = 0.25 + 0.25 = 0.5, residual mass
    0.375 + 0.125 = 0.5, rho(0) = 2.5, rho(2) = 0 (a truncated token is never accepted)."""
    tz = np.log(np.array([[0.5, 0.3, 0.15, 0.05]] * 2))
    dz = np.zeros((1, 4))
    o = one(tz, dz, [0], [0.9, 0.5], 1.0, top_p=0.75)
    assert o["req_status"][0] == 0
    np.testing.assert_allclose(o["alpha"][0], 0.5, rtol=1e-6)
    np.testing.assert_allclose(o["resid_mass"][0], 0.5, rtol=1e-6)
    np.testing.assert_allclose(o["rho"][0], 2.5, rtol=1e-6)
    assert o["trunc_keep"][0] == 2 and o["trunc_keep"][1] == 2
    np.testing.assert_allclose(o["trunc_margin"][0], 0.05, rtol=1e-5)
    o = one(tz, dz, [2], [0.0, 0.5], 1.0, top_p=0.75)
    assert o["rho"][0] == 0.0 and o["accept_len"][0] == 0
    # the frontier (slot A = 0) comes from max(p' - q, 0) = (0.375, 0.125, 0, 0), Z = 0.5
    assert o["out_tokens"][0] == 0  # u = 0.5: u Z = 0.25 < 0.375, token 0
    o = one(tz, dz, [2], [0.0, 0.8], 1.0, top_p=0.75)
    assert o["out_tokens"][0] == 1  # u = 0.8: u Z = 0.4 >= 0.375, token 1


def test_order_top_k_then_top_p():
    """p = (0.4, 0.3, 0.2, 0.1), top_k = 2, top_p = 0.5: the top-k head renormalised is
    (4/7, 3/7), whose first token already reaches 0.5, so one token is kept. Top-p first would
    keep {0, 1} (0.4 < 0.5 <= 0.7) and top-k would leave it at two."""
    tz = np.log(np.array([[0.4, 0.3, 0.2, 0.1]] * 2))
    dz = np.zeros((1, 4))
    o = one(tz, dz, [1], [0.0, 0.5], 1.0, top_k=2, top_p=0.5)
    assert o["trunc_keep"][0] == 1
    assert o["rho"][0] == 0.0  # token 1 is gone
    np.testing.assert_allclose(o["alpha"][0], 0.25, rtol=1e-6)  # min(1, 0.25) at token 0
    o = one(tz, dz, [1], [0.0, 0.5], 1.0, top_k=2)
    assert o["trunc_keep"][0] == 2
    np.testing.assert_allclose(o["rho"][0], (3 / 7) / 0.25, rtol=1e-6)


def test_ties_at_the_cut_break_by_token_id():
    """Logits (1, 2, 2, 2, 0): the ranking is 1, 2, 3, 0, 4; top_k = 2 keeps {1, 2}, each 1/2."""
    tz = np.array([[1.0, 2.0, 2.0, 2.0, 0.0]] * 2)
    dz = np.zeros((1, 5))
    for x, rho in [(1, 0.5 / 0.2), (2, 0.5 / 0.2), (3, 0.0), (0, 0.0)]:
        o = one(tz, dz, [x], [0.0, 0.5], 1.0, top_k=2)
        assert o["trunc_keep"][0] == 2
        np.testing.assert_allclose(o["rho"][0], rho, rtol=1e-6)


@pytest.mark.parametrize("seed", [3, 4])
def test_top_k_one_is_the_greedy_rule(seed):
    """With top_k = 1 the truncated law is the point mass at argmax p (smallest id on ties):
    Rule 2 then accepts exactly the drafts equal to it and draws the correction from it, i.e.
    it reduces to Rule 1 (SDCP "Acceptance Rules"). Compared with the oracle at T = 0."""
    rng = np.random.default_rng(seed)
    B, K, V = 40, 3, 9
    tz = rng.integers(-3, 4, size=(B * (K + 1), V)).astype(np.float32)  # many ties
    dz = rng.normal(0, 1, size=(B * K, V)).astype(np.float32)
    row_off = np.arange(B + 1, dtype=np.int32) * (K + 1)
    am = np.argmax(tz, axis=1).reshape(B, K + 1)
    xs = np.where(rng.random((B, K)) < 0.6, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    u = rng.random(B * (K + 1))
    t = oracle.verify(tz, dz, row_off, xs.reshape(-1), u, 0.8, top_k=1)
    g = oracle.verify(tz, dz, row_off, xs.reshape(-1), u, 0.0)
    assert (t["req_status"] == 0).all() and (g["req_status"] == 0).all()
    np.testing.assert_array_equal(t["accept_len"], g["accept_len"])
    np.testing.assert_array_equal(t["out_tokens"], g["out_tokens"])


def test_no_truncation_parameters_change_nothing():
    rng = np.random.default_rng(8)
    B, K, V = 20, 3, 50
    tz = rng.normal(0, 2, size=(B * (K + 1), V)).astype(np.float32)
    dz = (tz.reshape(B, K + 1, V)[:, :K].reshape(-1, V) + rng.normal(0, 1, (B * K, V))).astype(np.float32)
    row_off = np.arange(B + 1, dtype=np.int32) * (K + 1)
    xs = rng.integers(0, V, B * K).astype(np.int32)
    u = rng.random(B * (K + 1))
    a = oracle.verify(tz, dz, row_off, xs, u, 0.9)
    b = oracle.verify(tz, dz, row_off, xs, u, 0.9, top_k=np.zeros(B, np.int32), top_p=np.ones(B, np.float32))
    c = oracle.verify(tz, dz, row_off, xs, u, 0.9, top_k=np.full(B, V, np.int32))
    for o in (b, c):
        for key in ("accept_len", "out_tokens", "req_status"):
            np.testing.assert_array_equal(a[key], o[key])
        for key in ("alpha", "rho", "resid_mass"):
            np.testing.assert_array_equal(a[key], o[key])


def test_nan_top_p_is_a_bad_parameter():
    tz = np.zeros((2, 4))
    dz = np.zeros((1, 4))
    o = one(tz, dz, [0], [0.1, 0.5], 1.0, top_p=float("nan"))
    assert o["req_status"][0] == 8 and o["n_emitted"][0] == 0


@pytest.mark.parametrize("k,top_p", [(4, 0.9), (0, 0.7), (3, 1.0)])
def test_exactness_of_the_truncated_law(k, top_p):
    """Every emitted token, given its depth was reached, is distributed as the truncated law p'
    at that depth (the exactness theorem applied to p'). Drafts are sampled from q."""
    rng = np.random.default_rng(17)
    K, V, T = 2, 7, 1.0
    tz = rng.normal(0, 1.2, size=(K + 1, V)).astype(np.float32)
    dz = (tz[:K] + rng.normal(0, 0.9, size=(K, V))).astype(np.float32)
    pt = np.stack([truncated(tz[d], T, k, top_p) for d in range(K + 1)])
    q = law(dz, T)
    n = 400_000
    cdf = np.cumsum(q, axis=1)
    ux = rng.random((n, K))
    x = np.stack([np.minimum(np.searchsorted(cdf[j], ux[:, j], side="right"), V - 1) for j in range(K)], 1)
    row_off = np.arange(n + 1, dtype=np.int32) * (K + 1)
    out = oracle.verify(np.tile(tz, (n, 1)), np.tile(dz, (n, 1)), row_off, x.reshape(-1).astype(np.int32),
                        rng.random(n * (K + 1)), T, top_k=k, top_p=top_p)
    assert (out["req_status"] == 0).all()
    A = out["accept_len"]
    tok = out["out_tokens"].reshape(-1, K + 1)
    for d in range(K + 1):
        reached = A >= d
        counts = np.bincount(tok[reached, d], minlength=V)
        keep = pt[d] > 0
        assert counts[~keep].sum() == 0, (d, counts, pt[d])
        m = counts.sum()
        assert m > 10_000
        assert stats.chisquare(counts[keep], m * pt[d][keep]).pvalue > 1e-3, (d, counts, pt[d])


def test_top_p_margin_ignores_the_empty_head():
    """top_p <= 0 keeps the first token whatever the masses; the only cumulative mass at the cut
    is that token's. For p = (0.5, 0.3, 0.15, 0.05): margin 0.5 at top_p = 0, and at top_p = 0.6
    (cut after two tokens) min(|0.8 - 0.6|, |0.5 - 0.6|) = 0.1."""
    tz = np.log(np.array([[0.5, 0.3, 0.15, 0.05]] * 2))
    dz = np.zeros((1, 4))
    o = one(tz, dz, [0], [0.9, 0.5], 1.0, top_p=0.0)
    assert o["trunc_keep"][0] == 1
    np.testing.assert_allclose(o["trunc_margin"][0], 0.5, rtol=1e-6)
    o = one(tz, dz, [0], [0.9, 0.5], 1.0, top_p=0.6)
    assert o["trunc_keep"][0] == 2
    np.testing.assert_allclose(o["trunc_margin"][0], 0.1, rtol=1e-5)
