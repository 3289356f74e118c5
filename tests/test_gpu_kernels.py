"""GPU: which per-position kernel spec_verify launches, and the parity of each one.

spec_verify has two per-position kernels with the same results: spec_stream_kernel (row slices
streamed in tiles, pass 2 one item late) and spec_rows_kernel (row slices held whole, two CTAs
per SM). The library picks one per shape (spec_verify_plan); SPEC_VERIFY_KERNEL forces either,
and every case below runs under both, against the float64 oracle.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_43_gb300 import api
from speculative_decoding_verification_43_gb300 import workloads as W

import test_gpu_parity as G

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["rows", "stream"])
def kernel(request, monkeypatch):
    monkeypatch.setenv("SPEC_VERIFY_KERNEL", request.param)
    return request.param


def _rows(wl):
    return W.make_round(wl, seed=0, rnd=0, device="cuda").T


def test_plan_of_the_workloads(monkeypatch):
    """Every workload's row slices fit the streaming kernel's tiles: it runs them all, on
    clusters that keep at least 120 of the 152 SMs busy (c3: 4-CTA clusters)."""
    monkeypatch.delenv("SPEC_VERIFY_KERNEL", raising=False)
    for name in ("c1", "c2", "c3", "c4", "c5"):
        wl = W.WORKLOADS[name]
        kern, c, n = api.verify_plan(wl.B, wl.V, _rows(wl), wl.dtype)
        assert kern == "spec_stream_kernel", (name, kern, c, n)
        assert n * c >= min(120, _rows(wl) * c), (name, c, n)
        if name == "c3":
            assert c == 4


def test_forced_plan(kernel):
    c3 = W.WORKLOADS["c3"]
    name, c, n = api.verify_plan(c3.B, c3.V, _rows(c3), c3.dtype)
    assert name == f"spec_{kernel}_kernel"
    assert n >= 1 and c in (1, 2, 4, 8, 16)


def test_invalid_shapes_have_no_plan():
    assert api.verify_plan(0, 1000, 10, torch.float32) is None
    assert api.verify_plan(4, 1001, 10, torch.bfloat16) is None  # a row of 2002 bytes
    assert api.verify_plan(8, 1024, 7, torch.float32) is None    # fewer rows than requests


def test_c3_full_batch(kernel):
    G.test_c3_full_batch()


def test_c5_sampled(kernel):
    G.test_full_size_sampled("c5", 32)


@pytest.mark.parametrize("dtype,V,B,Kspec,T", [
    (torch.bfloat16, 50264, 40, "uniform:0:8", 0.8),
    (torch.float32, 12348, 24, "uniform:0:6", 1.3),
    (torch.float32, 8, 9, "uniform:0:3", 0.9),
    (torch.bfloat16, 262144, 6, "uniform:1:3", 1.0),
])
def test_shapes(kernel, dtype, V, B, Kspec, T):
    G.test_shapes(dtype, V, B, Kspec, T)


def test_greedy_and_mixed_temperatures(kernel):
    G.test_greedy_and_mixed_temperatures()


def test_bad_requests(kernel):
    G.test_bad_requests()
    G.test_k_max_exceeded_is_bad_shape()


def test_top_k_top_p(kernel):
    G.test_top_k_top_p(torch.bfloat16, 32000, "zipf")
    G.test_top_k_cuts_inside_ties()


def test_wide_logit_ranges(kernel):
    G.test_wide_logit_ranges(torch.bfloat16, 131072)


def _round_case(wl, seed, **verify_kw):
    rd = W.make_round(wl, seed=seed, rnd=0, device="cuda")
    ci = W.make_compaction_inputs(rd, 37, 16)
    outs = []
    for fused in (False, True):
        v = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype)
        v.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature, **verify_kw)
        c = api.Compactor(rd.B, rd.T)
        c.bind(rd.row_off, v.out.accept_len, v.out.n_emitted, v.out.out_tokens, v.out.req_status,
               ci["prefix_len"], ci["cand_kv_rows"], ci["block_table"], 16)
        if fused:
            vo, co, (g, a) = api.run_round(v, c, 0.4, 0.05, 1, 12)
        else:
            vo = v.run()
            co = c.run()
            g, a = api.choose_gamma(vo.alpha_sum, vo.alpha_count, 0.4, 0.05, 1, 12)
        torch.cuda.synchronize()
        d = {k: t.cpu().clone() for k, t in vars(vo).items() if isinstance(t, torch.Tensor)}
        d.update({"c_" + k: t.cpu().clone() for k, t in vars(co).items() if isinstance(t, torch.Tensor)})
        d["gamma"], d["alpha"] = g.cpu().clone(), a.cpu().clone()
        outs.append(d)
    return outs


@pytest.mark.parametrize("name,B", [("c3", None), ("c2", None), ("multi", 2600)])
def test_round_equals_the_three_calls(name, B):
    """spec_verify_round gives bit for bit the results of spec_verify, spec_compact and
    spec_choose_gamma called one after another (also with more requests than one compaction
    pass and with stop tokens / budgets)."""
    if B is None:
        wl, kw = W.WORKLOADS[name], {}
    else:
        wl = W.Workload("t", B=B, V=64, dtype=torch.float32, temperature=1.0, logits="normal", sigma=1.0,
                        draft_sigma=0.2, K="uniform:0:40")
        rng = np.random.default_rng(4)
        kw = {"stop_token": torch.as_tensor(rng.integers(-1, 64, B).astype(np.int32), device="cuda"),
              "max_new": torch.as_tensor(rng.integers(0, 30, B).astype(np.int32), device="cuda")}
    sep, fused = _round_case(wl, 5, **kw)
    assert sep.keys() == fused.keys()
    # the packed arrays hold out_off[B] tokens and kv_off[B] KV pairs; the rest is not written
    n_out, n_kv = int(sep["c_out_off"][-1]), int(sep["c_kv_off"][-1])
    assert n_out == int(fused["c_out_off"][-1]) and n_kv == int(fused["c_kv_off"][-1])
    cut = {"c_packed_tokens": n_out, "c_packed_pos": n_out, "c_kv_src": n_kv, "c_kv_dst": n_kv}
    for k in sep:
        a, b = sep[k], fused[k]
        if k in cut:
            a, b = a[:cut[k]], b[:cut[k]]
        if a.is_floating_point():
            assert torch.equal(torch.nan_to_num(a, nan=-7.0), torch.nan_to_num(b, nan=-7.0)), k
        else:
            assert torch.equal(a, b), k
