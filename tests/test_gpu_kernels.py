"""GPU: the verifier's kernel and its grid, and spec_verify_round against the three calls.

spec_verify launches four kernels: spec_stats_kernel (pass 1, a persistent grid that fills every
SM), spec_decide_kernel (decisions and each request's frontier), spec_pass2_kernel (pass 2) and
spec_finish_kernel (draws, selection). These tests check the plan the library reports, that a
workspace serves many calls of different shapes in a row (the statistics kernel zeroes the later
kernels' counters), and that the fused round equals the three calls.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_43_gb300 import api
from speculative_decoding_verification_43_gb300 import workloads as W

import test_gpu_parity as G

pytestmark = pytest.mark.gpu


def test_plan_of_the_workloads():
    """Every workload's statistics kernel runs a persistent grid with the same number of CTAs on
    every SM of the device."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for name in ("c1", "c2", "c3", "c4", "c5"):
        wl = W.WORKLOADS[name]
        rows = W.make_round(wl, seed=0, rnd=0, device="cuda").T
        kern, c, n = api.verify_plan(wl.B, wl.V, rows, wl.dtype)
        assert kern == "spec_stats_kernel" and c == 1, (name, kern, c, n)
        assert n >= sms and n % sms == 0, (name, n, sms)


def test_invalid_shapes_have_no_plan():
    assert api.verify_plan(0, 1000, 10, torch.float32) is None
    assert api.verify_plan(4, 1001, 10, torch.bfloat16) is None  # a row of 2002 bytes
    assert api.verify_plan(8, 1024, 7, torch.float32) is None    # fewer rows than requests


def test_one_workspace_serves_many_calls():
    """Rounds of different shapes through one workspace, sized for the largest: the layout of
    each call differs from the previous one's, and no call reads what an earlier one left."""
    big = W.scaled(W.WORKLOADS["c3"], B=24, V=32768)
    rd0 = W.make_round(big, seed=4, rnd=0, device="cuda")
    v = api.Verifier(rd0.B, rd0.target.shape[1], rd0.T, rd0.target.dtype, diagnostics=True)
    ws = v.workspace
    for rnd in range(6):
        rd = W.make_round(big, seed=4, rnd=rnd, device="cuda")
        if rd.T > rd0.T:
            continue
        w = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, diagnostics=True)
        assert w.ws_bytes <= ws.numel()
        w.workspace = ws
        w.ws_bytes = ws.numel()
        w.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
        w.run()
        fresh = api.verify(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature,
                           diagnostics=True)
        torch.cuda.synchronize()
        for k in ("accept_len", "n_emitted", "out_tokens", "req_status"):
            assert torch.equal(getattr(w.out, k), getattr(fresh, k)), (rnd, k)
        assert torch.equal(w.out.alpha_rows, fresh.alpha_rows), rnd
        G.assert_report(G.check_round(rd), max_near=1, name=f"workspace reuse #{rnd}")  # oracle: 0 each


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
