"""GPU: the index-checked debug build (libspecverify_debug.so, include/spec_debug.h).

The same sources compiled with -DSPEC_DEBUG check the index of each main global access of every
kernel against its array's length; a failed check records itself and skips the access instead of
trapping. On valid inputs no check may fail, and the results must equal the release library's bit
for bit (the checks change no arithmetic). The cases are small and span the shapes that stress
indexing: a vocabulary smaller than one vector per lane, partial chunks, K = 0 requests, the
largest K, greedy rows, top-k/top-p cuts, stop tokens and budgets, invalid requests, and the round
(compaction and gamma) through spec_verify_round. The parity of the results against the oracle is
checked as for the release library.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from speculative_decoding_verification_43_gb300 import _lib, api, build
from speculative_decoding_verification_43_gb300 import workloads as W

from parity import Report, compare, run_oracle

pytestmark = pytest.mark.gpu

FIELDS = ("accept_len", "n_emitted", "out_tokens", "req_status", "alpha_rows", "rho_rows", "resid_rows",
          "frontier_prob", "frontier_margin", "fallback", "alpha_sum", "alpha_count")


@pytest.fixture(scope="module")
def dbg():
    build.build()
    return _lib.load_library(build.DEBUG_LIB_PATH)


def fetch(dbg):
    words = np.zeros(4, np.uint32)
    assert dbg.spec_debug_fetch(words.ctypes.data_as(ctypes.c_void_p)) == _lib.SPEC_OK
    return words


def run_both(dbg, rd, **kw):
    """The same call through the release and the debug library, into separate outputs."""
    outs = []
    for which in ("release", "debug"):
        v = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, diagnostics=True)
        v.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature, **kw)
        if which == "release":
            v.run()
        else:
            stream = torch.cuda.current_stream()
            rc = dbg.spec_verify(ctypes.byref(v.args), ctypes.c_void_p(v.workspace.data_ptr()), v.ws_bytes,
                                 ctypes.c_void_p(stream.cuda_stream))
            _lib.check(rc, "spec_verify (debug build)")
        torch.cuda.synchronize()
        outs.append({k: getattr(v.out, k).cpu().numpy() for k in FIELDS})
    return outs


def same(a, b):
    for k in FIELDS:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


CASES = [
    ("f32 V=8", dict(B=9, V=8, dtype=torch.float32, temperature=0.9, logits="normal", sigma=2.0, draft_sigma=0.7,
                     K="uniform:0:3")),
    ("bf16 V=64", dict(B=7, V=64, dtype=torch.bfloat16, temperature=1.0, logits="normal", sigma=2.0, draft_sigma=0.5,
                       K="uniform:0:5")),
    ("bf16 V=1032", dict(B=12, V=1032, dtype=torch.bfloat16, temperature=0.7, logits="zipf", sigma=1.0,
                         draft_sigma=0.8, K="uniform:0:7")),
    ("f32 V=2052 K=64", dict(B=2, V=2052, dtype=torch.float32, temperature=1.0, logits="normal", sigma=1.0,
                             draft_sigma=0.2, K="fixed:64")),
]


@pytest.mark.parametrize("name,spec", CASES, ids=[c[0] for c in CASES])
def test_debug_build_matches_release_with_no_failed_check(dbg, name, spec):
    fetch(dbg)  # clear
    rd = W.make_round(W.Workload("t", **spec), seed=3, rnd=0, device="cuda")
    rel, deb = run_both(dbg, rd)
    same(rel, deb)
    words = fetch(dbg)
    assert words[3] == 0, (name, words)
    orc, sb, reqs = run_oracle(rd)
    rep = compare(deb, orc, sb, reqs, rd.row_off.cpu().numpy())
    assert rep.ok(), (rep.mismatches[:3], rep.value_failures[:3])


def test_debug_build_edge_inputs(dbg):
    """Greedy rows, top-k/top-p cuts, stop tokens and budgets, and invalid requests together."""
    fetch(dbg)
    base = W.Workload("t", B=16, V=520, dtype=torch.bfloat16, temperature=1.0, logits="normal", sigma=2.0,
                      draft_sigma=0.6, K="uniform:0:4")
    rd = W.make_round(base, seed=4, rnd=0, device="cuda")
    temp = rd.temperature.clone()
    temp[::5] = 0.0
    temp[7] = -1.0
    rd.temperature = temp
    ro = rd.row_off.cpu().numpy()
    rd.target[ro[3], 5] = float("nan")
    B = rd.B
    kw = dict(top_k=torch.as_tensor(np.array([0, 1, 3, 50, 600] * 4, np.int32)[:B], device="cuda"),
              top_p=torch.as_tensor(np.array([1.0, 0.9, 0.5, 0.0] * 4, np.float32)[:B], device="cuda"),
              stop_token=torch.full((B,), 7, dtype=torch.int32, device="cuda"),
              max_new=torch.as_tensor(np.array([1000, 1, 2, 0] * 4, np.int32)[:B], device="cuda"))
    rel, deb = run_both(dbg, rd, **kw)
    same(rel, deb)
    assert fetch(dbg)[3] == 0


def test_debug_build_round(dbg):
    """spec_verify_round (verify, compaction, gamma) through the debug build equals the release."""
    fetch(dbg)
    wl = W.Workload("t", B=24, V=1032, dtype=torch.bfloat16, temperature=0.8, logits="zipf", sigma=1.0,
                    draft_sigma=0.8, K="uniform:0:6")
    rd = W.make_round(wl, seed=6, rnd=0, device="cuda")
    ci = W.make_compaction_inputs(rd, 37, 16)
    res = []
    for which in ("release", "debug"):
        v = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, K_max=8)
        v.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
        c = api.Compactor(rd.B, rd.T)
        c.bind(rd.row_off, v.out.accept_len, v.out.n_emitted, v.out.out_tokens, v.out.req_status,
               ci["prefix_len"], ci["cand_kv_rows"], ci["block_table"], ci["page_size"])
        g = torch.empty(1, dtype=torch.int32, device="cuda")
        a = torch.empty(1, dtype=torch.float64, device="cuda")
        if which == "release":
            api.run_round(v, c, 0.5, 0.05, 0, 8, out=(g, a))
        else:
            stream = torch.cuda.current_stream()
            rc = dbg.spec_verify_round(ctypes.byref(v.args), ctypes.c_void_p(v.workspace.data_ptr()), v.ws_bytes,
                                       ctypes.byref(c.args), 0.5, 0.05, 0, 8, ctypes.c_void_p(g.data_ptr()),
                                       ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
            _lib.check(rc, "spec_verify_round (debug build)")
        torch.cuda.synchronize()
        n_out, n_kv = int(c.out.out_off[-1].item()), int(c.out.kv_off[-1].item())
        res.append([t.cpu().numpy() for t in (v.out.accept_len, v.out.out_tokens, c.out.out_off, c.out.kv_off,
                                              c.out.packed_tokens[:n_out], c.out.packed_pos[:n_out],
                                              c.out.kv_src[:n_kv], c.out.kv_dst[:n_kv], c.out.new_seq_len, g, a)])
    for x, y in zip(*res):
        np.testing.assert_array_equal(x, y)
    assert fetch(dbg)[3] == 0
