"""spec_verify_noalloc: the verifier entry point for callers that cannot allocate device memory.

Such callers (a serving engine whose memory planner owns all device memory, a plugin running
inside another runtime's callbacks) pass inputs and outputs but no workspace; the library
uses a fixed scratch array of its own. This test calls that entry point through the C ABI
and checks it against spec_verify with a caller-supplied workspace, on two calls in a row with
different rounds (the scratch keeps the previous call's contents, which must not matter).
It is collected last and needs nothing from the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _round(seed, rnd):
    from speculative_decoding_verification_43_gb300 import workloads as W
    wl = W.scaled(W.WORKLOADS["c3"], B=48, V=32768)
    return W.make_round(wl, seed=seed, rnd=rnd, device="cuda")


def _run_noalloc(lib, v, stream):
    rc = lib.lib.spec_verify_noalloc(ctypes.byref(v.args), ctypes.c_void_p(stream.cuda_stream))
    lib.check(rc, "spec_verify_noalloc")


def test_noalloc_matches_workspace_entry_point_twice():
    from speculative_decoding_verification_43_gb300 import _lib, api
    stream = torch.cuda.current_stream()
    for rnd in (0, 1):
        rd = _round(seed=21, rnd=rnd)
        ref = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, diagnostics=True)
        ref.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
        ref.run(stream)
        # same arguments, outputs in fresh buffers, no workspace
        nal = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, diagnostics=True)
        nal.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
        for name in ("accept_len", "out_tokens", "req_status", "n_emitted"):
            getattr(nal.out, name).fill_(-7)
        _run_noalloc(_lib, nal, stream)
        torch.cuda.synchronize()
        for name in ("accept_len", "n_emitted", "out_tokens", "req_status", "fallback"):
            np.testing.assert_array_equal(getattr(nal.out, name).cpu().numpy(),
                                          getattr(ref.out, name).cpu().numpy(), err_msg=name)
        for name in ("alpha_rows", "rho_rows", "frontier_prob"):
            np.testing.assert_allclose(getattr(nal.out, name).cpu().numpy(),
                                       getattr(ref.out, name).cpu().numpy(), rtol=1e-5, err_msg=name)
        np.testing.assert_allclose(nal.out.alpha_sum.cpu().numpy(), ref.out.alpha_sum.cpu().numpy(), rtol=1e-12)
        assert int(nal.out.alpha_count.item()) == int(ref.out.alpha_count.item())


def test_noalloc_at_its_row_limit():
    """Exactly the largest batch the fixed scratch takes (16384 target rows, here 2048 requests of
    seven drafts over a 2048-token vocabulary): accepted, and equal to the workspace entry point."""
    from speculative_decoding_verification_43_gb300 import _lib, api
    from speculative_decoding_verification_43_gb300 import workloads as W
    wl = W.Workload("limit", B=2048, V=2048, dtype=torch.bfloat16, temperature=0.9, logits="normal",
                    sigma=2.0, draft_sigma=0.6, K="fixed:7")
    rd = W.make_round(wl, seed=5, rnd=0, device="cuda")
    assert rd.T == _lib.NOALLOC_MAX_ROWS == 16384
    stream = torch.cuda.current_stream()
    ref = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, diagnostics=True)
    ref.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
    ref.run(stream)
    nal = api.Verifier(rd.B, rd.target.shape[1], rd.T, rd.target.dtype, diagnostics=True)
    nal.bind(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
    for name in ("accept_len", "out_tokens", "req_status", "n_emitted"):
        getattr(nal.out, name).fill_(-7)
    _run_noalloc(_lib, nal, stream)
    torch.cuda.synchronize()
    assert (ref.out.req_status == 0).all()
    for name in ("accept_len", "n_emitted", "out_tokens", "req_status", "fallback"):
        np.testing.assert_array_equal(getattr(nal.out, name).cpu().numpy(),
                                      getattr(ref.out, name).cpu().numpy(), err_msg=name)
    np.testing.assert_array_equal(nal.out.alpha_rows.cpu().numpy(), ref.out.alpha_rows.cpu().numpy())
    assert int(nal.out.alpha_count.item()) == int(ref.out.alpha_count.item()) == rd.T - rd.B


def test_noalloc_rejects_batches_beyond_its_scratch():
    from speculative_decoding_verification_43_gb300 import _lib, api
    T = _lib.NOALLOC_MAX_ROWS + 1
    B = T // 2 + 1
    v = api.Verifier(B, 1024, T, torch.bfloat16)
    rc = _lib.lib.spec_verify_noalloc(ctypes.byref(v.args), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.SPEC_ERR_UNSUPPORTED
