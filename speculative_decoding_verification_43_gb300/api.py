"""Python binding of the C ABI: argument marshalling only.

Every step of the verifier runs in the CUDA kernels of libspecverify.so. PyTorch supplies
device memory and the stream; this module fills the C structs with tensor pointers, allocates
output tensors on request, and raises when a call returns an error status.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import SpecCompactArgs, SpecVerifyArgs, check, lib

_DTYPE = {torch.float32: _lib.SPEC_F32, torch.bfloat16: _lib.SPEC_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _i32(t):
    assert t.dtype == torch.int32 and t.is_contiguous() and t.is_cuda, "int32 CUDA tensor expected"
    return t


def workspace_size(B: int, V: int, total_rows: int, dtype: torch.dtype) -> int:
    return int(lib.spec_verify_workspace_size(B, V, total_rows, _DTYPE[dtype]))


def verify_plan(B: int, V: int, total_rows: int, dtype: torch.dtype):
    """(kernel name, CTAs per cluster, CTAs) that spec_verify launches for this shape on the
    current device, or None when the device cannot host it (or the shape is invalid)."""
    c, n = ctypes.c_int32(0), ctypes.c_int32(0)
    name = lib.spec_verify_plan(B, V, total_rows, _DTYPE[dtype], ctypes.byref(c), ctypes.byref(n))
    return None if name is None else (name.decode(), c.value, n.value)


@dataclass
class VerifyOutputs:
    accept_len: torch.Tensor
    n_emitted: torch.Tensor
    out_tokens: torch.Tensor
    req_status: torch.Tensor
    alpha_rows: torch.Tensor
    alpha_sum: torch.Tensor
    alpha_count: torch.Tensor
    rho_rows: torch.Tensor | None = None
    resid_rows: torch.Tensor | None = None
    frontier_prob: torch.Tensor | None = None
    frontier_margin: torch.Tensor | None = None
    fallback: torch.Tensor | None = None
    depth_reached: torch.Tensor | None = None   # [K_max] requests that reached depth j
    depth_accepted: torch.Tensor | None = None  # [K_max] requests that accepted depth j


class Verifier:
    """A prepared spec_verify call for one batch shape.

    Holds the C struct, the workspace and the output tensors, so that repeated rounds on the
    same buffers cost one ctypes call each. Inputs are bound with ``bind``; ``run`` enqueues
    the verifier's kernel on the given (or current) stream and returns without synchronising.
    The workspace is zero-filled once, here: every call leaves it ready for the next one.
    """

    def __init__(self, B: int, V: int, total_rows: int, dtype: torch.dtype, *, K_max: int = 64,
                 device=None, diagnostics: bool = False):
        device = torch.device(device or "cuda")
        self.B, self.V, self.T, self.dtype, self.K_max = B, V, total_rows, dtype, K_max
        nd = max(total_rows - B, 1)
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.out = VerifyOutputs(
            accept_len=torch.empty(B, **i32), n_emitted=torch.empty(B, **i32),
            out_tokens=torch.empty(total_rows, **i32), req_status=torch.empty(B, **i32),
            alpha_rows=torch.empty(nd, **f32),
            alpha_sum=torch.empty(1, dtype=torch.float64, device=device),
            alpha_count=torch.empty(1, **i32),
            depth_reached=torch.empty(max(K_max, 1), **i32), depth_accepted=torch.empty(max(K_max, 1), **i32))
        if diagnostics:
            self.out.rho_rows = torch.empty(nd, **f32)
            self.out.resid_rows = torch.empty(nd, **f32)
            self.out.frontier_prob = torch.empty(B, **f32)
            self.out.frontier_margin = torch.empty(B, **f32)
            self.out.fallback = torch.empty(B, **i32)
        self.ws_bytes = workspace_size(B, V, total_rows, dtype)
        # 256-byte aligned (the caching allocator hands out 512-byte aligned blocks) and zeroed
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.args = SpecVerifyArgs()
        a = self.args
        a.B, a.V, a.K_max, a.total_rows, a.dtype = B, V, K_max, total_rows, _DTYPE[dtype]
        o = self.out
        for name in ("accept_len", "n_emitted", "out_tokens", "req_status", "alpha_rows", "alpha_sum",
                     "alpha_count", "rho_rows", "resid_rows", "frontier_prob", "frontier_margin",
                     "fallback", "depth_reached", "depth_accepted"):
            setattr(a, name, _ptr(getattr(o, name)))
        self._keep = ()

    def bind(self, target, draft, row_off, draft_tokens, uniforms, temperature=1.0, *,
             stop_token=None, max_new=None, top_k=None, top_p=None):
        B, V, T = self.B, self.V, self.T
        assert target.dtype == self.dtype and target.is_cuda and target.is_contiguous()
        assert target.shape == (T, V), (target.shape, (T, V))
        if T > B:
            assert draft is not None and draft.dtype == self.dtype and draft.is_contiguous()
            assert draft.shape == (T - B, V)
            _i32(draft_tokens)
        _i32(row_off)
        assert row_off.shape == (B + 1,)
        assert uniforms.dtype == torch.float64 and uniforms.is_cuda and uniforms.numel() >= T
        a = self.args
        a.target_logits = _ptr(target)
        a.draft_logits = _ptr(draft) if T > B else None
        a.row_off = _ptr(row_off)
        a.draft_tokens = _ptr(draft_tokens) if T > B else None
        a.uniforms = _ptr(uniforms)
        if isinstance(temperature, torch.Tensor):
            assert temperature.dtype == torch.float32 and temperature.is_cuda and temperature.numel() == B
            a.temperature = _ptr(temperature)
            a.temperature_scalar = 1.0
        else:
            a.temperature = None
            a.temperature_scalar = float(temperature)
        a.stop_token = _ptr(_i32(stop_token)) if stop_token is not None else None
        a.max_new = _ptr(_i32(max_new)) if max_new is not None else None
        # top-k / top-p of the target law, per request (None: no truncation)
        if top_p is not None:
            assert top_p.dtype == torch.float32 and top_p.is_cuda and top_p.numel() == B
        a.top_k = _ptr(_i32(top_k)) if top_k is not None else None
        a.top_p = _ptr(top_p) if top_p is not None else None
        self._keep = (target, draft, row_off, draft_tokens, uniforms, temperature, stop_token, max_new,
                      top_k, top_p)
        return self

    def time_rows_with(self, begin, end, stats_end=None):
        """On each following run, record torch.cuda.Event `begin` before the verifier's first
        kernel, `end` after its last and `stats_end` after the statistics kernel (each may be
        None; all None: stop)."""
        ev = lambda e: ctypes.c_void_p(e.cuda_event) if e is not None else None  # noqa: E731
        self.args.rows_event_begin = ev(begin)
        self.args.rows_event_end = ev(end)
        self.args.stats_event_end = ev(stats_end)
        self._events = (begin, end, stats_end)

    def run(self, stream=None) -> VerifyOutputs:
        rc = lib.spec_verify(ctypes.byref(self.args), ctypes.c_void_p(self.workspace.data_ptr()),
                             self.ws_bytes, _stream_handle(stream))
        check(rc, "spec_verify")
        return self.out


def verify(target, draft, row_off, draft_tokens, uniforms, temperature=1.0, *, K_max: int = 64,
           stop_token=None, max_new=None, top_k=None, top_p=None, diagnostics: bool = False,
           stream=None) -> VerifyOutputs:
    """One verifier round on device tensors (see include/spec_verify.h for the layout)."""
    T, V = target.shape
    B = row_off.numel() - 1
    v = Verifier(B, V, T, target.dtype, K_max=K_max, device=target.device, diagnostics=diagnostics)
    v.bind(target, draft, row_off, draft_tokens, uniforms, temperature, stop_token=stop_token,
           max_new=max_new, top_k=top_k, top_p=top_p)
    return v.run(stream)


@dataclass
class CompactOutputs:
    out_off: torch.Tensor
    packed_tokens: torch.Tensor
    packed_pos: torch.Tensor
    kv_off: torch.Tensor
    kv_src: torch.Tensor
    kv_dst: torch.Tensor
    new_seq_len: torch.Tensor
    new_kv_len: torch.Tensor
    new_draft_len: torch.Tensor
    compact_status: torch.Tensor


class Compactor:
    """A prepared spec_compact call for one batch shape."""

    def __init__(self, B: int, total_rows: int, device=None):
        device = torch.device(device or "cuda")
        i32 = dict(dtype=torch.int32, device=device)
        nd = max(total_rows - B, 1)
        self.B, self.T = B, total_rows
        self.out = CompactOutputs(
            out_off=torch.empty(B + 1, **i32), packed_tokens=torch.empty(total_rows, **i32),
            packed_pos=torch.empty(total_rows, **i32), kv_off=torch.empty(B + 1, **i32),
            kv_src=torch.empty(nd, **i32), kv_dst=torch.empty(nd, **i32),
            new_seq_len=torch.empty(B, **i32), new_kv_len=torch.empty(B, **i32),
            new_draft_len=torch.empty(B, **i32), compact_status=torch.empty(B, **i32))
        self.args = SpecCompactArgs()
        a = self.args
        a.B, a.total_rows = B, total_rows
        for name in ("out_off", "packed_tokens", "packed_pos", "kv_off", "kv_src", "kv_dst",
                     "new_seq_len", "new_kv_len", "new_draft_len", "compact_status"):
            setattr(a, name, _ptr(getattr(self.out, name)))
        self._keep = ()

    def bind(self, row_off, accept_len, n_emitted, out_tokens, req_status, prefix_len, cand_kv_rows,
             block_table, page_size: int):
        a = self.args
        assert block_table.dim() == 2 and block_table.shape[0] == self.B
        a.page_size = int(page_size)
        a.max_blocks = int(block_table.shape[1])
        for name, t in (("row_off", row_off), ("accept_len", accept_len), ("n_emitted", n_emitted),
                        ("out_tokens", out_tokens), ("req_status", req_status),
                        ("prefix_len", prefix_len), ("cand_kv_rows", cand_kv_rows),
                        ("block_table", block_table)):
            setattr(a, name, _ptr(_i32(t)) if t is not None else None)
        self._keep = (row_off, accept_len, n_emitted, out_tokens, req_status, prefix_len,
                      cand_kv_rows, block_table)
        return self

    def run(self, stream=None) -> CompactOutputs:
        check(lib.spec_compact(ctypes.byref(self.args), _stream_handle(stream)), "spec_compact")
        return self.out


def compact(row_off, accept_len, n_emitted, out_tokens, req_status, prefix_len, cand_kv_rows,
            block_table, page_size: int, stream=None) -> CompactOutputs:
    c = Compactor(row_off.numel() - 1, out_tokens.numel(), device=out_tokens.device)
    c.bind(row_off, accept_len, n_emitted, out_tokens, req_status, prefix_len, cand_kv_rows,
           block_table, page_size)
    return c.run(stream)


def run_round(verifier: "Verifier", compactor: "Compactor", alpha_prev: float, c: float, gamma_min: int = 0,
              gamma_max: int = 8, *, out=None, stream=None):
    """One round through spec_verify_round: the bound verifier, the bound compactor and the gamma
    choice in one call (the same results as verifier.run(), compactor.run() and choose_gamma()).
    Returns (verify outputs, compaction outputs, (gamma int32[1], alpha float64[1]))."""
    dev = verifier.out.alpha_sum.device
    if out is None:
        out = (torch.empty(1, dtype=torch.int32, device=dev), torch.empty(1, dtype=torch.float64, device=dev))
    g, a = out
    rc = lib.spec_verify_round(ctypes.byref(verifier.args), ctypes.c_void_p(verifier.workspace.data_ptr()),
                               verifier.ws_bytes, ctypes.byref(compactor.args), float(alpha_prev), float(c),
                               int(gamma_min), int(gamma_max), _ptr(g), _ptr(a), _stream_handle(stream))
    check(rc, "spec_verify_round")
    return verifier.out, compactor.out, (g, a)


def choose_gamma(alpha_sum, alpha_count, alpha_prev: float, c: float, gamma_min: int = 0,
                 gamma_max: int = 8, *, out=None, stream=None):
    """Device-side gamma choice; returns (gamma int32[1], alpha float64[1]) device tensors."""
    dev = alpha_sum.device
    if out is None:
        out = (torch.empty(1, dtype=torch.int32, device=dev), torch.empty(1, dtype=torch.float64, device=dev))
    g, a = out
    rc = lib.spec_choose_gamma(_ptr(alpha_sum), _ptr(alpha_count), float(alpha_prev), float(c),
                               int(gamma_min), int(gamma_max), _ptr(g), _ptr(a), _stream_handle(stream))
    check(rc, "spec_choose_gamma")
    return g, a


def choose_gamma_depth(depth_reached, depth_accepted, alpha_prev: float, c: float, gamma_min: int = 0,
                       gamma_max: int = 8, *, out=None, stream=None):
    """Device-side gamma choice from per-depth counts (as spec_verify writes them); returns
    (gamma int32[1], E[A] float64[1]) device tensors."""
    dev = depth_reached.device
    _i32(depth_reached)
    _i32(depth_accepted)
    assert depth_reached.numel() == depth_accepted.numel()
    if out is None:
        out = (torch.empty(1, dtype=torch.int32, device=dev), torch.empty(1, dtype=torch.float64, device=dev))
    g, ea = out
    rc = lib.spec_choose_gamma_depth(_ptr(depth_reached), _ptr(depth_accepted), int(depth_reached.numel()),
                                     float(alpha_prev), float(c), int(gamma_min), int(gamma_max), _ptr(g),
                                     _ptr(ea), _stream_handle(stream))
    check(rc, "spec_choose_gamma_depth")
    return g, ea


def depth_objective(n_reached, n_accepted, alpha_prev: float, c: float, gamma: int) -> float:
    """Host evaluation (double) of the depth-aware objective from host integer arrays."""
    import numpy as np
    nr = np.ascontiguousarray(n_reached, np.int32)
    na = np.ascontiguousarray(n_accepted, np.int32)
    assert nr.shape == na.shape
    return float(lib.spec_depth_objective(nr.ctypes.data_as(ctypes.c_void_p), na.ctypes.data_as(ctypes.c_void_p),
                                          int(nr.size), float(alpha_prev), float(c), int(gamma)))


def gamma_objective(alpha: float, c: float, gamma: int) -> float:
    return float(lib.spec_gamma_objective(float(alpha), float(c), int(gamma)))


def version() -> str:
    return lib.spec_version().decode()
