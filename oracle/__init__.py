"""Float64 CPU oracle for the batched speculative-decoding verifier.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline and reference arm may import this package. The product path never does: it shares
no code, header, helper or table with the CUDA library (``spec_oracle.c`` defines its own
structs and is compiled by ``gcc`` alone).

What the oracle computes, with the passages it follows, is in ``spec_oracle.h``. This module
only marshals numpy arrays into the C structs and back.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_HDR = os.path.join(_HERE, "spec_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, f"liboracle_{platform.machine()}.so")

REQ_BAD_PROPOSAL = 1
REQ_BAD_LOGITS = 2
REQ_BAD_SHAPE = 4
REQ_BAD_PARAM = 8
REQ_BAD_BLOCKS = 16

_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i32 = ctypes.c_int32


class _Batch(ctypes.Structure):
    _fields_ = [
        ("B", _i32), ("V", _i32), ("K_max", _i32), ("dtype", _i32),
        ("target", _p), ("draft", _p), ("row_off", _p), ("draft_tokens", _p),
        ("uniforms", _p), ("temperature", _p), ("stop_token", _p), ("max_new", _p),
        ("top_k", _p), ("top_p", _p),
    ]


class _Result(ctypes.Structure):
    _fields_ = [
        ("accept_len", _p), ("out_tokens", _p), ("n_emitted", _p), ("req_status", _p),
        ("alpha", _p), ("rho", _p), ("resid_mass", _p), ("accept_margin", _p),
        ("sample_margin", _p), ("sample_prob", _p), ("fallback", _p),
        ("trunc_margin", _p), ("trunc_keep", _p), ("resid_scale", _p), ("sample_cond", _p),
    ]


class _Compact(ctypes.Structure):
    _fields_ = [
        ("B", _i32), ("page_size", _i32), ("max_blocks", _i32),
        ("row_off", _p), ("accept_len", _p), ("n_emitted", _p), ("out_tokens", _p),
        ("req_status", _p), ("prefix_len", _p), ("cand_kv_rows", _p), ("block_table", _p),
        ("out_off", _p), ("packed_tokens", _p), ("packed_pos", _p), ("kv_off", _p),
        ("kv_src", _p), ("kv_dst", _p), ("new_seq_len", _p), ("new_kv_len", _p),
        ("new_draft_len", _p), ("compact_status", _p),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, no target-specific flags), with OpenMP for
    ``oracle_verify_threads`` where the compiler has it (else that entry runs serially)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                      os.path.getmtime(_HDR)))
        if force or stale:
            os.makedirs(_BUILD, exist_ok=True)
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            try:
                subprocess.check_call(cmd[:1] + ["-fopenmp"] + cmd[1:], stderr=subprocess.DEVNULL)
            except subprocess.CalledProcessError:
                subprocess.check_call(cmd)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_verify.argtypes = [ctypes.POINTER(_Batch), ctypes.POINTER(_Result)]
        lib.oracle_verify.restype = ctypes.c_int
        lib.oracle_verify_threads.argtypes = [ctypes.POINTER(_Batch), ctypes.POINTER(_Result), _i32]
        lib.oracle_verify_threads.restype = ctypes.c_int
        lib.oracle_compact.argtypes = [ctypes.POINTER(_Compact)]
        lib.oracle_compact.restype = ctypes.c_int
        lib.oracle_gamma_objective.argtypes = [ctypes.c_double, ctypes.c_double, _i32]
        lib.oracle_gamma_objective.restype = ctypes.c_double
        lib.oracle_choose_gamma.argtypes = [ctypes.c_double, _i32, ctypes.c_double,
                                            ctypes.c_double, _i32, _i32,
                                            ctypes.POINTER(ctypes.c_double)]
        lib.oracle_choose_gamma.restype = _i32
        _vp = ctypes.c_void_p
        lib.oracle_depth_counts.argtypes = [_i32, _vp, _vp, _vp, _i32, _vp, _vp]
        lib.oracle_depth_counts.restype = None
        lib.oracle_depth_alpha.argtypes = [_vp, _vp, _i32, ctypes.c_double, _i32, _vp]
        lib.oracle_depth_alpha.restype = None
        lib.oracle_depth_expected_accept.argtypes = [_vp, _vp, _i32, ctypes.c_double, _i32]
        lib.oracle_depth_expected_accept.restype = ctypes.c_double
        lib.oracle_depth_objective.argtypes = [_vp, _vp, _i32, ctypes.c_double, ctypes.c_double, _i32]
        lib.oracle_depth_objective.restype = ctypes.c_double
        lib.oracle_choose_gamma_depth.argtypes = [_vp, _vp, _i32, ctypes.c_double, ctypes.c_double,
                                                  _i32, _i32, ctypes.POINTER(ctypes.c_double)]
        lib.oracle_choose_gamma_depth.restype = _i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def verify(target, draft, row_off, draft_tokens, uniforms, temperature, *, V=None,
           K_max=64, stop_token=None, max_new=None, top_k=None, top_p=None, threads=None):
    """Run the verifier on host arrays.

    ``target``/``draft`` are 2-D float32 arrays, or uint16 arrays holding bfloat16 bits.
    Returns a dict of numpy arrays named like the fields of ``oracle_result``. With
    ``threads=n`` the requests are split over up to n OpenMP threads (same results); the dict
    then also holds ``threads_used``.
    """
    lib = _load()
    bf16 = target.dtype == np.uint16
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    if not bf16:
        target = target.astype(np.float32, copy=False)
        draft = draft.astype(np.float32, copy=False)
    row_off = _c(row_off, np.int32)
    B = row_off.shape[0] - 1
    T = int(row_off[-1])
    V = int(target.shape[1]) if V is None else V
    nd = T - B
    draft_tokens = _c(draft_tokens, np.int32)
    uniforms = _c(uniforms, np.float64)
    temperature = _c(np.broadcast_to(np.asarray(temperature, np.float32), (B,)), np.float32)
    stop_token = _c(stop_token, np.int32)
    max_new = _c(max_new, np.int32)
    top_k = None if top_k is None else _c(np.broadcast_to(np.asarray(top_k, np.int32), (B,)), np.int32)
    top_p = None if top_p is None else _c(np.broadcast_to(np.asarray(top_p, np.float32), (B,)), np.float32)
    assert uniforms.shape[0] >= T and draft_tokens.shape[0] >= nd

    out = {
        "accept_len": np.zeros(B, np.int32), "out_tokens": np.full(T, -1, np.int32),
        "n_emitted": np.zeros(B, np.int32), "req_status": np.zeros(B, np.int32),
        "alpha": np.zeros(nd, np.float64), "rho": np.zeros(nd, np.float64),
        "resid_mass": np.zeros(nd, np.float64), "accept_margin": np.zeros(nd, np.float64),
        "sample_margin": np.zeros(B, np.float64), "sample_prob": np.zeros(B, np.float64),
        "fallback": np.zeros(B, np.int32),
        "trunc_margin": np.full(T, np.nan, np.float64), "trunc_keep": np.full(T, V, np.int32),
        "resid_scale": np.zeros(nd, np.float64), "sample_cond": np.zeros(B, np.float64),
    }
    b = _Batch(B, V, K_max, 1 if bf16 else 0, _ptr(target), _ptr(draft), _ptr(row_off),
               _ptr(draft_tokens), _ptr(uniforms), _ptr(temperature), _ptr(stop_token),
               _ptr(max_new), _ptr(top_k), _ptr(top_p))
    r = _Result(*[_ptr(out[f]) for f, _ in _Result._fields_])
    if threads is None:
        rc = lib.oracle_verify(ctypes.byref(b), ctypes.byref(r))
        if rc != 0:
            raise RuntimeError(f"oracle_verify failed: {rc}")
    else:
        rc = lib.oracle_verify_threads(ctypes.byref(b), ctypes.byref(r), int(threads))
        if rc < 1:
            raise RuntimeError(f"oracle_verify_threads failed: {rc}")
        out["threads_used"] = rc
    return out


def compact(row_off, accept_len, n_emitted, out_tokens, req_status, prefix_len, cand_kv_rows,
            block_table, page_size):
    lib = _load()
    row_off = _c(row_off, np.int32)
    B = row_off.shape[0] - 1
    T = int(row_off[-1])
    block_table = _c(block_table, np.int32)
    max_blocks = int(block_table.shape[1]) if block_table.ndim == 2 else int(block_table.size // max(B, 1))
    args = {k: _c(v, np.int32) for k, v in dict(
        accept_len=accept_len, n_emitted=n_emitted, out_tokens=out_tokens, req_status=req_status,
        prefix_len=prefix_len, cand_kv_rows=cand_kv_rows).items()}
    out = {
        "out_off": np.zeros(B + 1, np.int32), "packed_tokens": np.full(T, -1, np.int32),
        "packed_pos": np.full(T, -1, np.int32), "kv_off": np.zeros(B + 1, np.int32),
        "kv_src": np.full(max(T - B, 0), -1, np.int32), "kv_dst": np.full(max(T - B, 0), -1, np.int32),
        "new_seq_len": np.zeros(B, np.int32), "new_kv_len": np.zeros(B, np.int32),
        "new_draft_len": np.zeros(B, np.int32), "compact_status": np.zeros(B, np.int32),
    }
    c = _Compact(B, page_size, max_blocks, _ptr(row_off), _ptr(args["accept_len"]),
                 _ptr(args["n_emitted"]), _ptr(args["out_tokens"]), _ptr(args["req_status"]),
                 _ptr(args["prefix_len"]), _ptr(args["cand_kv_rows"]), _ptr(block_table),
                 *[_ptr(out[k]) for k in ("out_off", "packed_tokens", "packed_pos", "kv_off",
                                          "kv_src", "kv_dst", "new_seq_len", "new_kv_len",
                                          "new_draft_len", "compact_status")])
    rc = lib.oracle_compact(ctypes.byref(c))
    if rc != 0:
        raise RuntimeError(f"oracle_compact failed: {rc}")
    n_out = int(out["out_off"][-1])
    n_kv = int(out["kv_off"][-1])
    for k in ("packed_tokens", "packed_pos"):
        out[k] = out[k][:n_out]
    for k in ("kv_src", "kv_dst"):
        out[k] = out[k][:n_kv]
    return out


def gamma_objective(alpha: float, c: float, gamma: int) -> float:
    return float(_load().oracle_gamma_objective(float(alpha), float(c), int(gamma)))


def choose_gamma(alpha_sum: float, alpha_count: int, alpha_prev: float, c: float,
                 gamma_min: int = 0, gamma_max: int = 8):
    a = ctypes.c_double(0.0)
    g = _load().oracle_choose_gamma(float(alpha_sum), int(alpha_count), float(alpha_prev),
                                    float(c), int(gamma_min), int(gamma_max), ctypes.byref(a))
    return int(g), float(a.value)


def depth_counts(row_off, accept_len, req_status, depth_max: int):
    """Per-depth counts of requests that reached / accepted depth j = 1..depth_max."""
    ro, al, rs = _c(row_off, np.int32), _c(accept_len, np.int32), _c(req_status, np.int32)
    nr = np.zeros(depth_max, np.int32)
    na = np.zeros(depth_max, np.int32)
    _load().oracle_depth_counts(len(al), _ptr(ro), _ptr(al), _ptr(rs), int(depth_max), _ptr(nr), _ptr(na))
    return nr, na


def depth_alpha(n_reached, n_accepted, alpha_prev: float, n_out: int):
    nr, na = _c(n_reached, np.int32), _c(n_accepted, np.int32)
    out = np.zeros(n_out, np.float64)
    _load().oracle_depth_alpha(_ptr(nr), _ptr(na), len(nr), float(alpha_prev), int(n_out), _ptr(out))
    return out


def depth_expected_accept(n_reached, n_accepted, alpha_prev: float, gamma: int) -> float:
    nr, na = _c(n_reached, np.int32), _c(n_accepted, np.int32)
    return float(_load().oracle_depth_expected_accept(_ptr(nr), _ptr(na), len(nr), float(alpha_prev), int(gamma)))


def depth_objective(n_reached, n_accepted, alpha_prev: float, c: float, gamma: int) -> float:
    nr, na = _c(n_reached, np.int32), _c(n_accepted, np.int32)
    return float(_load().oracle_depth_objective(_ptr(nr), _ptr(na), len(nr), float(alpha_prev), float(c),
                                                int(gamma)))


def choose_gamma_depth(n_reached, n_accepted, alpha_prev: float, c: float, gamma_min: int = 0,
                       gamma_max: int = 8):
    nr, na = _c(n_reached, np.int32), _c(n_accepted, np.int32)
    ea = ctypes.c_double(0.0)
    g = _load().oracle_choose_gamma_depth(_ptr(nr), _ptr(na), len(nr), float(alpha_prev), float(c),
                                          int(gamma_min), int(gamma_max), ctypes.byref(ea))
    return int(g), float(ea.value)
