"""ctypes view of the C ABI in include/spec_verify.h (libspecverify.so, built in-tree).

There is no fallback: if the library is missing or fails to load, importing this module
raises, and nothing in the package computes any part of the verifier on the CPU.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

_p = ctypes.c_void_p
_i32 = ctypes.c_int32

SPEC_F32 = 0
SPEC_BF16 = 1

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = -1
SPEC_ERR_WORKSPACE = -2
SPEC_ERR_CUDA = -3
SPEC_ERR_UNSUPPORTED = -4

REQ_BAD_PROPOSAL = 1
REQ_BAD_LOGITS = 2
REQ_BAD_SHAPE = 4
REQ_BAD_PARAM = 8
REQ_BAD_BLOCKS = 16
REQ_TIMEOUT = 32

NOALLOC_MAX_ROWS = 16384

STATUS_NAMES = {
    SPEC_OK: "SPEC_OK", SPEC_ERR_INVALID_ARG: "SPEC_ERR_INVALID_ARG",
    SPEC_ERR_WORKSPACE: "SPEC_ERR_WORKSPACE", SPEC_ERR_CUDA: "SPEC_ERR_CUDA",
    SPEC_ERR_UNSUPPORTED: "SPEC_ERR_UNSUPPORTED",
}


class SpecVerifyArgs(ctypes.Structure):
    _fields_ = [
        ("B", _i32), ("V", _i32), ("K_max", _i32), ("total_rows", _i32), ("dtype", ctypes.c_int),
        ("target_logits", _p), ("draft_logits", _p), ("row_off", _p), ("draft_tokens", _p),
        ("uniforms", _p), ("temperature", _p), ("temperature_scalar", ctypes.c_float),
        ("stop_token", _p), ("max_new", _p),
        ("accept_len", _p), ("n_emitted", _p), ("out_tokens", _p), ("req_status", _p),
        ("alpha_rows", _p), ("alpha_sum", _p), ("alpha_count", _p),
        ("rho_rows", _p), ("resid_rows", _p), ("frontier_prob", _p), ("frontier_margin", _p),
        ("fallback", _p), ("rows_event_begin", _p), ("rows_event_end", _p), ("stats_event_end", _p),
        ("depth_reached", _p), ("depth_accepted", _p),
        ("top_k", _p), ("top_p", _p),
    ]


class SpecCompactArgs(ctypes.Structure):
    _fields_ = [
        ("B", _i32), ("page_size", _i32), ("max_blocks", _i32), ("total_rows", _i32),
        ("row_off", _p), ("accept_len", _p), ("n_emitted", _p), ("out_tokens", _p),
        ("req_status", _p), ("prefix_len", _p), ("cand_kv_rows", _p), ("block_table", _p),
        ("out_off", _p), ("packed_tokens", _p), ("packed_pos", _p), ("kv_off", _p),
        ("kv_src", _p), ("kv_dst", _p), ("new_seq_len", _p), ("new_kv_len", _p),
        ("new_draft_len", _p), ("compact_status", _p),
    ]


# every symbol include/spec_verify.h declares
EXPORTS = ("spec_verify_workspace_size", "spec_verify", "spec_verify_noalloc", "spec_verify_plan",
           "spec_verify_round", "spec_compact",
           "spec_gamma_objective", "spec_choose_gamma", "spec_choose_gamma_depth", "spec_depth_objective",
           "spec_version")


def load_library(path: str):
    """The library at `path` (the release build, or the index-checked debug build) with the
    argument and result types of every call the header declares."""
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    lib.spec_verify_workspace_size.argtypes = [_i32, _i32, _i32, ctypes.c_int]
    lib.spec_verify_workspace_size.restype = ctypes.c_size_t
    lib.spec_verify.argtypes = [ctypes.POINTER(SpecVerifyArgs), _p, ctypes.c_size_t, _p]
    lib.spec_verify.restype = ctypes.c_int
    lib.spec_verify_noalloc.argtypes = [ctypes.POINTER(SpecVerifyArgs), _p]
    lib.spec_verify_noalloc.restype = ctypes.c_int
    lib.spec_verify_plan.argtypes = [_i32, _i32, _i32, ctypes.c_int, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
    lib.spec_verify_plan.restype = ctypes.c_char_p
    lib.spec_verify_round.argtypes = [ctypes.POINTER(SpecVerifyArgs), _p, ctypes.c_size_t,
                                      ctypes.POINTER(SpecCompactArgs), ctypes.c_double, ctypes.c_double, _i32, _i32,
                                      _p, _p, _p]
    lib.spec_verify_round.restype = ctypes.c_int
    lib.spec_compact.argtypes = [ctypes.POINTER(SpecCompactArgs), _p]
    lib.spec_compact.restype = ctypes.c_int
    lib.spec_gamma_objective.argtypes = [ctypes.c_double, ctypes.c_double, _i32]
    lib.spec_gamma_objective.restype = ctypes.c_double
    lib.spec_choose_gamma.argtypes = [_p, _p, ctypes.c_double, ctypes.c_double, _i32, _i32, _p, _p, _p]
    lib.spec_choose_gamma.restype = ctypes.c_int
    lib.spec_choose_gamma_depth.argtypes = [_p, _p, _i32, ctypes.c_double, ctypes.c_double, _i32, _i32, _p, _p, _p]
    lib.spec_choose_gamma_depth.restype = ctypes.c_int
    lib.spec_depth_objective.argtypes = [_p, _p, _i32, ctypes.c_double, ctypes.c_double, _i32]
    lib.spec_depth_objective.restype = ctypes.c_double
    lib.spec_version.argtypes = []
    lib.spec_version.restype = ctypes.c_char_p
    if hasattr(lib, "spec_debug_fetch"):  # the debug build (include/spec_debug.h)
        lib.spec_debug_fetch.argtypes = [_p]
        lib.spec_debug_fetch.restype = ctypes.c_int
    return lib


lib = load_library(LIB_PATH)


def check(rc: int, what: str) -> None:
    if rc != SPEC_OK:
        raise RuntimeError(f"{what} failed: {STATUS_NAMES.get(rc, rc)}")
