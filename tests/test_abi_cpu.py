"""CPU checks of the C ABI: the library loads, exports every declared symbol, and rejects bad
host arguments before touching the GPU. Also the host-side gamma objective and the seeded
input generators. No compute call here needs a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_43_gb300 import build
    build.build()
    from speculative_decoding_verification_43_gb300 import _lib
    return _lib


def declared_functions(header="spec_verify.h"):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(lib.EXPORTS), names
    raw = ctypes.CDLL(lib.LIB_PATH if hasattr(lib, "LIB_PATH") else lib.lib._name)
    for n in names:
        assert hasattr(raw, n), n


def test_debug_library_exports_everything_plus_its_fetch(lib):
    """libspecverify_debug.so (the -DSPEC_DEBUG build) exports every symbol of spec_verify.h and
    the one spec_debug.h adds; the release library does not export the debug call."""
    from speculative_decoding_verification_43_gb300 import build
    dbg = ctypes.CDLL(build.DEBUG_LIB_PATH)
    extra = declared_functions("spec_debug.h")
    assert extra == ["spec_debug_fetch"], extra
    for n in declared_functions() + extra:
        assert hasattr(dbg, n), n
    assert not hasattr(ctypes.CDLL(build.LIB_PATH), "spec_debug_fetch")
    dbg.spec_version.restype = ctypes.c_char_p
    assert b"debug" in dbg.spec_version()
    dbg.spec_debug_fetch.argtypes = [ctypes.c_void_p]
    dbg.spec_debug_fetch.restype = ctypes.c_int
    assert dbg.spec_debug_fetch(None) == lib.SPEC_ERR_INVALID_ARG


def test_version_string(lib):
    assert b"sm_103a" in lib.lib.spec_version()


def _args(lib, **kw):
    a = lib.SpecVerifyArgs()
    a.B, a.V, a.K_max, a.total_rows, a.dtype = 4, 1024, 4, 8, lib.SPEC_BF16
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    for f in ("target_logits", "draft_logits", "row_off", "draft_tokens", "uniforms", "accept_len",
              "out_tokens", "req_status"):
        setattr(a, f, fake)
    a.temperature_scalar = 1.0
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,want", [
    ("B", 0, -1), ("V", 0, -1), ("K_max", 65, -1), ("K_max", -1, -1), ("total_rows", 3, -1),
    ("total_rows", 100, -1), ("dtype", 7, -1), ("target_logits", None, -1), ("uniforms", None, -1),
    ("row_off", None, -1), ("accept_len", None, -1), ("draft_logits", None, -1),
    ("temperature_scalar", float("nan"), -1), ("temperature_scalar", -1.0, -1),
    ("V", 1001, -4),                                     # bf16 row of 2002 bytes: not 16-aligned
    ("target_logits", ctypes.c_void_p(0x10008), -4),     # misaligned base
])
def test_host_argument_checks(lib, field, value, want):
    a = _args(lib, **{field: value})
    ws = ctypes.c_void_p(0x20000)
    rc = lib.lib.spec_verify(ctypes.byref(a), ws, 1 << 20, None)
    assert rc == want


def test_workspace_checks(lib):
    a = _args(lib)
    need = lib.lib.spec_verify_workspace_size(4, 1024, 8, lib.SPEC_BF16)
    assert need > 0 and need % 256 == 0
    assert lib.lib.spec_verify(ctypes.byref(a), None, need, None) == -2
    assert lib.lib.spec_verify(ctypes.byref(a), ctypes.c_void_p(0x20000), need - 1, None) == -2
    assert lib.lib.spec_verify(ctypes.byref(a), ctypes.c_void_p(0x20010), need, None) == -2


def test_compact_and_gamma_argument_checks(lib):
    c = lib.SpecCompactArgs()
    c.B, c.page_size, c.max_blocks, c.total_rows = 4, 0, 8, 8
    assert lib.lib.spec_compact(ctypes.byref(c), None) == -1
    fake = ctypes.c_void_p(0x10000)
    assert lib.lib.spec_choose_gamma(fake, fake, 0.5, -1.0, 0, 8, fake, fake, None) == -1
    assert lib.lib.spec_choose_gamma(fake, fake, 0.5, 0.1, 5, 2, fake, fake, None) == -1
    assert lib.lib.spec_choose_gamma(None, fake, 0.5, 0.1, 0, 8, fake, fake, None) == -1
    assert lib.lib.spec_choose_gamma(fake, fake, 1.5, 0.1, 0, 8, fake, fake, None) == -1


def test_gamma_objective_matches_oracle(lib):
    import oracle
    rng = np.random.default_rng(0)
    for _ in range(500):
        a = float(rng.choice([rng.random(), 1.0, 0.0]))
        c = float(rng.random() * rng.choice([0.01, 0.3, 2.0]))
        g = int(rng.integers(0, 20))
        want = oracle.gamma_objective(a, c, g)
        got = lib.lib.spec_gamma_objective(a, c, g)
        assert abs(got - want) <= 1e-14 * max(1.0, abs(want))


def test_depth_objective_matches_oracle(lib):
    import oracle
    from speculative_decoding_verification_43_gb300 import api
    rng = np.random.default_rng(1)
    for _ in range(300):
        D = int(rng.integers(0, 10))
        nr = rng.integers(0, 50, size=D).astype(np.int32)
        na = np.array([rng.integers(0, r + 1) for r in nr], np.int32)
        nr[rng.random(D) < 0.2] = 0  # unobserved depths
        na[nr == 0] = 0
        prev = float(rng.random())
        c = float(rng.random() * rng.choice([0.01, 0.3, 2.0]))
        g = int(rng.integers(0, 16))
        want = oracle.depth_objective(nr, na, prev, c, g)
        got = api.depth_objective(nr, na, prev, c, g)
        assert abs(got - want) <= 1e-13 * max(1.0, abs(want))


def test_choose_gamma_depth_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(16)
    f = lib.lib.spec_choose_gamma_depth
    assert f(fake, fake, 4, 0.5, 0.1, 0, 8, None, fake, None) == -1
    assert f(fake, fake, 4, 0.5, 0.1, 0, 8, fake, None, None) == -1
    assert f(None, fake, 4, 0.5, 0.1, 0, 8, fake, fake, None) == -1
    assert f(fake, fake, -1, 0.5, 0.1, 0, 8, fake, fake, None) == -1
    assert f(fake, fake, 4, 0.5, -1.0, 0, 8, fake, fake, None) == -1
    assert f(fake, fake, 4, 0.5, 0.1, 5, 2, fake, fake, None) == -1
    assert f(fake, fake, 4, 1.5, 0.1, 0, 8, fake, fake, None) == -1
    assert f(fake, fake, 4, 0.5, 0.1, 0, 5000, fake, fake, None) == -1


def test_workload_generator_is_seeded_and_shaped():
    from speculative_decoding_verification_43_gb300 import workloads as W
    wl = W.scaled(W.WORKLOADS["c3"], B=8, V=2048)
    a = W.make_round(wl, seed=4, rnd=1)
    b = W.make_round(wl, seed=4, rnd=1)
    c = W.make_round(wl, seed=4, rnd=2)
    assert torch.equal(a.target, b.target) and torch.equal(a.draft_tokens, b.draft_tokens)
    assert not torch.equal(a.target, c.target)
    np.testing.assert_array_equal(a.K, c.K)  # the batch shape depends on the seed only
    assert a.target.dtype == torch.bfloat16 and a.target.shape == (int(a.row_off[-1]), 2048)
    assert a.draft.shape == (int(a.row_off[-1]) - 8, 2048)
    assert ((a.draft_tokens >= 0) & (a.draft_tokens < 2048)).all()
    u = a.uniforms.numpy()
    assert ((u >= 0) & (u < 1)).all()
    assert np.all(np.floor(u * 2.0 ** 53) == u * 2.0 ** 53)  # 53-bit values k / 2^53


def test_workload_k_distributions():
    from speculative_decoding_verification_43_gb300 import workloads as W
    k3 = W.WORKLOADS["c3"].k_values(0)
    assert len(k3) == 64 and k3.min() >= 0 and k3.max() <= 7
    k5 = W.WORKLOADS["c5"].k_values(0)
    assert (k5 == 2).sum() == 128 and (k5 == 1).sum() == 128 and (k5 == 0).sum() == 256
    assert (W.WORKLOADS["c4"].k_values(0) == 3).all()
    assert W.WORKLOADS["c5"].bytes_per_round(0) == 1280 * 256000 * 2


def test_zipf_rows_follow_the_recipe():
    from speculative_decoding_verification_43_gb300 import workloads as W
    wl = W.Workload("z", B=4, V=4096, dtype=torch.float32, temperature=1.0, logits="zipf", sigma=1.0,
                    draft_sigma=0.0, K="fixed:1")
    rd = W.make_round(wl, seed=1)
    row = rd.target[0].double().numpy()
    # sorted logits track -1.1 ln(rank) up to the N(0,1) noise
    ranks = np.arange(1, 4097)
    srt = np.sort(row)[::-1]
    assert np.abs(np.mean(srt[1000:3000] + 1.1 * np.log(ranks[1000:3000]))) < 0.5
    # draft noise 0 gives the same row
    assert torch.equal(rd.draft[0], rd.target[0])


def test_plan_rejects_invalid_shapes_without_a_device(lib):
    """spec_verify_plan checks the shape before it asks the device anything."""
    f = lib.lib.spec_verify_plan
    assert f(0, 1000, 10, lib.SPEC_F32, None, None) is None
    assert f(4, 1001, 10, lib.SPEC_BF16, None, None) is None
    assert f(8, 1024, 7, lib.SPEC_F32, None, None) is None
    assert f(4, 1024, 10, 7, None, None) is None


def test_round_argument_checks(lib):
    """spec_verify_round checks all three calls' arguments before it enqueues anything: each bad
    one fails without touching a device (every pointer here is fake)."""
    fake = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x20000)
    f = lib.lib.spec_verify_round

    def compact(**kw):
        c = lib.SpecCompactArgs()
        c.B, c.page_size, c.max_blocks, c.total_rows = 4, 16, 8, 8
        for n in ("row_off", "accept_len", "out_tokens", "prefix_len", "block_table", "out_off", "packed_tokens",
                  "packed_pos", "kv_off", "new_seq_len", "new_kv_len", "cand_kv_rows", "kv_src", "kv_dst"):
            setattr(c, n, fake)
        for k, v in kw.items():
            setattr(c, k, v)
        return c

    a = _args(lib, alpha_sum=fake, alpha_count=fake)
    good = compact()
    assert f(None, ws, 1 << 20, ctypes.byref(good), 0.5, 0.1, 0, 8, fake, fake, None) == -1
    assert f(ctypes.byref(a), ws, 1 << 20, None, 0.5, 0.1, 0, 8, fake, fake, None) == -1
    assert f(ctypes.byref(a), ws, 1 << 20, ctypes.byref(compact(page_size=0)), 0.5, 0.1, 0, 8, fake, fake, None) == -1
    assert f(ctypes.byref(a), ws, 1 << 20, ctypes.byref(compact(B=5, total_rows=9)), 0.5, 0.1, 0, 8, fake, fake,
             None) == -1
    assert f(ctypes.byref(a), ws, 1 << 20, ctypes.byref(good), 0.5, -1.0, 0, 8, fake, fake, None) == -1
    assert f(ctypes.byref(a), ws, 1 << 20, ctypes.byref(good), 0.5, 0.1, 5, 2, fake, fake, None) == -1
    b = _args(lib)  # no alpha_sum / alpha_count for the gamma step
    assert f(ctypes.byref(b), ws, 1 << 20, ctypes.byref(good), 0.5, 0.1, 0, 8, fake, fake, None) == -1
    # a verify argument that spec_verify rejects is rejected here too
    c = _args(lib, alpha_sum=fake, alpha_count=fake, V=1001)
    assert f(ctypes.byref(c), ws, 1 << 20, ctypes.byref(good), 0.5, 0.1, 0, 8, fake, fake, None) == -4


def test_ctypes_structs_match_the_header_layout():
    """The binding's ctypes structs against the C compiler's layout of include/spec_verify.h:
    every field at the same offset, and the same total size."""
    import shutil
    import subprocess
    import tempfile

    from speculative_decoding_verification_43_gb300 import _lib

    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if not shutil.which("gcc") or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    inc = os.path.join(ROOT, "include")
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "spec_verify.h"', "int main(void) {"]
    for cname, cls in (("spec_verify_args", _lib.SpecVerifyArgs), ("spec_compact_args", _lib.SpecCompactArgs)):
        lines.append(f'printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        open(src, "w").write("\n".join(lines))
        subprocess.check_call(["gcc", "-std=c11", "-I", inc, "-I", cuda_inc, src, "-o", exe])
        out = subprocess.check_output([exe], text=True)
    got = {(a, b): int(c) for a, b, c in (ln.split() for ln in out.splitlines())}
    for cname, cls in (("spec_verify_args", _lib.SpecVerifyArgs), ("spec_compact_args", _lib.SpecCompactArgs)):
        assert got[(cname, "sizeof")] == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert got[(cname, f)] == getattr(cls, f).offset, (cname, f)
