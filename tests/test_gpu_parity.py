"""GPU parity: the CUDA verifier against the float64 oracle, element by element.

Sizes: the five workloads (c1 and c2 over many rounds; c3 in full; c4 and c5 at full size with
the oracle run on a seeded sample of requests), plus smaller batches that still span several
1024-token groups, several CTAs of a cluster and a ragged tail, and the edge cases of the rule.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_43_gb300 import api
from speculative_decoding_verification_43_gb300 import workloads as W

from parity import Report, check_round, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu





def record(name, rep):
    """Append the report's counts as one JSON line to the file named by SPEC_PARITY_COUNTS (when
    set): the per-configuration table of requests, compared and band counts."""
    path = os.environ.get("SPEC_PARITY_COUNTS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(case=name, **rep.counts(), alpha_max_rel=rep.alpha_max_rel,
                                    rho_max_rel=rep.rho_max_rel, resid_max_rel=rep.resid_max_rel,
                                    prob_max_rel=rep.prob_max_rel)) + "\n")


def assert_report(rep, max_near, name=None):
    """No mismatch and no value failure outside the band. The band is the oracle's alone, so
    its size is fixed by the seeded inputs: `max_near` bounds it per configuration at about
    twice the oracle's own count on those inputs (plus one), so that a workload change that
    pushes many draws into the band cannot pass unnoticed. A request that only the kernel's
    margin would place in the band is compared all the same; at most one per case is expected
    (its margin differs from the oracle's by rounding only)."""
    print(rep.summary())
    if name:
        record(name, rep)
    assert rep.ok(), (rep.mismatches[:5], rep.value_failures[:5])
    assert rep.near_boundary <= max_near, rep.summary()
    assert rep.gpu_near_only <= 1, rep.summary()


def test_c1_all_rounds():
    # the oracle's band count on these 100 rounds: 0
    wl = W.WORKLOADS["c1"]
    tot = Report()
    for rnd in range(wl.rounds):
        rd = W.make_round(wl, seed=0, rnd=rnd, device="cuda")
        tot.add(check_round(rd))
    assert_report(tot, max_near=1, name="c1 (100 rounds)")


def test_c2_rounds():
    # the oracle's band count on these 60 rounds of 8 requests: 11
    wl = W.WORKLOADS["c2"]
    tot = Report()
    for rnd in range(60):
        rd = W.make_round(wl, seed=0, rnd=rnd, device="cuda")
        tot.add(check_round(rd))
    assert_report(tot, max_near=23, name="c2 (60 rounds)")


def test_c3_full_batch():
    # the oracle's band count on this round: 1 of 64
    wl = W.WORKLOADS["c3"]
    rd = W.make_round(wl, seed=0, rnd=0, device="cuda")
    assert_report(check_round(rd), max_near=3, name="c3")


# the oracle's band counts on these samples: 1 of 24 (c4) and 10 of 64 (c5: flat Zipf tails over
# 256000 tokens)
@pytest.mark.parametrize("name,n_sample,max_near", [("c4", 24, 3), ("c5", 64, 21)])
def test_full_size_sampled(name, n_sample, max_near):
    wl = W.WORKLOADS[name]
    rd = W.make_round(wl, seed=0, rnd=0, device="cuda")
    rng = np.random.default_rng(7)
    reqs = sorted(rng.choice(rd.B, size=n_sample, replace=False).tolist())
    assert_report(check_round(rd, reqs), max_near=max_near, name=f"{name} (sample of {n_sample})")


# the oracle's band counts over the three rounds of each shape: 6, 2, 0, 0, 2
@pytest.mark.parametrize("dtype,V,B,Kspec,T,max_near", [
    (torch.bfloat16, 50264, 40, "uniform:0:8", 0.8, 13),   # many chunks per row, ragged tail
    (torch.float32, 12348, 24, "uniform:0:6", 1.3, 5),     # fp32, ragged
    (torch.bfloat16, 1032, 12, "uniform:0:4", 1.0, 1),     # one partial chunk per row
    (torch.float32, 8, 9, "uniform:0:3", 0.9, 1),          # V smaller than one vector per lane
    (torch.bfloat16, 262144, 6, "uniform:1:3", 1.0, 5),    # large V: flat rows over 2^18 tokens
])
def test_shapes(dtype, V, B, Kspec, T, max_near):
    base = W.Workload("t", B=B, V=V, dtype=dtype, temperature=T, logits="normal", sigma=2.0,
                      draft_sigma=0.7, K=Kspec)
    tot = Report()
    for rnd in range(3):
        rd = W.make_round(base, seed=11, rnd=rnd, device="cuda")
        tot.add(check_round(rd))
    assert_report(tot, max_near=max_near, name=f"shape {str(dtype)[6:]} V={V} B={B} K~{Kspec} T={T} (3 rounds)")


def test_zipf_small_vocab_many_rounds():
    # the oracle's band count over these 8 rounds of 32 requests: 1
    base = W.scaled(W.WORKLOADS["c3"], B=32, V=8192)
    tot = Report()
    for rnd in range(8):
        rd = W.make_round(base, seed=3, rnd=rnd, device="cuda")
        tot.add(check_round(rd))
    assert_report(tot, max_near=3, name="c3 head at B=32 V=8192 (8 rounds)")


def test_k0_only_and_max_k():
    base = W.Workload("t", B=16, V=4096, dtype=torch.bfloat16, temperature=1.0, logits="normal",
                      sigma=2.0, draft_sigma=0.5, K="fixed:0")
    rd = W.make_round(base, seed=5, device="cuda")
    assert_report(check_round(rd), max_near=3, name="k0_only_and_max_k#1")  # oracle: 1
    base = W.Workload("t", B=2, V=2048, dtype=torch.float32, temperature=1.0, logits="normal",
                      sigma=1.0, draft_sigma=0.2, K="fixed:64")
    rd = W.make_round(base, seed=6, device="cuda")
    assert_report(check_round(rd), max_near=1, name="k0_only_and_max_k#2")  # oracle: 0


def test_forced_accept_all_and_reject_first():
    base = W.Workload("t", B=10, V=6000, dtype=torch.bfloat16, temperature=1.0, logits="normal",
                      sigma=2.0, draft_sigma=0.8, K="fixed:4")
    rd = W.make_round(base, seed=8, device="cuda")
    K = 4
    u = rd.uniforms.clone()
    for i in range(rd.B):
        for j in range(K):
            u[i * (K + 1) + j] = 0.0 if i % 2 == 0 else 1.0 - 2 ** -53
    rd.uniforms = u
    gpu = run_gpu(rd)
    assert (gpu["accept_len"][0::2] == K).all()
    rep = check_round(rd)
    assert_report(rep, max_near=1, name="forced_accept_all_and_reject_first#1")  # oracle: 0


def test_greedy_and_mixed_temperatures():
    base = W.Workload("t", B=12, V=5000, dtype=torch.float32, temperature=1.0, logits="normal",
                      sigma=2.0, draft_sigma=0.6, K="uniform:0:5")
    temps = np.array([0.0, 0.5, 1.0, 2.0] * 3, np.float32)
    rd = W.make_round(base, seed=9, device="cuda", temperature=temps)
    assert_report(check_round(rd), max_near=1, name="greedy_and_mixed_temperatures#1")  # oracle: 0
    # greedy rows with ties: the smallest index wins on both sides
    rd.target[:, 17] = 100.0
    rd.target[:, 3] = 100.0
    assert_report(check_round(rd), max_near=1, name="greedy_and_mixed_temperatures#2")  # oracle: 0


def _resample_drafts(rd, seed):
    """Draft tokens drawn again from q = softmax(draft / T) after the logits were rewritten."""
    gen = torch.Generator(device=rd.draft.device)
    gen.manual_seed(seed)
    K = np.asarray(rd.K)
    req = torch.as_tensor(np.repeat(np.arange(rd.B), K), device=rd.draft.device)
    t = rd.temperature[req].unsqueeze(1)
    z = rd.draft.float()
    u = torch.rand(z.shape, generator=gen, device=z.device).clamp_(min=1e-38)
    score = torch.where(t > 0, z / t.clamp(min=1e-30) - torch.log(-torch.log(u)), z)
    rd.draft_tokens = score.argmax(dim=1).to(torch.int32)


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 131072), (torch.float32, 65536)])
def test_wide_logit_ranges(dtype, V):
    """Rows whose logits span hundreds of units within one thread's share of the slice (a ramp
    across the vocabulary, rising and falling), and rows whose vocabulary is mostly masked to
    -inf: the per-thread reference of pass 1 then takes its exact path."""
    base = W.Workload("t", B=64, V=V, dtype=dtype, temperature=1.0, logits="normal", sigma=1.0,
                      draft_sigma=0.5, K="uniform:0:3")
    rd = W.make_round(base, seed=21, device="cuda")
    ramp = torch.linspace(-300.0, 300.0, V, device="cuda")
    tz = rd.target.float()
    dz = rd.draft.float()
    # rising ramp on even requests, falling ramp on odd ones; every third request mostly masked
    row_req = np.repeat(np.arange(rd.B), np.asarray(rd.K) + 1)
    drow_req = np.repeat(np.arange(rd.B), np.asarray(rd.K))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    mask = torch.rand(rd.B, V, generator=gen, device="cuda") < 0.9
    for i in range(rd.B):
        rr = torch.as_tensor(np.nonzero(row_req == i)[0], device="cuda")
        dr = torch.as_tensor(np.nonzero(drow_req == i)[0], device="cuda")
        if i % 3 == 2:
            tz[rr] = tz[rr].masked_fill(mask[i], float("-inf"))
            if len(dr):
                dz[dr] = dz[dr].masked_fill(mask[i], float("-inf"))
        else:
            sgn = 1.0 if i % 2 == 0 else -1.0
            tz[rr] += sgn * ramp
            if len(dr):
                dz[dr] += sgn * ramp
    rd.target = tz.to(dtype).contiguous()
    rd.draft = dz.to(dtype).contiguous()
    _resample_drafts(rd, 17)
    assert_report(check_round(rd), max_near=1, name=f"wide_logit_ranges V={V}")  # oracle: 0 and 0


def test_bad_requests():
    base = W.Workload("t", B=10, V=3000, dtype=torch.bfloat16, temperature=1.0, logits="normal",
                      sigma=2.0, draft_sigma=0.6, K="fixed:3")
    rd = W.make_round(base, seed=10, device="cuda")
    ro = rd.row_off.cpu().numpy()
    rd.target[ro[1] + 1, 7] = float("nan")                 # request 1: NaN target
    rd.draft_tokens[3 * 3 + 0] = 3000                      # request 3: token out of range
    x = int(rd.draft_tokens[5 * 3 + 2])
    rd.draft[5 * 3 + 2, x] = float("-inf")                 # request 5: q(x) == 0
    rd.target[ro[7] + 3, 11] = float("inf")               # request 7: +inf in the bonus row
    rd.draft[8 * 3 + 1, :] = float("-inf")                 # request 8: a draft row with no mass
    rd.temperature[9] = -1.0                               # request 9: bad temperature
    rep = check_round(rd)
    assert_report(rep, max_near=1, name="bad_requests#1")  # oracle: 0
    gpu = run_gpu(rd)
    assert gpu["req_status"][1] == api._lib.REQ_BAD_LOGITS
    assert gpu["req_status"][3] == api._lib.REQ_BAD_PROPOSAL
    assert gpu["req_status"][5] == api._lib.REQ_BAD_PROPOSAL
    assert gpu["req_status"][7] == api._lib.REQ_BAD_LOGITS
    assert gpu["req_status"][9] & api._lib.REQ_BAD_PARAM
    for i in (0, 2, 4, 6):
        assert gpu["req_status"][i] == 0


def test_k_max_exceeded_is_bad_shape():
    base = W.Workload("t", B=6, V=2048, dtype=torch.float32, temperature=1.0, logits="normal",
                      sigma=1.0, draft_sigma=0.5, K="uniform:0:6")
    rd = W.make_round(base, seed=12, device="cuda")
    gpu = run_gpu(rd, K_max=3)
    for i, k in enumerate(rd.K):
        assert (gpu["req_status"][i] == api._lib.REQ_BAD_SHAPE) == (k > 3)
    rep = check_round(rd, K_max=3)
    assert_report(rep, max_near=1, name="k_max_exceeded_is_bad_shape#1")  # oracle: 0


def test_stop_token_and_budget():
    base = W.Workload("t", B=24, V=3000, dtype=torch.bfloat16, temperature=1.0, logits="normal",
                      sigma=1.0, draft_sigma=0.3, K="fixed:5")
    rd = W.make_round(base, seed=13, device="cuda")
    plain = run_gpu(rd)
    stop = np.full(rd.B, -1, np.int32)
    budget = np.full(rd.B, 1000, np.int32)
    for i in range(rd.B):
        n = plain["n_emitted"][i]
        toks = plain["out_tokens"][i * 6:i * 6 + n]
        if i % 3 == 0 and n > 1:
            stop[i] = toks[n // 2]
        if i % 3 == 1:
            budget[i] = max(0, n - 2)
    stop_t = torch.as_tensor(stop, device="cuda")
    budget_t = torch.as_tensor(budget, device="cuda")
    rep = check_round(rd, stop_token=stop_t, max_new=budget_t)
    assert_report(rep, max_near=1, name="stop_token_and_budget#1")  # oracle: 0


def test_determinism():
    rd = W.make_round(W.scaled(W.WORKLOADS["c3"], B=16, V=32768), seed=2, device="cuda")
    a = run_gpu(rd)
    b = run_gpu(rd)
    for k in ("accept_len", "out_tokens", "alpha_rows", "rho_rows", "alpha_sum"):
        np.testing.assert_array_equal(a[k], b[k])


def test_alpha_sum_and_count():
    rd = W.make_round(W.WORKLOADS["c5"], seed=1, device="cuda")
    gpu = run_gpu(rd)
    ok = gpu["req_status"] == 0
    K = rd.K
    want = sum(gpu["alpha_rows"][int(rd.row_off[i]) - i: int(rd.row_off[i]) - i + K[i]].astype(np.float64).sum()
               for i in range(rd.B) if ok[i])
    assert gpu["alpha_count"][0] == K[ok].sum()
    assert abs(gpu["alpha_sum"][0] - want) <= 1e-9 * max(1.0, want)


def test_choose_gamma_device_matches_oracle():
    for alpha, count, prev, c in ((0.7, 40, 0.1, 0.05), (1.0, 5, 0.0, 1.0), (0.0, 0, 0.7, 0.05),
                                  (0.93, 128, 0.5, 0.02), (0.31, 7, 0.5, 0.3)):
        s = torch.tensor([alpha * count], dtype=torch.float64, device="cuda")
        n = torch.tensor([count], dtype=torch.int32, device="cuda")
        g, a = api.choose_gamma(s, n, prev, c, 0, 8)
        want_g, want_a = oracle.choose_gamma(alpha * count, count, prev, c, 0, 8)
        assert int(g.item()) == want_g
        assert abs(float(a.item()) - want_a) < 1e-12  # float-pair arithmetic on the device


def test_depth_counts_and_depth_gamma():
    """Per-depth counts written by spec_verify equal the censored counts of its own accept
    lengths (requests with status bits excluded), and the device's depth-aware gamma choice
    equals the oracle's on those counts and on constructed ones."""
    wl = W.WORKLOADS["c3"]
    rd = W.make_round(wl, seed=0, device="cuda")
    temps = rd.temperature.clone()
    temps[5] = -1.0  # a bad request: excluded from the counts
    gpu = run_gpu(rd, temperature=temps)
    ro = rd.row_off.cpu().numpy()
    nr, na = oracle.depth_counts(ro, gpu["accept_len"], gpu["req_status"], 64)
    assert gpu["req_status"][5] != 0
    np.testing.assert_array_equal(gpu["depth_reached"], nr)
    np.testing.assert_array_equal(gpu["depth_accepted"], na)
    assert nr[0] > 0 and nr[7] == 0  # K_i <= 7 in this workload
    cases = [(nr, na)]
    rng = np.random.default_rng(3)
    for _ in range(6):
        D = int(rng.integers(1, 12))
        r = rng.integers(0, 200, size=D).astype(np.int32)
        r[rng.random(D) < 0.25] = 0
        a = np.array([rng.integers(0, x + 1) for x in r], np.int32)
        cases.append((r, a))
    cases.append((np.zeros(4, np.int32), np.zeros(4, np.int32)))          # nothing observed
    cases.append((np.array([64, 32, 16], np.int32), np.array([32, 16, 8], np.int32)))  # constant 1/2
    for r, a in cases:
        for prev, c, gmin, gmax in ((0.5, 0.05, 0, 8), (0.2, 0.3, 1, 12), (0.9, 0.01, 0, 20)):
            g, ea = api.choose_gamma_depth(torch.as_tensor(r, device="cuda"), torch.as_tensor(a, device="cuda"),
                                           prev, c, gmin, gmax)
            og, oea = oracle.choose_gamma_depth(r, a, prev, c, gmin, gmax)
            assert int(g.item()) == og, (r, a, prev, c)
            assert abs(float(ea.item()) - oea) <= 1e-6 * max(1.0, oea)


def test_compaction_bit_exact_c4():
    wl = W.WORKLOADS["c4"]
    rd = W.make_round(wl, seed=0, device="cuda")
    out = api.verify(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
    ci = W.make_compaction_inputs(rd, wl.prefix_len, wl.page_size)
    c = api.compact(rd.row_off, out.accept_len, out.n_emitted, out.out_tokens, out.req_status,
                    ci["prefix_len"], ci["cand_kv_rows"], ci["block_table"], ci["page_size"])
    torch.cuda.synchronize()
    o = oracle.compact(rd.row_off.cpu().numpy(), out.accept_len.cpu().numpy(), out.n_emitted.cpu().numpy(),
                       out.out_tokens.cpu().numpy(), out.req_status.cpu().numpy(),
                       ci["prefix_len"].cpu().numpy(), ci["cand_kv_rows"].cpu().numpy(),
                       ci["block_table"].cpu().numpy(), ci["page_size"])
    n_out, n_kv = int(o["out_off"][-1]), int(o["kv_off"][-1])
    for k in ("out_off", "kv_off", "new_seq_len", "new_kv_len", "new_draft_len", "compact_status"):
        np.testing.assert_array_equal(getattr(c, k).cpu().numpy(), o[k], err_msg=k)
    for k, n in (("packed_tokens", n_out), ("packed_pos", n_out), ("kv_src", n_kv), ("kv_dst", n_kv)):
        np.testing.assert_array_equal(getattr(c, k).cpu().numpy()[:n], o[k], err_msg=k)


def test_compaction_of_more_requests_than_one_pass():
    """B = 2600 requests: the compaction kernel scans and copies them in three passes of 1024,
    carrying the offsets across passes; K up to 40, so that some requests copy more tokens than
    a warp has lanes."""
    base = W.Workload("t", B=2600, V=64, dtype=torch.float32, temperature=1.0, logits="normal",
                      sigma=1.0, draft_sigma=0.2, K="uniform:0:40")
    rd = W.make_round(base, seed=21, device="cuda")
    out = api.verify(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature)
    ci = W.make_compaction_inputs(rd, 37, 16)
    c = api.compact(rd.row_off, out.accept_len, out.n_emitted, out.out_tokens, out.req_status,
                    ci["prefix_len"], ci["cand_kv_rows"], ci["block_table"], 16)
    torch.cuda.synchronize()
    o = oracle.compact(rd.row_off.cpu().numpy(), out.accept_len.cpu().numpy(), out.n_emitted.cpu().numpy(),
                       out.out_tokens.cpu().numpy(), out.req_status.cpu().numpy(),
                       ci["prefix_len"].cpu().numpy(), ci["cand_kv_rows"].cpu().numpy(),
                       ci["block_table"].cpu().numpy(), 16)
    assert int(o["kv_off"][-1]) > 0 and int(out.accept_len.max()) > 32
    n_out, n_kv = int(o["out_off"][-1]), int(o["kv_off"][-1])
    for k in ("out_off", "kv_off", "new_seq_len", "new_kv_len", "new_draft_len", "compact_status"):
        np.testing.assert_array_equal(getattr(c, k).cpu().numpy(), o[k], err_msg=k)
    for k, n in (("packed_tokens", n_out), ("packed_pos", n_out), ("kv_src", n_kv), ("kv_dst", n_kv)):
        np.testing.assert_array_equal(getattr(c, k).cpu().numpy()[:n], o[k], err_msg=k)


def test_compaction_with_stops_and_bad_blocks():
    base = W.Workload("t", B=300, V=1024, dtype=torch.float32, temperature=1.0, logits="normal",
                      sigma=1.0, draft_sigma=0.4, K="uniform:0:6")
    rd = W.make_round(base, seed=14, device="cuda")
    rng = np.random.default_rng(3)
    stop = torch.as_tensor(rng.integers(-1, 1024, rd.B).astype(np.int32), device="cuda")
    budget = torch.as_tensor(rng.integers(0, 8, rd.B).astype(np.int32), device="cuda")
    out = api.verify(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, rd.temperature,
                     stop_token=stop, max_new=budget)
    ci = W.make_compaction_inputs(rd, 100, 16)
    bt = ci["block_table"].clone()
    bt[5, :] = -1
    P = ci["prefix_len"].clone()
    P[7] = bt.shape[1] * 16 - 1
    c = api.compact(rd.row_off, out.accept_len, out.n_emitted, out.out_tokens, out.req_status, P,
                    ci["cand_kv_rows"], bt, 16)
    torch.cuda.synchronize()
    o = oracle.compact(rd.row_off.cpu().numpy(), out.accept_len.cpu().numpy(), out.n_emitted.cpu().numpy(),
                       out.out_tokens.cpu().numpy(), out.req_status.cpu().numpy(), P.cpu().numpy(),
                       ci["cand_kv_rows"].cpu().numpy(), bt.cpu().numpy(), 16)
    n_out, n_kv = int(o["out_off"][-1]), int(o["kv_off"][-1])
    for k in ("out_off", "kv_off", "new_seq_len", "new_kv_len", "new_draft_len", "compact_status"):
        np.testing.assert_array_equal(getattr(c, k).cpu().numpy(), o[k], err_msg=k)
    for k, n in (("packed_tokens", n_out), ("packed_pos", n_out), ("kv_src", n_kv), ("kv_dst", n_kv)):
        np.testing.assert_array_equal(getattr(c, k).cpu().numpy()[:n], o[k], err_msg=k)


def _trunc_params(B, V, seed):
    """Per-request top-k / top-p values: off, extreme and ordinary ones, mixed."""
    rng = np.random.default_rng(seed)
    ks = np.array([0, 1, 3, 50, 1000, V - 1, V + 7], np.int32)
    ps = np.array([1.0, 0.9, 0.5, 0.99, 0.0, 0.7, 0.95], np.float32)
    top_k = torch.as_tensor(ks[rng.integers(0, len(ks), B)], device="cuda")
    top_p = torch.as_tensor(ps[rng.integers(0, len(ps), B)], device="cuda")
    return top_k, top_p


# the oracle's band counts: 10, 12 and 7 (a target row whose top-p cut lies within 1e-5 of top_p
# counts as well as the draws)
@pytest.mark.parametrize("dtype,V,logits,max_near", [(torch.bfloat16, 32000, "zipf", 21),
                                                     (torch.float32, 20000, "normal", 25),
                                                     (torch.bfloat16, 128256, "zipf", 15)])
def test_top_k_top_p(dtype, V, logits, max_near):
    """Top-k then top-p of the target law (SDCP "Session Model"): the cut of each target row by
    the truncation kernel, the masked rows in the per-position kernel, every draw of the
    truncated law. Some requests use the greedy rule, which ignores truncation."""
    base = W.Workload("t", B=48 if V < 100000 else 24, V=V, dtype=dtype, temperature=0.8, logits=logits,
                      sigma=2.0, draft_sigma=0.7, K="uniform:0:5")
    rd = W.make_round(base, seed=31, device="cuda")
    temp = rd.temperature.clone()
    temp[::11] = 0.0
    rd.temperature = temp
    top_k, top_p = _trunc_params(rd.B, V, 7)
    assert_report(check_round(rd, top_k=top_k, top_p=top_p), max_near=max_near, name=f"top_k_top_p V={V}")


def test_top_k_cuts_inside_ties():
    """Integer-valued logits put many tokens at the cut's logit: the kept ones are the
    smallest ids among them, on both sides."""
    base = W.Workload("t", B=40, V=4096, dtype=torch.bfloat16, temperature=1.0, logits="normal", sigma=2.0,
                      draft_sigma=0.5, K="uniform:0:3")
    rd = W.make_round(base, seed=5, device="cuda")
    rd.target = torch.round(rd.target.float()).to(torch.bfloat16).contiguous()
    top_k = torch.as_tensor(np.random.default_rng(2).integers(1, 400, rd.B).astype(np.int32), device="cuda")
    top_p = torch.full((rd.B,), 0.9, dtype=torch.float32, device="cuda")
    top_p[::2] = 1.0
    assert_report(check_round(rd, top_k=top_k, top_p=top_p), max_near=5, name="top_k_cuts_inside_ties#1")  # oracle: 2


def test_nan_top_p_is_a_bad_parameter_on_device():
    base = W.Workload("t", B=8, V=2048, dtype=torch.float32, temperature=1.0, logits="normal", sigma=1.0,
                      draft_sigma=0.5, K="fixed:2")
    rd = W.make_round(base, seed=9, device="cuda")
    top_p = torch.ones(rd.B, dtype=torch.float32, device="cuda")
    top_p[3] = float("nan")
    g = run_gpu(rd, top_p=top_p)
    assert g["req_status"][3] == 8 and g["n_emitted"][3] == 0
    assert (np.delete(g["req_status"], 3) == 0).all()


def test_all_64_drafts_accepted():
    """K = K_max = 64 with every accept draw at 0: A = 64 and the frontier token is drawn from
    the 65th target row (the selection's third slot per warp)."""
    base = W.Workload("t", B=3, V=2048, dtype=torch.float32, temperature=1.0, logits="normal",
                      sigma=1.0, draft_sigma=0.2, K="fixed:64")
    rd = W.make_round(base, seed=12, device="cuda")
    u = rd.uniforms.clone()
    for i in range(rd.B):
        u[i * 65:i * 65 + 64] = 0.0
    rd.uniforms = u
    gpu = run_gpu(rd)
    assert (gpu["accept_len"] == 64).all() and (gpu["n_emitted"] == 65).all()
    assert (gpu["out_tokens"].reshape(rd.B, 65) >= 0).all()
    assert_report(check_round(rd), max_near=1, name="all_64_drafts_accepted")


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 32000), (torch.float32, 12348)])
def test_extreme_temperatures(dtype, V):
    """Temperatures near the greedy limit (s = log2(e)/T up to 144: exponent arguments far beyond
    the float range, so the statistics take their exact form) and a very flat law (T = 50), mixed
    in one batch."""
    base = W.Workload("t", B=20, V=V, dtype=dtype, temperature=1.0, logits="normal", sigma=2.0,
                      draft_sigma=0.3, K="uniform:0:4")
    temps = np.array([0.01, 0.02, 0.05, 0.1, 50.0] * 4, np.float32)
    tot = Report()
    for rnd in range(2):
        rd = W.make_round(base, seed=14, rnd=rnd, device="cuda", temperature=temps)
        tot.add(check_round(rd))
    # the oracle's band count on these rounds: 0 (both configurations)
    assert_report(tot, max_near=1, name=f"extreme temperatures {str(dtype)[6:]} V={V} (2 rounds)")


@pytest.mark.parametrize("dtype,V,shift", [(torch.bfloat16, 32000, 1000.0), (torch.bfloat16, 32000, -3000.0),
                                           (torch.float32, 12348, 30000.0)])
def test_large_logit_offsets(dtype, V, shift):
    """Every logit of the batch shifted by one large constant (the law is unchanged; the products
    y s reach ~4e4, so every exponent argument depends on the reference being subtracted before
    rounding, and the low part of s on the row's top logit). Temperatures 0.7 and 1.3."""
    base = W.Workload("t", B=16, V=V, dtype=dtype, temperature=1.0, logits="normal", sigma=2.0,
                      draft_sigma=0.6, K="uniform:0:5")
    temps = np.array([0.7, 1.3] * 8, np.float32)
    rd = W.make_round(base, seed=15, device="cuda", temperature=temps)
    rd.target = (rd.target.float() + shift).to(dtype).contiguous()
    rd.draft = (rd.draft.float() + shift).to(dtype).contiguous()
    _resample_drafts(rd, 19)
    # the oracle's band count on each of these rounds: 0
    assert_report(check_round(rd), max_near=1, name=f"logits shifted by {shift:g} {str(dtype)[6:]} V={V}")


def test_degenerate_laws():
    """Laws at the edges of the rule, in one batch (SOTA-227 "What to do", steps 3-4):
    - constant rows: p = q uniform, every draft accepted, the extra token drawn over equal weights;
    - one-hot drafts (every draft logit -inf but the proposed token's): q(x) = 1, rho = p(x), and
      the residual is p with x removed;
    - sparse targets (all but 16 logits -inf) against dense drafts: p(x) = 0 rejects, and the
      residual lives on p's 16 tokens."""
    V = 4096
    base = W.Workload("t", B=24, V=V, dtype=torch.float32, temperature=1.0, logits="normal", sigma=2.0,
                      draft_sigma=0.5, K="uniform:1:4")
    rd = W.make_round(base, seed=16, device="cuda")
    tz, dz = rd.target.clone(), rd.draft.clone()
    row_req = np.repeat(np.arange(rd.B), np.asarray(rd.K) + 1)
    drow_req = np.repeat(np.arange(rd.B), np.asarray(rd.K))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    keep = torch.zeros(rd.B, V, dtype=torch.bool, device="cuda")
    for i in range(rd.B):
        keep[i, torch.randperm(V, generator=gen, device="cuda")[:16]] = True
    for i in range(rd.B):
        rr = torch.as_tensor(np.nonzero(row_req == i)[0], device="cuda")
        dr = torch.as_tensor(np.nonzero(drow_req == i)[0], device="cuda")
        if i % 3 == 0:      # constant rows
            tz[rr] = 0.5
            dz[dr] = 0.5
        elif i % 3 == 2:    # sparse targets
            tz[rr] = tz[rr].masked_fill(~keep[i], float("-inf"))
    rd.target = tz.contiguous()
    rd.draft = dz.contiguous()
    _resample_drafts(rd, 23)
    # one-hot drafts on the second kind, around the proposed token
    dz = rd.draft.clone()
    toks = rd.draft_tokens.cpu().numpy()
    for i in range(rd.B):
        if i % 3 == 1:
            for j in np.nonzero(drow_req == i)[0]:
                row = torch.full((V,), float("-inf"), device="cuda")
                row[int(toks[j])] = 1.0
                dz[int(j)] = row
    rd.draft = dz.contiguous()
    rep = check_round(rd)
    # the oracle's band count on this round: 0
    assert_report(rep, max_near=1, name="degenerate laws")
