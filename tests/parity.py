"""Comparison of the CUDA verifier against the float64 oracle on the same seeded inputs.

The bar:
  * accept lengths, emitted tokens and status bits are bit-exact, except for requests with a
    draw whose uniform lies, on the ORACLE's side, within BAND = 1e-6 of an acceptance ratio
    or of a CDF boundary of the frontier draw; those requests are counted and reported, not
    compared. The kernel's own margins decide nothing: a request that only the kernel places
    in the band is compared like any other and counted in `gpu_near_only`.
  * alpha (sum of min(p, q)), the accept ratio p/q, the residual mass and the frontier token's
    probability are within RTOL = 1e-5 relative.

Float decisions on each side are taken in each side's own precision (the oracle in float64,
the kernels in float32 with wider accumulation), which is why a band exists at all.

alpha is a sum of positive terms; below ALPHA_FLOOR = 1e-6 (a mass of a few float32 units of a
unit sum) it is held to RTOL * ALPHA_FLOOR absolute and the rows are counted
(`alpha_below_floor`). The residual mass Z = sum max(p - q, 0) and a residual draw's probability
(p(x) - q(x)) / Z are differences: computed from float32 p and q they would lose accuracy in
proportion to the conditioning figures the oracle reports (`resid_scale / Z`, `sample_cond`). The
kernels form each residual weight without cancellation, so these two are held to RTOL relative
whatever the conditioning; the largest conditioning figure among the compared rows is reported
(`resid_cond_max`, `prob_cond_max`) to show the range the bound was met over.

With top-p, the cut of a target row is a boundary too: a request with a row whose cumulative
mass at the oracle's cut lies within TRUNC_BAND of top_p is counted with the band (the kernel
sums the masses of the cut in fixed point from float32 exponentials).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
from speculative_decoding_verification_43_gb300 import api
from speculative_decoding_verification_43_gb300.workloads import Round, to_numpy_logits

BAND = 1e-6
RTOL = 1e-5
TRUNC_BAND = 1e-5
ALPHA_FLOOR = 1e-6


def run_gpu(rd: Round, *, K_max=64, stop_token=None, max_new=None, temperature=None, top_k=None, top_p=None):
    temp = rd.temperature if temperature is None else temperature
    out = api.verify(rd.target, rd.draft, rd.row_off, rd.draft_tokens, rd.uniforms, temp,
                     K_max=K_max, stop_token=stop_token, max_new=max_new, top_k=top_k, top_p=top_p,
                     diagnostics=True)
    torch.cuda.synchronize()
    return {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in out.__dict__.items()}


def sub_batch(rd: Round, reqs):
    """Host arrays of the sub-batch made of requests `reqs` (oracle inputs), with the maps
    from sub-batch rows back to the full batch."""
    row_off = rd.row_off.cpu().numpy()
    t_rows, d_rows, off = [], [], [0]
    for i in reqs:
        r0, r1 = int(row_off[i]), int(row_off[i + 1])
        K = r1 - r0 - 1
        t_rows.extend(range(r0, r1))
        d_rows.extend(range(r0 - i, r0 - i + K))
        off.append(off[-1] + K + 1)
    t_idx = torch.as_tensor(t_rows, dtype=torch.long, device=rd.target.device)
    d_idx = torch.as_tensor(d_rows, dtype=torch.long, device=rd.target.device)
    V = rd.target.shape[1]
    tgt = to_numpy_logits(rd.target.index_select(0, t_idx))
    if len(d_rows):
        drf = to_numpy_logits(rd.draft.index_select(0, d_idx))
    else:
        drf = np.zeros((0, V), tgt.dtype)
    return dict(target=tgt, draft=drf, row_off=np.asarray(off, np.int32),
                draft_tokens=rd.draft_tokens.cpu().numpy()[d_rows] if d_rows else np.zeros(0, np.int32),
                uniforms=rd.uniforms.cpu().numpy()[t_rows],
                temperature=rd.temperature.cpu().numpy()[list(reqs)],
                t_rows=np.asarray(t_rows), d_rows=np.asarray(d_rows, np.int64))


def run_oracle(rd: Round, reqs=None, **kw):
    reqs = list(range(rd.B)) if reqs is None else list(reqs)
    sb = sub_batch(rd, reqs)
    extra = {}
    for k in ("stop_token", "max_new", "top_k", "top_p"):
        if kw.get(k) is not None:
            extra[k] = np.asarray(kw[k].cpu().numpy() if isinstance(kw[k], torch.Tensor) else kw[k])[reqs]
    out = oracle.verify(sb["target"], sb["draft"], sb["row_off"], sb["draft_tokens"], sb["uniforms"],
                        sb["temperature"], K_max=kw.get("K_max", 64), **extra)
    return out, sb, reqs


@dataclass
class Report:
    requests: int = 0
    compared: int = 0
    near_boundary: int = 0
    near_matched: int = 0
    gpu_near_only: int = 0
    alpha_below_floor: int = 0
    mismatches: list = field(default_factory=list)
    alpha_max_rel: float = 0.0
    rho_max_rel: float = 0.0
    resid_max_rel: float = 0.0
    prob_max_rel: float = 0.0
    resid_cond_max: float = 0.0
    prob_cond_max: float = 0.0
    value_failures: list = field(default_factory=list)

    def ok(self):
        return not self.mismatches and not self.value_failures

    def summary(self):
        return (f"requests={self.requests} compared={self.compared} near_boundary={self.near_boundary} "
                f"(of which matched anyway: {self.near_matched}) gpu_near_only={self.gpu_near_only} "
                f"mismatches={len(self.mismatches)} value_failures={len(self.value_failures)} "
                f"alpha_rel={self.alpha_max_rel:.2e} rho_rel={self.rho_max_rel:.2e} "
                f"resid_rel={self.resid_max_rel:.2e} prob_rel={self.prob_max_rel:.2e} "
                f"alpha_below_floor={self.alpha_below_floor} resid_cond_max={self.resid_cond_max:.3g} "
                f"prob_cond_max={self.prob_cond_max:.3g}")

    def counts(self):
        return dict(requests=self.requests, compared=self.compared, near_boundary=self.near_boundary,
                    near_matched=self.near_matched, gpu_near_only=self.gpu_near_only,
                    mismatches=len(self.mismatches), value_failures=len(self.value_failures),
                    alpha_below_floor=self.alpha_below_floor, resid_cond_max=self.resid_cond_max,
                    prob_cond_max=self.prob_cond_max)

    def add(self, o: "Report"):
        """Accumulate another round's report (counts summed, maxima kept)."""
        for k in ("requests", "compared", "near_boundary", "near_matched", "gpu_near_only",
                  "alpha_below_floor"):
            setattr(self, k, getattr(self, k) + getattr(o, k))
        for k in ("alpha_max_rel", "rho_max_rel", "resid_max_rel", "prob_max_rel", "resid_cond_max",
                  "prob_cond_max"):
            setattr(self, k, max(getattr(self, k), getattr(o, k)))
        self.mismatches += o.mismatches
        self.value_failures += o.value_failures
        return self


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-300)


def oracle_near(orc, sb, k) -> bool:
    """Whether request k of the oracle's sub-batch has a draw inside the band, judged from the
    oracle's own margins only: an accept test it walked (u - rho within BAND), its frontier
    draw (u*Z within BAND of a CDF boundary, in units of Z), or a top-p cut (TRUNC_BAND)."""
    ro = sb["row_off"]
    r0, r1 = int(ro[k]), int(ro[k + 1])
    K = r1 - r0 - 1
    d0 = r0 - k
    if int(orc["req_status"][k]) != 0:
        return False
    tm = orc["trunc_margin"][r0:r1]
    if np.any(np.isfinite(tm) & (tm < TRUNC_BAND)):
        return True
    if float(sb["temperature"][k]) == 0.0:
        return False
    A_o = int(orc["accept_len"][k])
    for j in range(min(A_o + 1, K)):
        if abs(orc["accept_margin"][d0 + j]) < BAND:
            return True
    m_o = orc["sample_margin"][k]
    return bool(np.isfinite(m_o) and m_o < BAND)


def compare(gpu, orc, sb, reqs, full_row_off) -> Report:
    rep = Report(requests=len(reqs))
    ro = sb["row_off"]
    for k, i in enumerate(reqs):
        r0, r1 = int(ro[k]), int(ro[k + 1])
        K = r1 - r0 - 1
        d0 = r0 - k
        g_r0 = int(full_row_off[i])
        g_d0 = g_r0 - i
        st_o = int(orc["req_status"][k])
        st_g = int(gpu["req_status"][i])
        if st_o != st_g:
            rep.mismatches.append((i, "status", st_g, st_o))
            continue
        if st_o != 0:
            rep.compared += 1
            if not (gpu["out_tokens"][g_r0:g_r0 + K + 1] == -1).all() or gpu["n_emitted"][i] != 0:
                rep.mismatches.append((i, "bad request emitted", gpu["out_tokens"][g_r0:g_r0 + K + 1]))
            # its draft rows carry no result either (NaN, as the oracle's)
            if K > 0 and not np.isnan(gpu["alpha_rows"][g_d0:g_d0 + K]).all():
                rep.mismatches.append((i, "bad request alpha", gpu["alpha_rows"][g_d0:g_d0 + K]))
            continue
        greedy = float(sb["temperature"][k]) == 0.0
        tm = orc["trunc_margin"][r0:r1]
        if np.any(np.isfinite(tm) & (tm < TRUNC_BAND)):
            # a top-p cut at the boundary: the two sides may keep different sets
            rep.near_boundary += 1
            continue
        # values: alpha and rho for every draft row, residual mass where the kernel formed it
        for j in range(K):
            a_o, a_g = orc["alpha"][d0 + j], gpu["alpha_rows"][g_d0 + j]
            if a_o >= ALPHA_FLOOR:
                ra = float(_rel(a_g, a_o))
                rep.alpha_max_rel = max(rep.alpha_max_rel, ra)
                if ra > RTOL:
                    rep.value_failures.append((i, j, "alpha", a_g, a_o))
            else:
                rep.alpha_below_floor += 1
                if abs(a_g - a_o) > RTOL * ALPHA_FLOOR:
                    rep.value_failures.append((i, j, "alpha(below floor)", a_g, a_o))
            if not greedy:
                rho_o, rho_g = orc["rho"][d0 + j], gpu["rho_rows"][g_d0 + j]
                # the ratio is reported in float32: values outside its normal range are not compared
                if np.isfinite(rho_o) and 1e-30 < rho_o < 1e30:
                    rr = float(_rel(rho_g, rho_o))
                    rep.rho_max_rel = max(rep.rho_max_rel, rr)
                    if rr > RTOL:
                        rep.value_failures.append((i, j, "rho", rho_g, rho_o))
                z_g = gpu["resid_rows"][g_d0 + j]
                if z_g >= 0:
                    z_o = orc["resid_mass"][d0 + j]
                    err = abs(z_g - z_o)
                    if z_o > 0:
                        rep.resid_max_rel = max(rep.resid_max_rel, err / z_o)
                        rep.resid_cond_max = max(rep.resid_cond_max, orc["resid_scale"][d0 + j] / z_o)
                    if err > RTOL * z_o:
                        rep.value_failures.append((i, j, "resid", z_g, z_o))
        # decisions: skip requests the oracle places inside the band
        A_o, A_g = int(orc["accept_len"][k]), int(gpu["accept_len"][i])
        near = oracle_near(orc, sb, k)
        if not near and not greedy:
            m_g = gpu["frontier_margin"][i]
            if np.isfinite(m_g) and m_g < BAND:
                rep.gpu_near_only += 1
        n_o, n_g = int(orc["n_emitted"][k]), int(gpu["n_emitted"][i])
        t_o = orc["out_tokens"][r0:r1]
        t_g = gpu["out_tokens"][g_r0:g_r0 + K + 1]
        same = A_o == A_g and n_o == n_g and np.array_equal(t_o, t_g)
        if near:
            rep.near_boundary += 1
            rep.near_matched += int(same)
            continue
        rep.compared += 1
        if not same:
            rep.mismatches.append((i, "tokens", A_g, A_o, t_g.tolist(), t_o.tolist()))
            continue
        if int(orc["fallback"][k]) != int(gpu["fallback"][i]):
            rep.mismatches.append((i, "fallback", gpu["fallback"][i], orc["fallback"][k]))
        p_o, p_g = orc["sample_prob"][k], gpu["frontier_prob"][i]
        if np.isfinite(p_o):
            rp = float(_rel(p_g, p_o))
            rep.prob_max_rel = max(rep.prob_max_rel, rp)
            rep.prob_cond_max = max(rep.prob_cond_max, float(orc["sample_cond"][k]))
            if rp > RTOL:
                rep.value_failures.append((i, "frontier_prob", p_g, p_o))
    return rep


def check_round(rd: Round, reqs=None, **kw) -> Report:
    gpu = run_gpu(rd, K_max=kw.get("K_max", 64), stop_token=kw.get("stop_token"), max_new=kw.get("max_new"),
                  top_k=kw.get("top_k"), top_p=kw.get("top_p"))
    orc, sb, reqs = run_oracle(rd, reqs, **kw)
    return compare(gpu, orc, sb, reqs, rd.row_off.cpu().numpy())
