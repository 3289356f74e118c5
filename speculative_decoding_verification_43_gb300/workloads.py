"""Seeded synthetic inputs for the verifier: the workloads and their generators.

This module holds none of the verifier's arithmetic. It produces what a serving system hands
the verifier: target logits, draft logits, the drafter's tokens and the verifier's uniforms.
Both the CUDA path and the oracle consume the same arrays it returns.

The drafter samples each draft token from its own distribution q = softmax(z_draft / T); it
does so here with the Gumbel-max trick (argmax of z/T + Gumbel noise), which is the drafter's
sampler, not the verifier's, and involves no normalisation. At T = 0 the drafter proposes its
argmax.

Uniforms are float64 values k / 2^53 from numpy's Philox counter-based generator keyed by
(seed, round): slot j < K_i of request i is its accept draw for draft j, slot K_i the draw of
the frontier token (SDCP Rule 2 keeps these two purposes apart).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    V: int
    dtype: torch.dtype
    temperature: float
    logits: str                  # "normal" (N(0, sigma)) or "zipf" (-1.1 ln(rank) + N(0, 1))
    sigma: float                 # target std for "normal"
    draft_sigma: float | tuple   # std of the draft's noise, or (lo, hi) drawn per request
    K: str                       # "fixed:<k>", "uniform:<lo>:<hi>", "schedule"
    rounds: int = 1
    prefix_len: int = 4096       # P_i for compaction
    page_size: int = 16
    note: str = ""

    def k_values(self, seed: int) -> np.ndarray:
        rng = np.random.default_rng([seed, 0x4B])
        kind, *args = self.K.split(":")
        if kind == "fixed":
            return np.full(self.B, int(args[0]), np.int64)
        if kind == "uniform":
            return rng.integers(int(args[0]), int(args[1]) + 1, size=self.B)
        if kind == "schedule":
            # a quarter of the batch drafts 2, a quarter 1, half does not draft
            ks = np.array([2] * (self.B // 4) + [1] * (self.B // 4) + [0] * (self.B - 2 * (self.B // 4)))
            return rng.permutation(ks)
        raise ValueError(self.K)

    def rows(self, seed: int) -> int:
        return int((self.k_values(seed) + 1).sum())

    def bytes_per_round(self, seed: int) -> int:
        k = self.k_values(seed)
        esize = 2 if self.dtype == torch.bfloat16 else 4
        return int((2 * k + 1).sum()) * self.V * esize


WORKLOADS = {
    "c1": Workload("c1", B=1, V=1000, dtype=torch.float32, temperature=1.0, logits="normal",
                   sigma=2.0, draft_sigma=0.5, K="fixed:4", rounds=100,
                   note="B=1, gamma=4, V=1000, fp32 N(0,2), draft noise N(0,0.5), T=1"),
    "c2": Workload("c2", B=8, V=32000, dtype=torch.bfloat16, temperature=1.0, logits="normal",
                   sigma=3.0, draft_sigma=1.0, K="fixed:5", rounds=1000,
                   note="B=8, gamma=5, V=32000, bf16 N(0,3), draft noise N(0,1), T=1"),
    "c3": Workload("c3", B=64, V=128256, dtype=torch.bfloat16, temperature=0.7, logits="zipf",
                   sigma=1.0, draft_sigma=0.8, K="uniform:0:7",
                   note="B=64 ragged K in {0..7}, V=128256, bf16 Zipf head, draft noise N(0,0.8), T=0.7"),
    "c4": Workload("c4", B=256, V=151936, dtype=torch.float32, temperature=1.0, logits="normal",
                   sigma=1.0, draft_sigma=(0.2, 2.0), K="fixed:3",
                   note="B=256, gamma=3, V=151936, fp32 N(0,1), draft noise sigma~U(0.2,2) per request, "
                        "compaction over 4096-token prefixes"),
    "c5": Workload("c5", B=512, V=256000, dtype=torch.bfloat16, temperature=1.0, logits="zipf",
                   sigma=1.0, draft_sigma=0.8, K="schedule",
                   note="B=512, K schedule {2:25%,1:25%,0:50%}, V=256000, bf16 Zipf, T=1, alpha -> gamma"),
}


def scaled(wl: Workload, *, B: int | None = None, V: int | None = None, K: str | None = None,
           name: str | None = None) -> Workload:
    """The same recipe at another size (parity tests run the oracle on smaller batches)."""
    d = dict(wl.__dict__)
    if B is not None:
        d["B"] = B
    if V is not None:
        d["V"] = V
    if K is not None:
        d["K"] = K
    d["name"] = name or f"{wl.name}-scaled"
    return Workload(**d)


def uniforms(seed: int, rnd: int, n: int) -> np.ndarray:
    """n float64 uniforms in [0, 1) with 53 random bits, from Philox keyed by (seed, round)."""
    g = np.random.Generator(np.random.Philox(key=[seed & 0xFFFFFFFFFFFFFFFF, rnd]))
    return g.random(n)


@dataclass
class Round:
    target: torch.Tensor        # [T][V]
    draft: torch.Tensor         # [T-B][V]
    row_off: torch.Tensor       # [B+1] int32
    draft_tokens: torch.Tensor  # [T-B] int32
    uniforms: torch.Tensor      # [T] float64
    temperature: torch.Tensor   # [B] float32
    K: np.ndarray
    extra: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.row_off.numel() - 1

    @property
    def T(self):
        return self.target.shape[0]


def _zipf_logits(n_rows: int, V: int, gen: torch.Generator, device) -> torch.Tensor:
    """logit = -1.1 ln(rank) + N(0, 1), rank a fresh random permutation of 1..V per row."""
    out = torch.empty(n_rows, V, dtype=torch.float32, device=device)
    step = max(1, (1 << 26) // V)  # bound the temporaries of the permutation
    base = -1.1 * torch.log(torch.arange(1, V + 1, dtype=torch.float32, device=device))
    for s in range(0, n_rows, step):
        e = min(n_rows, s + step)
        perm = torch.argsort(torch.rand(e - s, V, generator=gen, device=device), dim=1)
        out[s:e] = base[perm]
        out[s:e] += torch.randn(e - s, V, generator=gen, device=device)
    return out


def make_round(wl: Workload, seed: int = 0, rnd: int = 0, device="cpu", K=None,
               temperature=None) -> Round:
    """One round of wl's workload: seed fixes the batch shape, (seed, rnd) the values."""
    device = torch.device(device)
    Ks = np.asarray(wl.k_values(seed) if K is None else K, np.int64)
    B = len(Ks)
    V = wl.V
    row_off = np.concatenate([[0], np.cumsum(Ks + 1)]).astype(np.int32)
    T = int(row_off[-1])
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1_000_003 + rnd) & 0x7FFFFFFFFFFFFFFF)

    if wl.logits == "zipf":
        tz = _zipf_logits(T, V, gen, device)
    else:
        tz = torch.randn(T, V, generator=gen, device=device) * wl.sigma

    # the draft row of position j is the target row of position j plus noise
    draft_rows = np.concatenate([np.arange(row_off[i], row_off[i] + Ks[i]) for i in range(B)]).astype(np.int64) \
        if T > B else np.zeros(0, np.int64)
    req_of_draft = np.repeat(np.arange(B), Ks)
    if isinstance(wl.draft_sigma, tuple):
        lo, hi = wl.draft_sigma
        sig_req = torch.rand(B, generator=gen, device=device) * (hi - lo) + lo
    else:
        sig_req = torch.full((B,), float(wl.draft_sigma), device=device)
    idx = torch.as_tensor(draft_rows, device=device)
    sig = sig_req[torch.as_tensor(req_of_draft, device=device)].unsqueeze(1) if T > B else None
    nd = T - B
    dz = torch.empty(nd, V, dtype=torch.float32, device=device)
    step = max(1, (1 << 26) // V)
    for s in range(0, nd, step):
        e = min(nd, s + step)
        dz[s:e] = tz[idx[s:e]] + torch.randn(e - s, V, generator=gen, device=device) * sig[s:e]

    target = tz.to(wl.dtype).contiguous()
    draft = dz.to(wl.dtype).contiguous()
    del tz, dz

    Tval = wl.temperature if temperature is None else temperature
    temp = torch.full((B,), float(Tval), dtype=torch.float32, device=device) \
        if not isinstance(Tval, (list, np.ndarray, torch.Tensor)) else \
        torch.as_tensor(np.asarray(Tval, np.float32), device=device)

    # the drafter's tokens: samples from q = softmax(draft / T) (Gumbel-max), argmax at T = 0
    toks = torch.empty(nd, dtype=torch.int32, device=device)
    tq = temp[torch.as_tensor(req_of_draft, device=device)] if nd else None
    for s in range(0, nd, step):
        e = min(nd, s + step)
        z = draft[s:e].float()
        t = tq[s:e].unsqueeze(1)
        u = torch.rand(e - s, V, generator=gen, device=device).clamp_(min=1e-38)
        g = -torch.log(-torch.log(u))
        score = torch.where(t > 0, z / t.clamp(min=1e-30) + g, z)
        toks[s:e] = score.argmax(dim=1).to(torch.int32)

    u = torch.as_tensor(uniforms(seed, rnd, T), dtype=torch.float64, device=device)
    return Round(target=target, draft=draft, row_off=torch.as_tensor(row_off, device=device),
                 draft_tokens=toks, uniforms=u, temperature=temp, K=Ks)


def make_compaction_inputs(rd: Round, prefix_len: int, page_size: int, seed: int = 0):
    """Prefix lengths, candidate KV rows and a shuffled page table for spec_compact."""
    B, T = rd.B, rd.T
    device = rd.target.device
    rng = np.random.default_rng([seed, 0xC0])
    P = np.full(B, prefix_len, np.int32)
    max_pos = int(P.max()) + int(rd.K.max()) + 1 if B else 1
    nblk = (max_pos + page_size - 1) // page_size
    block_table = rng.permutation(B * nblk).astype(np.int32).reshape(B, nblk)
    cand = (rng.permutation(max(T - B, 1)).astype(np.int32) + B * nblk * page_size)[: max(T - B, 0)]
    to = lambda a: torch.as_tensor(a, device=device)
    return dict(prefix_len=to(P), cand_kv_rows=to(cand), block_table=to(block_table), page_size=page_size)


def to_numpy_logits(t: torch.Tensor) -> np.ndarray:
    """Host copy for the oracle: float32 as is, bfloat16 as its raw 16-bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
