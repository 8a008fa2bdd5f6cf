"""Seeded synthetic workloads shaped like the verify steps the pages describe.

This module only builds inputs: logits, drafts, sampling parameters and
confidences.  It holds none of the verify arithmetic (no target distribution,
acceptance, resampling or planning), so the CUDA path and the CPU oracle can
both consume what it makes without sharing any step of the method; the
drafter below samples its own tokens with torch primitives, and neither side
runs it.

Workloads (sizes as the benchmark configurations state them):

* ``tiny``        4 requests, K=4 (5 target rows each), vocab 1024, fp32
                  logits N(0, 2^2), draft = target + N(0, 1); requests 0-1
                  greedy, 2-3 at T=0.7, top-k 20, top-p 0.9.
* ``medium``      32 x K=5, vocab 151,936, bf16 N(0, 3^2) with one token per
                  row planted at 30% of the row's softmax mass; draft
                  correlated rho = 0.8; T=1.0, top-p 0.95, no top-k.
* ``large``       128 x 8-token blocks (K=7 drafts + 1 bonus row = 1024
                  target rows), vocab 248,320, bf16 N(0, 3^2) whose 32 largest
                  entries per row get + 3|t_3| (Student-t, 3 dof); draft
                  rho = 0.8; T=0.6, top-k 20, top-p 0.95.
* ``greedy_wide`` 512 x 8-token blocks (4096 rows), vocab 129,280, bf16
                  N(0, 2^2); greedy only; the drafts hit the planted top token
                  with per-position probability 0.74/0.49/0.30/0.18/0.10/0.06/
                  0.04; 1% of rows carry an exact duplicate of the top value.
* ``ragged``      256 requests drafting 16-token blocks; confidence
                  Beta(4, 2) * 0.85^i; budget 2048 tokens, bucket 2048; vocab
                  248,320 bf16 N(0, 3^2); even requests greedy, odd ones
                  T ~ U[0.3, 1.2], top-p 0.9.

The simulated drafter draws each drafted token from its own draft row, as the
configurations state ("draft tokens sampled from the draft softmax"; drafts
distributed as q): softmax(l / T) over the request's top-k, cut to its top-p
(the crossing token kept), in fp32 with torch primitives and the workload's
seeded generator; a greedy request's drafter samples the plain softmax at
T = 1.  Neither side of the comparison runs this code: the CUDA path and the
oracle both read only the tokens it drew.  ``drafter="rank"`` keeps the older
stand-in, the token at rank rho of the draft row (rho in {0, 1, 2, 3} with
probabilities 0.55, 0.25, 0.13, 0.07; ``torch.topk`` ordering); the verify
step is defined for any proposal.  ``greedy_wide`` states its own drafter
(per-position match probabilities) and keeps it.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

NAMES = ("tiny", "medium", "large", "greedy_wide", "ragged")
SEEDS = {"tiny": 1, "medium": 2, "large": 3, "greedy_wide": 4, "ragged": 5}
RANK_PROBS = (0.55, 0.25, 0.13, 0.07)
GREEDY_WIDE_MATCH = (0.74, 0.49, 0.30, 0.18, 0.10, 0.06, 0.04)


@dataclasses.dataclass
class Workload:
    name: str
    layout: str                      # "chain" (uniform) or "ragged"
    n: int                           # requests
    K: int                           # drafted positions per request
    V: int                           # vocabulary
    dtype: torch.dtype               # logits dtype
    target: torch.Tensor             # chain: [n, K+1, V]; ragged: block layout [n, K+1, V]
    draft: Optional[torch.Tensor]    # [n, K, V] or None when every request is greedy
    draft_tokens: torch.Tensor       # [n, K] int32
    temperature: torch.Tensor        # [n] fp32, 0 = greedy
    top_k: torch.Tensor              # [n] int32, <= 0 = off
    top_p: torch.Tensor              # [n] fp32, >= 1 = off
    seed: int = 0                    # key of the method's Philox uniforms
    conf: Optional[torch.Tensor] = None   # ragged: [n, K] fp32 per-position confidence
    budget: int = 0
    bucket: int = 0

    @property
    def target_rows(self) -> int:
        return self.n * (self.K + 1)

    def to(self, device) -> "Workload":
        out = dataclasses.replace(self)
        for f in ("target", "draft", "draft_tokens", "temperature", "top_k", "top_p", "conf"):
            t = getattr(self, f)
            if t is not None:
                setattr(out, f, t.to(device))
        return out


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _correlated(target32, g, rho=0.8, std=3.0):
    noise = torch.randn(target32.shape, generator=g, device=target32.device) * std
    return rho * target32 + (1.0 - rho * rho) ** 0.5 * noise


def _rank_drafts(draft32, g, n, K):
    """Drafter stand-in: the token at rank rho of each draft row."""
    if n * K == 0:
        return torch.zeros((n, K), dtype=torch.int32, device=draft32.device)
    top4 = torch.topk(draft32.reshape(n * K, -1), 4, dim=-1).indices
    probs = torch.tensor(RANK_PROBS, device=draft32.device)
    rho = torch.multinomial(probs.expand(n * K, 4), 1, generator=g)
    return top4.gather(1, rho).reshape(n, K).to(torch.int32)


def _sampled_drafts(draft32, T, top_k, top_p, g, chunk_rows=128):
    """Drafter: every drafted token drawn from its draft row's distribution at
    the request's settings (see the module docstring).  T, top_k, top_p: [n]."""
    n, K, V = draft32.shape
    dev = draft32.device
    out = torch.empty((n * K,), dtype=torch.int64, device=dev)
    x = draft32.reshape(n * K, V)
    t_row = torch.where(T > 0, T, torch.ones_like(T)).repeat_interleave(K).float()
    k_row = torch.where((T > 0) & (top_k > 0) & (top_k < V), top_k, torch.full_like(top_k, V)).repeat_interleave(K)
    p_row = torch.where(T > 0, top_p, torch.ones_like(top_p)).repeat_interleave(K).float()
    rank = torch.arange(V, device=dev)
    for r0 in range(0, n * K, chunk_rows):
        r1 = min(n * K, r0 + chunk_rows)
        vals, idx = torch.sort(x[r0:r1], dim=-1, descending=True, stable=True)
        e = torch.exp((vals - vals[:, :1]) / t_row[r0:r1, None])
        e = torch.where(rank[None, :] < k_row[r0:r1, None], e, torch.zeros_like(e))
        cum = torch.cumsum(e, dim=-1)
        before = cum - e                       # mass ahead of each token in sorted order
        keep = before < p_row[r0:r1, None] * cum[:, -1:]
        w = torch.where(keep, e, torch.zeros_like(e))
        pick = torch.multinomial(w, 1, generator=g)
        out[r0:r1] = idx.gather(1, pick).squeeze(1)
    return out.reshape(n, K).to(torch.int32)


def _drafts(drafter, draft32, T, top_k, top_p, g, n, K):
    if drafter == "rank":
        return _rank_drafts(draft32, g, n, K)
    if drafter != "q":
        raise ValueError(f"unknown drafter {drafter!r}: 'q' or 'rank'")
    if n * K == 0:
        return torch.zeros((n, K), dtype=torch.int32, device=draft32.device)
    return _sampled_drafts(draft32, T, top_k, top_p, g)


def make(name: str, device="cpu", scale: Optional[dict] = None, drafter: str = "q") -> Workload:
    """Build workload ``name`` on ``device``.

    ``scale`` overrides sizes (keys n, K, V) to make a smaller case with the
    same value distributions, for tests that the oracle must finish quickly.
    ``drafter``: "q" (drafts drawn from the draft distribution, the default)
    or "rank" (the rank-rho stand-in); greedy_wide keeps its own drafter.
    """
    if name not in NAMES:
        raise ValueError(f"unknown workload {name!r}; choose from {NAMES}")
    scale = scale or {}
    g = _gen(device, SEEDS[name])
    if name == "tiny":
        n, K, V = scale.get("n", 4), scale.get("K", 4), scale.get("V", 1024)
        tgt = torch.randn((n, K + 1, V), generator=g, device=device) * 2.0
        drf = tgt[:, :K, :] + torch.randn((n, K, V), generator=g, device=device)
        T = torch.tensor([0.0, 0.0, 0.7, 0.7] * ((n + 3) // 4), device=device)[:n]
        tk = torch.tensor([0, 0, 20, 20] * ((n + 3) // 4), device=device, dtype=torch.int32)[:n]
        tp = torch.tensor([1.0, 1.0, 0.9, 0.9] * ((n + 3) // 4), device=device)[:n]
        toks = _drafts(drafter, drf, T, tk, tp, g, n, K)
        return Workload(name, "chain", n, K, V, torch.float32, tgt.contiguous(), drf.contiguous(), toks,
                        T.float(), tk, tp.float())
    if name == "medium":
        n, K, V = scale.get("n", 32), scale.get("K", 5), scale.get("V", 151_936)
        tgt = torch.randn((n, K + 1, V), generator=g, device=device) * 3.0
        # Plant one token per row at 30% of the row's T=1 softmax mass:
        # l* = log(0.3 / 0.7 * sum over the other tokens of exp(l)).
        star = torch.randint(0, V, (n, K + 1, 1), generator=g, device=device)
        tgt.scatter_(2, star, torch.full_like(star, -float("inf"), dtype=tgt.dtype))
        lse = torch.logsumexp(tgt, dim=-1, keepdim=True)
        tgt.scatter_(2, star, lse + torch.log(torch.tensor(0.3 / 0.7, device=device)))
        drf = _correlated(tgt[:, :K, :], g)
        tgt16, drf16 = tgt.to(torch.bfloat16), drf.to(torch.bfloat16)
        T, tk, tp = (torch.full((n,), 1.0, device=device), torch.zeros(n, dtype=torch.int32, device=device),
                     torch.full((n,), 0.95, device=device))
        toks = _drafts(drafter, drf16.float(), T, tk, tp, g, n, K)
        return Workload(name, "chain", n, K, V, torch.bfloat16, tgt16.contiguous(), drf16.contiguous(), toks,
                        T, tk, tp)
    if name == "large":
        n, K, V = scale.get("n", 128), scale.get("K", 7), scale.get("V", 248_320)
        tgt = torch.randn((n, K + 1, V), generator=g, device=device) * 3.0
        top = torch.topk(tgt, min(32, V), dim=-1).indices
        # Student-t with 3 dof: N(0,1) / sqrt(chi2_3 / 3).
        z = torch.randn(top.shape, generator=g, device=device)
        chi = (torch.randn(top.shape + (3,), generator=g, device=device) ** 2).sum(-1)
        t3 = z / torch.sqrt(chi / 3.0)
        tgt.scatter_add_(2, top, 3.0 * t3.abs())
        drf = _correlated(tgt[:, :K, :], g)
        tgt16, drf16 = tgt.to(torch.bfloat16), drf.to(torch.bfloat16)
        T, tk, tp = (torch.full((n,), 0.6, device=device), torch.full((n,), 20, dtype=torch.int32, device=device),
                     torch.full((n,), 0.95, device=device))
        toks = _drafts(drafter, drf16.float(), T, tk, tp, g, n, K)
        return Workload(name, "chain", n, K, V, torch.bfloat16, tgt16.contiguous(), drf16.contiguous(), toks,
                        T, tk, tp)
    if name == "greedy_wide":
        n, K, V = scale.get("n", 512), scale.get("K", 7), scale.get("V", 129_280)
        tgt = torch.randn((n, K + 1, V), generator=g, device=device) * 2.0
        rows = n * (K + 1)
        flat = tgt.view(rows, V)
        # Planted top token: 16.0 is 8 standard deviations above the bulk.
        top_idx = torch.randint(0, V, (rows,), generator=g, device=device)
        flat[torch.arange(rows, device=device), top_idx] = 16.0
        # 1% of rows: an exact duplicate of the top value at another index,
        # above the planted one in half of them and below it in the other half.
        tie = torch.rand(rows, generator=g, device=device) < 0.01
        upper = torch.rand(rows, generator=g, device=device) < 0.5
        upper = torch.where(top_idx == V - 1, torch.zeros_like(upper), upper)
        upper = torch.where(top_idx == 0, torch.ones_like(upper), upper)
        u = torch.rand(rows, generator=g, device=device)
        above = top_idx + 1 + (u * (V - 1 - top_idx).float()).long().clamp(min=0)
        below = (u * top_idx.float()).long()
        dup = torch.where(upper, above.clamp(max=V - 1), below.clamp(max=V - 1))
        tie = tie & (dup != top_idx)
        ti = torch.nonzero(tie).flatten()
        flat[ti, dup[ti]] = 16.0
        tgt16 = tgt.to(torch.bfloat16)
        # Drafts: the planted token with probability p_i; otherwise a uniform
        # other token, or, in half of the tie rows, the duplicate.
        pm = torch.tensor(GREEDY_WIDE_MATCH[:K] + (0.02,) * max(0, K - len(GREEDY_WIDE_MATCH)), device=device)
        hit = torch.rand((n, K), generator=g, device=device) < pm[:K]
        top_nk = top_idx.view(n, K + 1)[:, :K]
        dup_nk = dup.view(n, K + 1)[:, :K]
        tie_nk = tie.view(n, K + 1)[:, :K]
        other = (top_nk + torch.randint(1, V, (n, K), generator=g, device=device)) % V
        pick_dup = tie_nk & (torch.rand((n, K), generator=g, device=device) < 0.5)
        miss = torch.where(pick_dup, dup_nk, other)
        toks = torch.where(hit, top_nk, miss).to(torch.int32)
        return Workload(name, "chain", n, K, V, torch.bfloat16, tgt16.contiguous(), None, toks,
                        torch.zeros(n, device=device), torch.zeros(n, dtype=torch.int32, device=device),
                        torch.ones(n, device=device))
    # ragged
    n, K, V = scale.get("n", 256), scale.get("K", 16), scale.get("V", 248_320)
    budget = scale.get("budget", 2048)
    bucket = scale.get("bucket", budget)
    cpu_g = _gen("cpu", SEEDS[name])
    # Beta(4, 2) via two gammas drawn from uniforms: -log(prod of 4 U) and -log(prod of 2 U).
    u4 = torch.rand((n, K, 4), generator=cpu_g)
    u2 = torch.rand((n, K, 2), generator=cpu_g)
    ga, gb = -torch.log(u4).sum(-1), -torch.log(u2).sum(-1)
    b = ga / (ga + gb)
    decay = 0.85 ** torch.arange(K, dtype=torch.float32)
    conf = (b * decay).to(torch.float32).to(device)
    tgt = torch.randn((n, K + 1, V), generator=g, device=device) * 3.0
    drf = _correlated(tgt[:, :K, :], g)
    tgt16, drf16 = tgt.to(torch.bfloat16), drf.to(torch.bfloat16)
    odd = (torch.arange(n, device=device) % 2) == 1
    Tr = 0.3 + 0.9 * torch.rand(n, generator=g, device=device)
    T = torch.where(odd, Tr, torch.zeros_like(Tr)).float()
    tk = torch.zeros(n, dtype=torch.int32, device=device)
    tp = torch.where(odd, torch.full_like(Tr, 0.9), torch.ones_like(Tr)).float()
    toks = _drafts(drafter, drf16.float(), T, tk, tp, g, n, K)
    return Workload(name, "ragged", n, K, V, torch.bfloat16, tgt16.contiguous(), drf16.contiguous(), toks,
                    T, tk, tp, conf=conf, budget=budget, bucket=bucket)


def pack_rows(block: torch.Tensor, qo_indptr, verify_lens, bucket: int) -> torch.Tensor:
    """Lay request r's first verify_lens[r] + 1 rows of a block-layout tensor
    [n, K+1, V] at rows qo_indptr[r] ... of a [bucket, V] tensor; padding rows
    past the last window are left zero.  This stands in for a target forward
    that emits logits for the packed windows only."""
    n, _, V = block.shape
    out = torch.zeros((bucket, V), dtype=block.dtype, device=block.device)
    qo = [int(x) for x in qo_indptr]
    vl = [int(x) for x in verify_lens]
    for r in range(n):
        out[qo[r]:qo[r] + vl[r] + 1] = block[r, :vl[r] + 1]
    return out


def random_case(seed: int, n: int, K: int, V: int, dtype=torch.bfloat16, device="cpu", std: float = 3.0,
                mode: str = "mixed") -> Workload:
    """A small random uniform-layout case for property and parity tests.

    mode: "mixed" draws per-request (T, top-k, top-p) from a menu that covers
    greedy, top-k only, top-p only, both, neither, k in {1, 2, 20, V-1, V};
    "topk" keeps k <= 20; "full" turns top-k off.
    """
    g = _gen(device, 1000 + seed)
    tgt = torch.randn((n, K + 1, V), generator=g, device=device) * std
    drf = _correlated(tgt[:, :K, :], g, std=std)
    if dtype == torch.bfloat16:
        tgt, drf = tgt.to(dtype), drf.to(dtype)
    toks = _rank_drafts(drf.float(), g, n, K) if V >= 4 else torch.randint(0, V, (n, K), generator=g,
                                                                           device=device).to(torch.int32)
    menu_T = [0.0, 0.3, 0.7, 1.0, 1.5]
    menu_k = {"mixed": [0, 1, 2, 20, V - 1, V, 64], "topk": [1, 2, 5, 20], "full": [0]}[mode]
    menu_p = [1.0, 0.9, 0.5, 0.1]
    pick = lambda menu: torch.tensor(menu, device=device)[torch.randint(0, len(menu), (n,), generator=g,
                                                                          device=device)]
    T = pick(menu_T).float()
    if mode != "mixed":
        T = torch.where(T == 0, torch.full_like(T, 0.8), T)
    return Workload(f"random{seed}", "chain", n, K, V, dtype, tgt.contiguous(), drf.contiguous(), toks, T,
                    pick(menu_k).to(torch.int32), pick(menu_p).float())
