"""Full-row resample (kept sets above 32 tokens) against the oracle, through
sv_verify_chain (needs a GB300).

Rows here span several 8,192-element chunks of the resample kernel, so
the cases reach its combine step: tie groups at a partially kept cutoff that
run across chunks (for p and for q), cutoffs at zero (-0 and +0 tied) and
below it, residuals that vanish, bonus tokens, rows too unaligned for
16-byte vector loads, and whole-row kept sets (top-p 1, no top-k) whose
small-magnitude keys get per-key weights.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_rows_gb300 import build as sv_build
from speculative_decoding_verification_rows_gb300 import sv, workloads
from tests.compare import compare_verify
from tests.conftest import np_logits

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv_build.build()
    sv.load()


def _check(tgt, drf, toks, T, tk, tp, seed):
    n, K = toks.shape
    V = tgt.shape[-1]
    g = sv.verify_chain(tgt.to(DEV), drf.to(DEV), toks.to(DEV), T.to(DEV), tk.to(DEV), tp.to(DEV), seed=seed)
    torch.cuda.synchronize()
    o = oracle.verify_chain(np_logits(tgt), np_logits(drf), toks.numpy(), T.numpy(), tk.numpy(), tp.numpy(),
                            seed=seed)
    compare_verify(o, g, toks.numpy(), np.full(n, K), V)
    return o, g


def _few_values(rng, shape, vals, probs):
    return torch.from_numpy(rng.choice(np.array(vals, np.float32), shape, p=probs)).to(torch.bfloat16)


@pytest.mark.parametrize("seed", range(3))
def test_tie_groups_across_chunks(seed):
    # few distinct logits: p's and q's cutoffs fall inside tie groups of
    # thousands of tokens spread over every chunk of the row
    rng = np.random.default_rng(40 + seed)
    n, K, V = 24, 3, 60_000
    tgt = _few_values(rng, (n, K + 1, V), [0.0, 0.5, 1.0, 1.5, 2.0], [0.4, 0.3, 0.15, 0.1, 0.05])
    drf = _few_values(rng, (n, K, V), [0.0, 0.5, 1.0, 1.5, 2.0], [0.3, 0.3, 0.2, 0.1, 0.1])
    toks = torch.from_numpy(rng.integers(0, V, (n, K)).astype(np.int32))
    T = torch.from_numpy(rng.choice([0.7, 1.0, 1.3], n).astype(np.float32))
    tk = torch.zeros(n, dtype=torch.int32)
    tp = torch.from_numpy(rng.choice([0.2, 0.45, 0.7, 0.9], n).astype(np.float32))
    o, g = _check(tgt, drf, toks, T, tk, tp, seed)
    assert (o["accept_len"] < K).sum() > n // 4          # residual resamples happened


@pytest.mark.parametrize("seed", range(3))
def test_tie_groups_at_zero_and_below(seed):
    # few distinct logits around zero, -0 and +0 among them: the cutoffs fall
    # at zero (both zeros in one tie group) or at a negative value
    rng = np.random.default_rng(90 + seed)
    n, K, V = 24, 3, 40_000
    vals = [-1.5, -1.0, -0.5, -0.0, 0.0, 0.5]
    tgt = _few_values(rng, (n, K + 1, V), vals, [0.1, 0.15, 0.2, 0.2, 0.2, 0.15])
    drf = _few_values(rng, (n, K, V), vals, [0.15, 0.15, 0.15, 0.2, 0.2, 0.15])
    toks = torch.from_numpy(rng.integers(0, V, (n, K)).astype(np.int32))
    T = torch.from_numpy(rng.choice([0.7, 1.0, 1.3], n).astype(np.float32))
    tk = torch.zeros(n, dtype=torch.int32)
    tp = torch.from_numpy(rng.choice([0.3, 0.5, 0.75, 0.95], n).astype(np.float32))
    o, g = _check(tgt, drf, toks, T, tk, tp, seed)
    assert (o["accept_len"] < K).sum() > n // 4


@pytest.mark.parametrize("seed", range(2))
def test_multi_chunk_rows(seed):
    w = workloads.random_case(60 + seed, 16, 4, 70_000, device="cpu", mode="full")
    tp = torch.from_numpy(np.random.default_rng(seed).choice([0.5, 0.9, 0.97], 16).astype(np.float32))
    _check(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, tp, seed)


@pytest.mark.parametrize("seed", range(2))
def test_whole_row_kept_sets(seed):
    # no top-k and top-p 1: every finite logit is kept, from the most negative
    # binade up, through the small magnitudes around zero
    w = workloads.random_case(70 + seed, 8, 3, 70_000, device="cpu", mode="full")
    tp = torch.ones(8)
    o, g = _check(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, tp, 7 + seed)
    assert (g.row_status.cpu().numpy() & sv.ROW_UNSUPPORTED == 0).all()


@pytest.mark.parametrize("V", [50_001, 33_333])
def test_unaligned_rows(V):
    w = workloads.random_case(80, 6, 3, V, device="cpu", mode="full")
    tp = torch.full((6,), 0.9)
    _check(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, tp, 3)


def test_bonus_after_full_acceptance():
    # draft rows equal to the target rows: every draft is accepted and the
    # bonus token is drawn from p over the whole row
    rng = np.random.default_rng(9)
    n, K, V = 12, 2, 70_000
    tgt = torch.from_numpy(rng.normal(0, 3, (n, K + 1, V)).astype(np.float32)).to(torch.bfloat16)
    drf = tgt[:, :K].clone()
    toks = torch.from_numpy(rng.integers(0, V, (n, K)).astype(np.int32))
    # drafts must lie in q's kept set for the ratio to be 1: take q's argmax
    toks = drf.float().argmax(-1).to(torch.int32)
    T = torch.ones(n)
    tp = torch.full((n,), 0.95)
    o, g = _check(tgt, drf, toks, T, torch.zeros(n, dtype=torch.int32), tp, 11)
    assert (o["accept_len"] == K).all()


def test_repeated_runs_identical_on_medium():
    w = workloads.make("medium", device=DEV, scale=dict(n=16))
    first = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=2)
    ref = [x.clone() for x in (first.accept_len, first.out_tokens, first.num_emitted, first.row_status)]
    for _ in range(10):
        o = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=2)
        for a, b in zip(ref, (o.accept_len, o.out_tokens, o.num_emitted, o.row_status)):
            assert torch.equal(a, b)
