"""Budget from a step-cost table and the acceptance-against-trimming counters:
the CUDA path (through the C ABI) against the oracle (needs a GB300).

The chosen budget must equal the oracle's unless the oracle reports the two
best Theta within 1e-9 of each other (then the GPU's choice must reach the
best Theta within that margin); the plan for the chosen budget is compared
bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_rows_gb300 import build as sv_build
from speculative_decoding_verification_rows_gb300 import sv, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv_build.build()
    sv.load()


def _t(a, dtype):
    return None if a is None else torch.as_tensor(np.asarray(a), dtype=dtype, device=DEV)


def _staircase(rng, n, b_hi):
    """A profiled-looking table: shelves at a power-of-two-ish ladder of token
    counts, costs rising with occasional jumps (graph buckets)."""
    n_sh = int(rng.integers(1, 12))
    toks = np.unique(rng.integers(max(1, n - 2), b_hi + 8, n_sh)).astype(np.int32)
    costs = np.cumsum(rng.uniform(0.05, 1.0, len(toks)) * (1 + 4 * (rng.uniform(size=len(toks)) < 0.2)))
    return toks, (0.5 + costs).astype(np.float32)


def _check_case(conf, toks, costs, bucket, fixed=0.0, bsz=None, bov=None, dl=None):
    n, K = conf.shape
    ob, oth, omargin, ost = oracle.choose_budget(conf, toks, costs, bucket, fixed, bsz, bov, dl)
    g = sv.plan_budget_cost(_t(conf, torch.float32), _t(toks, torch.int32), _t(costs, torch.float32), bucket,
                            fixed, _t(bsz, torch.int32), _t(bov, torch.float32), _t(dl, torch.int32))
    torch.cuda.synchronize()
    gb, gst = int(g[0]), int(g[1])
    assert gst == ost, (gst, ost)
    if omargin >= 1e-9:
        assert gb == ob, (gb, ob, omargin)
    else:   # near tie: the GPU's budget must reach the best Theta
        _, th_at, _, _ = oracle.choose_budget(conf, toks, costs, gb, fixed, bsz, bov, dl)
        assert th_at == pytest.approx(oth, rel=1e-9)
    vl, qo, tot, pst = oracle.plan_budget(conf, gb, max(bucket, gb), dl)
    assert g[2].cpu().numpy().tolist() == vl.tolist()
    assert g[3].cpu().numpy().tolist() == qo.tolist()
    assert int(g[4]) == tot and int(g[5]) == pst
    return gb


def test_budget_random_tables():
    rng = np.random.default_rng(11)
    for trial in range(60):
        n, K = int(rng.integers(1, 48)), int(rng.integers(0, 24))
        conf = (rng.uniform(0.0, 1.0, (n, K)) if trial % 3 else
                rng.choice([0.0, 0.3, 0.7, 0.95, 1.0, 1.2, np.nan], (n, K))).astype(np.float32)
        bucket = n + int(rng.integers(0, n * K + 4))
        toks, costs = _staircase(rng, n, n * (K + 1))
        fixed = float(np.float32(rng.uniform(0, 2))) if trial % 2 else 0.0
        bsz = bov = None
        if trial % 4 == 1:
            bsz = np.sort(rng.choice(np.arange(1, 128), 3, replace=False)).astype(np.int32)
            bov = rng.uniform(0, 1, 3).astype(np.float32)
        dl = rng.integers(-1, K + 2, n).astype(np.int32) if trial % 5 == 0 else None
        _check_case(conf, toks, costs, bucket, fixed, bsz, bov, dl)


def test_budget_uniform_confidence_ties_and_ragged_shape():
    # uniform confidence: every depth ties, the choice sits on a shelf edge
    n, K = 32, 8
    conf = np.full((n, K), 0.85, np.float32)
    toks = np.array([n * (m + 1) for m in range(K + 1)], np.int32)
    costs = np.array([1.0 + 0.3 * m + (2.0 if m >= 4 else 0.0) for m in range(K + 1)], np.float32)
    b = _check_case(conf, toks, costs, n * (K + 1))
    assert b % n == 0
    # the ragged workload's shape: 256 requests x 16 drafts, bucket 2048
    w = workloads.make("ragged", device=DEV, scale=dict(V=64))
    conf = w.conf.cpu().numpy()
    rng = np.random.default_rng(2)
    for _ in range(5):
        toks, costs = _staircase(rng, conf.shape[0], w.bucket)
        _check_case(conf, toks, costs, w.bucket, float(np.float32(rng.uniform(0, 3))))


def test_budget_fallbacks():
    rng = np.random.default_rng(4)
    conf = rng.uniform(0.1, 1.0, (20, 6)).astype(np.float32)
    n, K = conf.shape
    assert _check_case(conf, None, None, 200) == n + n * K                      # no table: no trimming
    assert _check_case(conf, [50, 100, 200], [2.0, 2.0, 2.0], 200) == n + n * K  # flat table
    assert _check_case(conf, [5, 10], [1.0, 2.0], 200) == n + n * K             # no shelf holds n
    assert _check_case(conf, [64, 64, 128], [1.0, 1.5, 2.0], 200) == n + n * K  # not ascending
    assert _check_case(conf, [64, 128], [1.0, float("nan")], 200) == n + n * K
    assert _check_case(conf, [64, 128], [1.0, 2.0], 60) <= 60                    # bucket caps it
    with pytest.raises(sv.SVError):                                              # beyond the sort capacity
        sv.plan_budget_cost(torch.rand(1025, 16, device=DEV), _t([2048], torch.int32),
                            _t([1.0], torch.float32), 20000)


def test_budget_then_ragged_verify_sync_free():
    # choose the budget and plan with no host readback; pack the target rows
    # of the planned windows (a stand-in for the target forward), verify, and
    # count acceptance against trimming, again without readback
    w = workloads.make("ragged", device=DEV, scale=dict(V=4096))
    rng = np.random.default_rng(9)
    toks, costs = _staircase(rng, w.n, w.bucket)
    toks_d, costs_d = _t(toks, torch.int32), _t(costs, torch.float32)
    ws_p, ws_v = sv.Workspace(DEV), sv.Workspace(DEV)
    sv.plan_budget_cost(w.conf, toks_d, costs_d, w.bucket, 0.5, ws=ws_p)     # sizes the workspace
    torch.cuda.synchronize()
    torch.cuda.set_sync_debug_mode("error")
    try:
        b, bst, vl, qo, tot, st = sv.plan_budget_cost(w.conf, toks_d, costs_d, w.bucket, 0.5, ws=ws_p)
    finally:
        torch.cuda.set_sync_debug_mode("default")
    packed = workloads.pack_rows(w.target, qo.cpu(), vl.cpu(), w.bucket)
    o = sv.verify_ragged(packed, w.draft, qo, vl, w.draft_tokens, w.temperature, w.top_k, w.top_p,
                         seed=w.seed, ws=ws_v)
    torch.cuda.synchronize()
    torch.cuda.set_sync_debug_mode("error")
    try:
        stats = sv.verify_stats(o.accept_len, o.num_emitted, vl, w.K)
    finally:
        torch.cuda.set_sync_debug_mode("default")
    torch.cuda.synchronize()
    ref = oracle.verify_stats(o.accept_len.cpu().numpy(), o.num_emitted.cpu().numpy(), vl.cpu().numpy(), w.K)
    assert tuple(stats.cpu().numpy().tolist()) == ref
    assert ref[1] == int(tot) <= int(b)      # tokens submitted = the plan's total, within the budget


def test_verify_stats_random():
    rng = np.random.default_rng(8)
    for trial in range(20):
        n, K = int(rng.integers(1, 3000)), int(rng.integers(0, 17))
        dl = rng.integers(-1, K + 2, n).astype(np.int32) if trial % 2 else None
        kr = np.clip(dl if dl is not None else np.full(n, K), 0, K)
        vl = (rng.integers(0, 1 << 30, n) % (kr + 1)).astype(np.int32)
        acc = (rng.integers(0, 1 << 30, n) % (vl + 1)).astype(np.int32)
        emitted = np.where(rng.uniform(size=n) < 0.05, 0, acc + 1).astype(np.int32)
        g = sv.verify_stats(_t(acc, torch.int32), _t(emitted, torch.int32), _t(vl, torch.int32), K,
                            _t(dl, torch.int32))
        assert tuple(g.cpu().numpy().tolist()) == oracle.verify_stats(acc, emitted, vl, K, dl)
