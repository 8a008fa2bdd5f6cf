"""Online acceptance estimator through the C ABI against the oracle's
(needs a GB300): features and predictions per draft row, the Newton
statistics and refits over a run of observe calls, and the sync-free
predict -> plan -> observe sequence.
"""
import numpy as np
import pytest
import scipy.special
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


@pytest.mark.parametrize("seed,mode,V", [(0, "topk", 4099), (1, "mixed", 3000), (2, "topk", 248_320),
                                         (3, "mixed", 129)])
def test_features_and_predictions_match_the_oracle(seed, mode, V):
    w = workloads.random_case(seed, 12, 5, V, device=DEV, mode=mode)
    if w.draft is None:
        pytest.skip("no draft rows")
    est = sv.Estimator(w.K)
    x, p = est.predict(w.draft, w.temperature, w.top_k, w.top_p)
    torch.cuda.synchronize()
    ox = oracle.est_features(np_logits(w.draft), w.temperature.cpu().numpy(), w.top_k.cpu().numpy(),
                             w.top_p.cpu().numpy())
    gx = x.cpu().numpy().astype(np.float64)
    both_nan = np.isnan(ox) & np.isnan(gx)
    ok = both_nan | (np.abs(gx - ox) <= 1e-5 * np.maximum(1.0, np.abs(ox))) | (ox > 25.0) & (gx > 24.0)
    assert ok.all(), (gx[~ok], ox[~ok])
    # the prediction from the GPU's own features
    op = oracle.Estimator(w.K).predict(gx)
    gp = p.cpu().numpy().astype(np.float64)
    fin = np.isfinite(op)
    assert np.allclose(gp[fin], op[fin], rtol=1e-6, atol=1e-7)
    assert np.isnan(gp[~fin]).all()


def _calls(rng, n, K, n_calls):
    for _ in range(n_calls):
        x = rng.normal(0.0, 2.0, (n, K)).astype(np.float32)
        alive = rng.uniform(size=(n, K)) < scipy.special.expit(x + np.linspace(1.0, -0.5, K))
        acc = np.array([np.argmin(a) if not a.all() else K for a in alive], np.int32)
        vl = rng.integers(0, K + 1, n).astype(np.int32)
        acc = np.minimum(acc, vl).astype(np.int32)
        emitted = np.where(rng.uniform(size=n) < 0.05, 0, acc + 1).astype(np.int32)
        x[rng.uniform(size=(n, K)) < 0.02] = np.nan
        yield x, acc, emitted, vl


@pytest.mark.parametrize("K,n", [(4, 300), (1, 2_500), (40, 37), (63, 20)])
def test_observe_and_refit_match_the_oracle(K, n):
    # items (request, position) spread over the CTAs of the observe cluster in
    # one or several rounds, positions repeating inside a warp (K = 1, 4) or
    # not (K = 40, 63)
    rng = np.random.default_rng(7 + K)
    g = sv.Estimator(K)
    g.state[0] = 3.0
    o = oracle.Estimator(K)
    o.state[0] = 3.0
    for x, acc, emitted, vl in _calls(rng, n, K, 23):
        g.observe(torch.from_numpy(x).to(DEV), torch.from_numpy(acc).to(DEV), torch.from_numpy(emitted).to(DEV),
                  torch.from_numpy(vl).to(DEV), refit_every=5)
        o.observe(x.astype(np.float64), acc, emitted, vl, refit_every=5)
    gs = g.state.cpu().numpy()
    assert np.allclose(gs, o.state, rtol=1e-9, atol=1e-9), (gs[:1 + K], o.state[:1 + K])
    assert gs[4 * K + 4] == 23 and gs[0] != 3.0          # four refits happened


def test_predict_plan_observe_sync_free():
    w = workloads.make("large", device=DEV, scale=dict(n=16, V=8192))
    est = sv.Estimator(w.K)
    ws_p = sv.Workspace(DEV)
    x, p = est.predict(w.draft, w.temperature, w.top_k, w.top_p)   # sizes the workspace
    sv.plan_budget(p, w.n + 40, w.n * (w.K + 1), ws=ws_p)
    torch.cuda.synchronize()
    torch.cuda.set_sync_debug_mode("error")
    try:
        x, p = est.predict(w.draft, w.temperature, w.top_k, w.top_p)
        vl, qo, tot, st = sv.plan_budget(p, w.n + 40, w.n * (w.K + 1), ws=ws_p)
        o = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, verify_len=vl)
        est.observe(x, o.accept_len, o.num_emitted, vl, refit_every=1)
    finally:
        torch.cuda.set_sync_debug_mode("default")
    torch.cuda.synchronize()
    assert int(tot) <= w.n + 40
    assert torch.isfinite(est.state).all()
    assert est.state[4 * w.K + 4].item() == 1.0


def test_refit_on_gpu_reaches_the_generating_slope():
    rng = np.random.default_rng(11)
    K, n = 4, 64
    g = sv.Estimator(K)
    g.state[0] = 3.0
    bias = np.array([1.0, 0.5, 0.0, -0.5])
    for _ in range(1000):
        x = rng.normal(0.0, 2.0, (n, K)).astype(np.float32)
        alive = rng.uniform(size=(n, K)) < scipy.special.expit(x.astype(np.float64) + bias)
        acc = np.array([np.argmin(a) if not a.all() else K for a in alive], np.int32)
        g.observe(torch.from_numpy(x).to(DEV), torch.from_numpy(acc).to(DEV), torch.from_numpy(acc + 1).to(DEV))
    slope = g.state[0].item()
    assert 0.85 < slope < 1.15, slope


@pytest.mark.parametrize("name,scale", [("tiny", None), ("large", dict(n=6)), ("medium", dict(n=4, V=30000))])
def test_predict_q_then_verify_q_equals_predict_then_verify(name, scale):
    # the draft rows' results made by predict_q serve the verify that follows: the same features
    # and predictions as predict, the same outputs as sv_verify_chain on the whole batch
    w = workloads.make(name, device=DEV, scale=scale)
    est_a, est_b = sv.Estimator(w.K, DEV), sv.Estimator(w.K, DEV)
    x0, p0 = est_a.predict(w.draft, w.temperature, w.top_k, w.top_p)
    x1, p1, q_rows = est_b.predict_q(w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p)
    ref = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=3)
    got = sv.verify_chain_q(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, q_rows, seed=3)
    torch.cuda.synchronize()
    # bit for bit (NaN where a feature has no value, e.g. fp32 rows a greedy request reads at T = 1
    # over the whole vocabulary)
    torch.testing.assert_close(x1, x0, rtol=0, atol=0, equal_nan=True)
    torch.testing.assert_close(p1, p0, rtol=0, atol=0, equal_nan=True)
    for f in ("accept_len", "out_tokens", "num_emitted", "row_status"):
        assert torch.equal(getattr(got, f), getattr(ref, f)), f


def test_verify_q_with_windows_matches_the_oracle():
    w = workloads.random_case(5, 7, 4, 4099, device=DEV, mode="mixed")
    vl = torch.tensor([4, 0, 2, 3, 1, 4, 4], dtype=torch.int32, device=DEV)
    est = sv.Estimator(w.K, DEV)
    _, _, q_rows = est.predict_q(w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p)
    g = sv.verify_chain_q(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, q_rows,
                          verify_len=vl, seed=9)
    torch.cuda.synchronize()
    o = oracle.verify_chain(np_logits(w.target), np_logits(w.draft), w.draft_tokens.cpu().numpy(),
                            w.temperature.cpu().numpy(), w.top_k.cpu().numpy(), w.top_p.cpu().numpy(),
                            verify_len=vl.cpu().numpy(), seed=9)
    compare_verify(o, g, w.draft_tokens.cpu().numpy(), vl.cpu().numpy(), w.V)
