"""fp32 rows whose kept set is too large to list (top-k above 32 or off, top-p
over the vocabulary) against the oracle, through sv_build_target_probs,
sv_verify_chain and sv_verify_block (needs a GB300).

fp32 values are rarely equal, so besides plain random logits the rows here
are also rounded to coarse grids, which makes long runs of exact ties at the
top-k and top-p cutoffs (the token's rank among them then decides its
probability), and carry the special values (-0 and +0 at the maximum, -inf,
NaN, +inf, rows of nothing but -inf).
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


def _check_rows(logits: torch.Tensor, T, tk, tp, toks):
    """build_target_probs on [rows, V] fp32 logits, one request per row, against the oracle."""
    rows, V = logits.shape
    Tt = torch.tensor(T, dtype=torch.float32, device=DEV)
    kt = torch.tensor(tk, dtype=torch.int32, device=DEV)
    pt = torch.tensor(tp, dtype=torch.float32, device=DEV)
    tt = torch.tensor(toks, dtype=torch.int32, device=DEV)
    desc, ptok, dense = sv.build_target_probs(logits.to(DEV), Tt, kt, pt, tokens=tt, dense=True)
    torch.cuda.synchronize()
    d = sv.desc_fields(desc)
    host = np_logits(logits)
    checked = 0
    for i in range(rows):
        od, op = oracle.row_transform(host[i], float(T[i]), int(tk[i]), float(tp[i]))
        assert d["status"][i] == od["status"], (i, d["status"][i], od["status"])
        if od["status"] != 0:
            continue
        assert d["argmax"][i] == od["argmax"], (i, d["argmax"][i], od["argmax"])
        if od["cut_margin"] < 1e-9:
            continue
        assert d["kept"][i] == od["kept"] and d["cutoff_ties"][i] == od["cutoff_ties"], (i, d["kept"][i], od)
        assert d["cutoff_logit"][i] == np.float32(od["cutoff_logit"])
        assert d["max_logit"][i] == np.float32(od["max_logit"])
        assert abs(d["log_norm"][i] - od["log_norm"]) <= 1e-5 * max(1.0, abs(od["log_norm"]))
        np.testing.assert_allclose(dense[i].cpu().numpy().astype(np.float64), op, rtol=1e-5, atol=1e-30)
        t = int(toks[i])
        assert abs(float(ptok[i]) - op[t]) <= 1e-5 * op[t] + 1e-30, (i, float(ptok[i]), op[t])
        checked += 1
    return checked


@pytest.mark.parametrize("V", [1, 2, 3, 4, 5, 6, 7, 33, 4099, 151_936])
def test_row_transform_matches_oracle(V):
    rng = np.random.default_rng(V)
    rows = 12
    x = torch.from_numpy(rng.normal(0.0, 3.0, (rows, V)).astype(np.float32))
    T = rng.choice([0.3, 0.7, 1.0, 1.5], rows).tolist()
    tk = rng.choice([0, 0, 40, max(1, V - 1), V, 33], rows).tolist()
    tp = rng.choice([1.0, 0.95, 0.9, 0.5, 0.1], rows).tolist()
    toks = rng.integers(0, V, rows).tolist()
    assert _check_rows(x, T, tk, tp, toks) >= rows // 2


@pytest.mark.parametrize("grid", [0.5, 0.125, 1.0 / 64])
def test_exact_ties_at_the_cutoffs(grid):
    # values on a coarse grid: long tie groups wherever a cutoff falls, and
    # the token placed first, in the middle and last of its tie group
    rng = np.random.default_rng(int(1 / grid))
    rows, V = 18, 9_000
    x = np.round(rng.normal(0.0, 2.0, (rows, V)) / grid) * grid
    T = [1.0] * rows
    tk = [0, 50, 300, 0, 0, 1000] * 3
    tp = [0.9, 1.0, 0.95, 0.5, 0.2, 0.99] * 3
    logits = torch.from_numpy(x.astype(np.float32))
    host = np_logits(logits)
    toks = []
    for i in range(rows):
        od, _ = oracle.row_transform(host[i], T[i], tk[i], tp[i])
        same = np.flatnonzero(host[i] == od["cutoff_logit"])
        toks.append(int(same[[0, len(same) // 2, -1][i % 3]]))
    assert _check_rows(logits, T, tk, tp, toks) >= rows - 2


def test_special_values():
    rng = np.random.default_rng(5)
    V = 4_000
    x = rng.normal(0, 3, (7, V)).astype(np.float32)
    x[0, 123] = np.nan
    x[1, 77] = np.inf
    x[2, :] = -np.inf
    x[3, 10] = -np.inf                # one -inf among finite values: fine
    x[4, :] = -np.inf                 # -0 and +0 the largest values
    x[4, 5], x[4, 9] = -0.0, 0.0
    x[5, ::2] = -np.inf               # half the row -inf, kept set through all of it
    x[6, 100] = -np.nan
    logits = torch.from_numpy(x)
    n = _check_rows(logits, [1.0] * 7, [0, 0, 0, 0, 0, 0, 0], [0.9, 0.9, 0.9, 0.9, 1.0, 1.0, 0.9],
                    [0, 1, 2, 10, 5, 3, 4])
    assert n >= 2


@pytest.mark.parametrize("seed", range(6))
def test_verify_full_vocab_kept_sets(seed):
    rng = np.random.default_rng(200 + seed)
    V = int(rng.choice([1, 2, 3, 5, 7, 33, 4099, 9000]))
    mode = ["full", "mixed"][seed % 2]
    w = workloads.random_case(seed, 8, 4, V, dtype=torch.float32, device=DEV, mode=mode)
    g = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=seed)
    torch.cuda.synchronize()
    o = oracle.verify_chain(np_logits(w.target), np_logits(w.draft), w.draft_tokens.cpu().numpy(),
                            w.temperature.cpu().numpy(), w.top_k.cpu().numpy(), w.top_p.cpu().numpy(), seed=seed)
    assert ((g.row_status.cpu().numpy() & sv.ROW_UNSUPPORTED) == 0).all()
    compare_verify(o, g, w.draft_tokens.cpu().numpy(), np.full(w.n, w.K), w.V)


@pytest.mark.parametrize("seed", range(3))
def test_verify_block_full_vocab_kept_sets(seed):
    w = workloads.random_case(50 + seed, 6, 4, 4099, dtype=torch.float32, device=DEV, mode="full")
    g = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=seed, block=True)
    torch.cuda.synchronize()
    o = oracle.verify_chain(np_logits(w.target), np_logits(w.draft), w.draft_tokens.cpu().numpy(),
                            w.temperature.cpu().numpy(), w.top_k.cpu().numpy(), w.top_p.cpu().numpy(), seed=seed,
                            block=True)
    compare_verify(o, g, w.draft_tokens.cpu().numpy(), np.full(w.n, w.K), w.V)


def test_residual_draws_follow_the_residual():
    # one request, every draft token rejected (target logit -inf there): the
    # emitted tokens over many seeds are draws from max(0, p - q) / W
    V, K = 64, 1
    rng = np.random.default_rng(9)
    t = rng.normal(0, 1.0, (1, K + 1, V)).astype(np.float32)
    d = rng.normal(0, 1.0, (1, K, V)).astype(np.float32)
    t[0, 0, 0] = -np.inf
    toks = torch.zeros((1, K), dtype=torch.int32, device=DEV)
    tgt, drf = torch.from_numpy(t).to(DEV), torch.from_numpy(d).to(DEV)
    T = torch.ones(1, device=DEV)
    tp = torch.full((1,), 0.999, device=DEV)
    counts = np.zeros(V)
    for s in range(1500):
        g = sv.verify_chain(tgt, drf, toks, T, None, tp, seed=s)
        counts[int(g.out_tokens[0, 0])] += 1
    _, p = oracle.row_transform(t[0, 0], 1.0, 0, 0.999)
    _, q = oracle.row_transform(d[0, 0], 1.0, 0, 0.999)
    r = np.maximum(p - q, 0.0)
    r /= r.sum()
    keep = r * 1500 >= 5
    exp_c = r[keep] * 1500
    chi2 = float((((counts[keep] - exp_c) ** 2) / exp_c).sum())
    assert counts[~keep].sum() <= 0.02 * 1500 + 10
    assert chi2 < 2.5 * keep.sum() + 30, (chi2, keep.sum())
