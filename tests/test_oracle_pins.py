"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here retypes the oracle's formulas: each check is a closed form, a
library routine on a special case, a brute force on tiny inputs, a value the
pages print, or a theorem (the accept/resample sampler emits exactly p).
"""
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
from tests.conftest import bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# Philox4x32-10 and the uniforms
# --------------------------------------------------------------------------
def test_philox_known_answers():
    n = 0
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w = [int(x, 16) for x in line.split()]
            out = oracle.philox4x32_10(w[0:4], w[4:6])
            assert list(out) == w[6:10]
            n += 1
    assert n == 3


def test_uniform_is_word0_top24_bits():
    for seed, r, j, d in [(0, 0, 0, 0), (12345678901, 7, 3, 1), (2**64 - 1, 2**32 - 1, 5, 0)]:
        w = oracle.philox4x32_10([r, j, d, 0], [seed & 0xFFFFFFFF, seed >> 32])
        u = oracle.uniform(seed, r, j, d)
        assert u == (int(w[0]) >> 8) / 2**24
        assert 0.0 <= u < 1.0


def test_uniforms_are_uniform():
    # chi-square over 64 equal bins, 2*10^5 draws across (request, position, draw)
    us = np.array([oracle.uniform(0, r, j, d) for r in range(25000) for j in range(4) for d in range(2)])
    counts = np.bincount((us * 64).astype(int), minlength=64)
    p = scipy.stats.chisquare(counts).pvalue
    assert p > 1e-3, p


# --------------------------------------------------------------------------
# Row transform: closed forms and library special cases
# --------------------------------------------------------------------------
def _row(values):
    return np.asarray(values, dtype=np.float32)


def test_softmax_special_case_matches_scipy():
    rng = np.random.default_rng(0)
    for T in (0.3, 1.0, 2.5):
        row = rng.normal(0, 3, 257).astype(np.float32)
        d, p = oracle.row_transform(row, T, 0, 1.0)
        ref = scipy.special.softmax(row.astype(np.float64) / float(np.float32(T)))   # T is an fp32 argument
        np.testing.assert_allclose(p, ref, rtol=1e-12, atol=1e-300)
        assert d["kept"] == 257 and d["status"] == 0
        ref_z = np.exp((row.astype(np.float64) - row.max()) / float(np.float32(T))).sum()
        assert d["log_norm"] == pytest.approx(np.log(ref_z), rel=1e-12)


def test_top_p_closed_form():
    probs = np.array([0.05, 0.5, 0.15, 0.3])
    row = _row(np.log(probs))
    # sorted masses 0.5, 0.3, 0.15, 0.05 -> prefixes 0.5, 0.8, 0.95, 1.0
    d, p = oracle.row_transform(row, 1.0, 0, 0.79)
    assert d["kept"] == 2
    np.testing.assert_allclose(p, [0, 0.5 / 0.8, 0, 0.3 / 0.8], rtol=1e-6)
    d, p = oracle.row_transform(row, 1.0, 0, 0.81)
    assert d["kept"] == 3
    np.testing.assert_allclose(p, [0, 0.5 / 0.95, 0.15 / 0.95, 0.3 / 0.95], rtol=1e-6)
    d, p = oracle.row_transform(row, 1.0, 0, 0.4)           # the crossing token is kept: >= 1 token
    assert d["kept"] == 1 and p[1] == 1.0
    d, p = oracle.row_transform(row, 1.0, 2, 1.0)           # top-k 2
    np.testing.assert_allclose(p, [0, 0.5 / 0.8, 0, 0.3 / 0.8], rtol=1e-6)
    # temperature 2 on log-probabilities gives p proportional to sqrt(probs)
    d, p = oracle.row_transform(row, 2.0, 0, 1.0)
    ref = np.sqrt(probs) / np.sqrt(probs).sum()
    np.testing.assert_allclose(p, ref, rtol=1e-6)
    # top-p mass is measured after top-k: k = 3 renormalises to 0.5/0.95, 0.3/0.95, ...
    d, p = oracle.row_transform(row, 1.0, 3, 0.84)          # 0.8/0.95 = 0.842 >= 0.84 -> 2 kept
    assert d["kept"] == 2
    d, p = oracle.row_transform(row, 1.0, 3, 0.85)
    assert d["kept"] == 3


def test_uniform_row_ties_keep_lowest_indices():
    row = np.zeros(8, np.float32)
    d, p = oracle.row_transform(row, 1.0, 0, 0.3)           # 2/8 < 0.3 <= 3/8
    assert d["kept"] == 3 and d["cutoff_ties"] == 3
    np.testing.assert_allclose(p, [1 / 3] * 3 + [0] * 5, rtol=1e-15)
    d, p = oracle.row_transform(row, 0.5, 5, 1.0)
    np.testing.assert_allclose(p, [0.2] * 5 + [0] * 3, rtol=1e-15)
    d, p = oracle.row_transform(_row([1, 3, 3, 3, 0]), 1.0, 2, 1.0)
    assert np.nonzero(p)[0].tolist() == [1, 2] and d["cutoff_ties"] == 2
    assert d["cutoff_logit"] == 3.0


def test_negative_zero_ties_with_positive_zero():
    d, p = oracle.row_transform(_row([-0.0, 0.0, -1.0]), 1.0, 1, 1.0)
    assert p[0] == 1.0
    d, _ = oracle.row_transform(_row([-0.0, 0.0, -1.0]), 0.0)
    assert d["argmax"] == 0
    d, _ = oracle.row_transform(_row([-1.0, 0.0, -0.0]), 0.0)
    assert d["argmax"] == 1


def test_top_k_set_matches_torch_topk_without_ties():
    rng = np.random.default_rng(1)
    for k in (1, 2, 20, 100):
        row = rng.permutation(1000).astype(np.float32) / 10.0          # distinct values
        _, p = oracle.row_transform(row, 0.7, k, 1.0)
        ref = set(torch.topk(torch.from_numpy(row), k).indices.tolist())
        assert set(np.nonzero(p)[0].tolist()) == ref
        # the top-k set does not depend on the temperature
        _, p2 = oracle.row_transform(row, 3.0, k, 1.0)
        assert set(np.nonzero(p2)[0].tolist()) == ref
        assert p.sum() == pytest.approx(1.0, abs=1e-12)


def test_top_p_cutoff_brute_force_on_bf16_rows():
    rng = np.random.default_rng(2)
    for trial in range(20):
        V = int(rng.integers(5, 300))
        vals = rng.normal(0, 3, V).astype(np.float32)
        bits = bf16_bits(vals)
        f = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        T, top_p = float(rng.choice([0.4, 1.0, 1.7])), float(rng.choice([0.5, 0.9, 0.99]))
        d, p = oracle.row_transform(bits, T, 0, top_p)
        # brute force: every prefix of the (value desc, index asc) order, kept = shortest reaching top_p
        order = sorted(range(V), key=lambda x: (-f[x], x))
        m = f[order[0]]
        masses = [np.exp((f[x] - m) / np.float32(T)) for x in order]
        total = sum(masses)
        kept = next(i + 1 for i in range(V) if sum(masses[: i + 1]) >= np.float32(top_p) * total)
        assert d["kept"] == kept or d["cut_margin"] < 1e-9
        assert set(np.nonzero(p)[0]) <= set(order[:kept])


def test_status_bits():
    d, _ = oracle.row_transform(_row([0, np.nan, 1]), 1.0)
    assert d["status"] == oracle.NONFINITE
    d, _ = oracle.row_transform(_row([0, np.inf, 1]), 0.0)
    assert d["status"] == oracle.NONFINITE
    d, _ = oracle.row_transform(_row([-np.inf] * 4), 1.0)
    assert d["status"] == oracle.EMPTY
    d, p = oracle.row_transform(_row([-np.inf] * 4), 0.0)   # greedy argmax stays defined
    assert d["status"] == 0 and d["argmax"] == 0
    d, p = oracle.row_transform(_row([-np.inf, 2, -np.inf]), 0.5, 0, 1.0)
    assert d["status"] == 0 and p.tolist() == [0, 1, 0]
    for T, tp in [(-1.0, 1.0), (np.nan, 1.0), (np.inf, 1.0), (1.0, 0.0), (1.0, np.nan)]:
        d, _ = oracle.row_transform(_row([0, 1]), T, 0, tp)
        assert d["status"] == oracle.BAD_PARAM


def test_greedy_argmax_first_occurrence_matches_numpy():
    rng = np.random.default_rng(3)
    for _ in range(50):
        row = rng.integers(-3, 4, int(rng.integers(1, 64))).astype(np.float32)   # many ties
        d, p = oracle.row_transform(row, 0.0)
        assert d["argmax"] == int(np.argmax(row))
        assert p[int(np.argmax(row))] == 1.0 and p.sum() == 1.0


def test_small_temperature_limit_is_greedy():
    rng = np.random.default_rng(4)
    row = rng.permutation(100).astype(np.float32)
    _, p = oracle.row_transform(row, 1e-3, 0, 1.0)
    assert int(np.argmax(p)) == int(np.argmax(row)) and p.max() == 1.0


# --------------------------------------------------------------------------
# Inverse CDF against numpy's searchsorted
# --------------------------------------------------------------------------
def test_bonus_token_is_inverse_cdf_of_p():
    # K = 0 windows emit only the bonus token: InvCDF(p, u(r, 0, 1)).
    rng = np.random.default_rng(5)
    n, V = 300, 16
    logits = rng.normal(0, 1, (n, 1, V)).astype(np.float32)
    o = oracle.verify_chain(logits, None, np.zeros((n, 0), np.int32), np.ones(n, np.float32), seed=77)
    for r in range(n):
        p = scipy.special.softmax(logits[r, 0].astype(np.float64))
        u = oracle.uniform(77, r, 0, 1)
        ref = int(np.searchsorted(np.cumsum(p), u * p.sum(), side="right"))
        assert o["out_tokens"][r, 0] == ref or o["flags"][r]
        assert o["accept_len"][r] == 0 and o["num_emitted"][r] == 1


# --------------------------------------------------------------------------
# Greedy chain: brute force
# --------------------------------------------------------------------------
def test_greedy_chain_brute_force():
    rng = np.random.default_rng(6)
    n, K, V = 200, 5, 7
    tgt = rng.integers(-2, 3, (n, K + 1, V)).astype(np.float32)        # ties everywhere
    am = tgt.argmax(-1)
    toks = np.where(rng.random((n, K)) < 0.7, am[:, :K], rng.integers(0, V, (n, K))).astype(np.int32)
    vl = rng.integers(0, K + 1, n).astype(np.int32)
    o = oracle.verify_chain(tgt, None, toks, np.zeros(n, np.float32), verify_len=vl)
    for r in range(n):
        a = 0
        while a < vl[r] and toks[r, a] == am[r, a]:
            a += 1
        assert o["accept_len"][r] == a
        assert o["out_tokens"][r, :a].tolist() == toks[r, :a].tolist()
        assert o["out_tokens"][r, a] == am[r, a]
        assert (o["out_tokens"][r, a + 1:] == -1).all()


def test_greedy_chain_rejects_higher_index_duplicate():
    # a draft equal to the higher-index copy of a tied maximum is rejected
    tgt = np.zeros((1, 2, 6), np.float32)
    tgt[0, 0, [2, 4]] = 5.0
    tgt[0, 1, 3] = 1.0
    o = oracle.verify_chain(tgt, None, np.array([[4]], np.int32), np.zeros(1, np.float32))
    assert o["accept_len"][0] == 0 and o["out_tokens"][0].tolist() == [2, -1]
    o = oracle.verify_chain(tgt, None, np.array([[2]], np.int32), np.zeros(1, np.float32))
    assert o["accept_len"][0] == 1 and o["out_tokens"][0].tolist() == [2, 3]


def test_greedy_wide_mean_accept_length_closed_form():
    from speculative_decoding_verification_rows_gb300 import workloads
    from tests.conftest import np_logits
    w = workloads.make("greedy_wide", scale=dict(n=4000, V=512))
    o = oracle.verify_chain(np_logits(w.target), None, w.draft_tokens.numpy(), w.temperature.numpy())
    pm = np.array(workloads.GREEDY_WIDE_MATCH)
    expect = np.cumprod(pm).sum()                            # sum over i of prod_{l<=i} p_l = 1.23304
    assert expect == pytest.approx(1.23304, abs=1e-5)
    a = o["accept_len"].astype(float)
    sd = a.std() / np.sqrt(len(a))
    assert abs(a.mean() - expect) < 4 * sd + 0.01, (a.mean(), expect)


# --------------------------------------------------------------------------
# Sampler: the emitted token is distributed exactly as p (the theorem)
# --------------------------------------------------------------------------
PAIRS = {
    "generic": (np.arange(1, 17, dtype=float), np.arange(16, 0, -1, dtype=float)),
    "q_has_zeros": (np.ones(16), np.r_[np.ones(8), np.zeros(8)]),
    "equal": (np.arange(1, 17, dtype=float) ** 2, np.arange(1, 17, dtype=float) ** 2),
    "disjoint": (np.r_[np.zeros(8), np.ones(8)], np.r_[np.ones(8), np.zeros(8)]),
}


def _chi2_first_token(p_w, q_w, n, seed):
    """Draft d ~ q (numpy), verify with K=1 at T=1 on logits log(w); the
    first emitted token must follow p = w / sum(w)."""
    p = p_w / p_w.sum()
    q = q_w / q_w.sum()
    with np.errstate(divide="ignore"):
        lp, lq = np.log(p).astype(np.float32), np.log(q).astype(np.float32)
    rng = np.random.default_rng(seed)
    d = rng.choice(16, size=n, p=q).astype(np.int32)
    tgt = np.broadcast_to(lp, (n, 2, 16)).copy()
    drf = np.broadcast_to(lq, (n, 1, 16)).copy()
    o = oracle.verify_chain(tgt, drf, d.reshape(n, 1), np.ones(n, np.float32), seed=seed)
    first = o["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=16)
    support = p > 0
    assert counts[~support].sum() == 0
    stat = scipy.stats.chisquare(counts[support], n * p[support])
    accept_rate = o["accept_len"].mean()
    return stat.pvalue, accept_rate, np.minimum(p, q).sum()


@pytest.mark.parametrize("name", list(PAIRS))
def test_emitted_token_follows_p(name):
    n = 1_000_000 if name == "generic" else 200_000
    pv, acc, acc_ref = _chi2_first_token(*PAIRS[name], n=n, seed=11)
    assert pv > 1e-3, (name, pv)
    # P(accept) = sum_x min(p, q)
    assert abs(acc - acc_ref) < 5 * np.sqrt(acc_ref * (1 - acc_ref) / n) + 1e-12


def test_pins_catch_planted_mistakes(tmp_path):
    """Each deliberate mistake built into a separate oracle library fails the
    pin that is meant to catch it (the mistakes are listed at ORC_PLANT)."""
    p_w, q_w = PAIRS["generic"]
    with oracle.planted(1, str(tmp_path)):                    # residual q - p
        pv, _, _ = _chi2_first_token(p_w, q_w, n=100_000, seed=13)
        assert pv < 1e-6
    with oracle.planted(5, str(tmp_path)):                    # resample reuses draw 0
        pv, _, _ = _chi2_first_token(p_w, q_w, n=100_000, seed=13)
        assert pv < 1e-6
    with oracle.planted(2, str(tmp_path)):                    # top-p drops the crossing token
        d, _ = oracle.row_transform(_row(np.log([0.05, 0.5, 0.15, 0.3])), 1.0, 0, 0.79)
        assert d["kept"] != 2
    with oracle.planted(3, str(tmp_path)):                    # argmax takes the last tie
        row = np.array([1, 5, 2, 5], np.float32)
        d, _ = oracle.row_transform(row, 0.0)
        assert d["argmax"] != int(np.argmax(row))
    with oracle.planted(4, str(tmp_path)):                    # request before position
        conf = np.ones((3, 4), np.float32)
        vl, _, _, _ = oracle.plan_budget(conf, 3 + 5, 16)
        sel = _brute_plan(conf, 3 + 5)
        assert vl.tolist() != np.bincount([r for _, _, r in sel], minlength=3).tolist()


# --------------------------------------------------------------------------
# Planner
# --------------------------------------------------------------------------
def _golden_layouts():
    rows = []
    with open(os.path.join(GOLDEN, "ragged_layouts.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w, qo, tot = [x.strip() for x in line.split(";")]
            rows.append(([int(x) for x in w.split(",")], [int(x) for x in qo.split(",")], int(tot)))
    return rows


def test_planner_reproduces_printed_layout():
    # confidences that make the global rank hand out 5 and 3 drafts: windows 6, 4, 1, 1
    conf = np.zeros((4, 6), np.float32)
    conf[0, :5] = 0.9
    conf[1, :3] = 0.9
    windows, qo_ref, total_ref = _golden_layouts()[0]
    vl, qo, total, st = oracle.plan_budget(conf, budget=total_ref, bucket=total_ref)
    assert (vl + 1).tolist() == windows and qo.tolist() == qo_ref and total == total_ref and st == 0


def _brute_plan(conf, budget, draft_len=None):
    n, K = conf.shape
    cands = []
    for r in range(n):
        kr = K if draft_len is None else int(np.clip(draft_len[r], 0, K))
        c = np.nan_to_num(conf[r, :kr], nan=0.0).clip(0, 1).astype(np.float32)
        s = np.cumprod(c, dtype=np.float32)
        cands += [(-float(s[i]), i, r) for i in range(kr)]
    cands.sort()
    sel = cands[: max(0, min(budget - n, len(cands)))]
    return sel


def test_planner_brute_force_and_invariants():
    rng = np.random.default_rng(7)
    for trial in range(40):
        n, K = int(rng.integers(1, 9)), int(rng.integers(0, 7))
        conf = rng.choice([0.0, 0.3, 0.5, 0.9, 1.0, 1.2, np.nan], size=(n, K)).astype(np.float32) \
            if trial % 2 else rng.random((n, K)).astype(np.float32)
        budget = int(rng.integers(n, n * (K + 1) + 3))
        dl = rng.integers(-1, K + 2, n).astype(np.int32) if trial % 3 == 0 else None
        vl, qo, total, st = oracle.plan_budget(conf, budget, budget + 5, draft_len=dl)
        sel = _brute_plan(conf, budget, dl)
        counts = np.bincount([r for _, _, r in sel], minlength=n)
        assert vl.tolist() == counts.tolist()
        for r in range(n):                                    # prefix-closed per request
            assert sorted(i for _, i, rr in sel if rr == r) == list(range(vl[r]))
        assert vl.sum() == len(sel) and total == n + vl.sum() and qo[0] == 0
        assert (np.diff(qo) == vl + 1).all()
        assert (st != 0) == (dl is not None and bool(((dl < 0) | (dl > K)).any()))


def test_planner_permutation_invariance_of_equal_survival_rows():
    rng = np.random.default_rng(8)
    row = rng.random(6).astype(np.float32)
    conf = np.stack([row, rng.random(6).astype(np.float32), row, row])
    for budget in range(4, 4 + 25):
        vl, _, _, _ = oracle.plan_budget(conf, budget, 64)
        for perm in ([2, 1, 0, 3], [3, 1, 2, 0], [0, 1, 3, 2]):
            vl2, _, _, _ = oracle.plan_budget(conf[perm], budget, 64)
            assert vl2.tolist() == vl.tolist()      # equal rows: the window vector is unchanged
    # with distinct rows the windows move with their request
    conf = rng.random((5, 6)).astype(np.float32)
    perm = rng.permutation(5)
    vl, _, _, _ = oracle.plan_budget(conf, 17, 64)
    vl2, _, _, _ = oracle.plan_budget(conf[perm], 17, 64)
    assert vl2.tolist() == vl[perm].tolist()


def test_planner_rejects_bad_arguments():
    conf = np.ones((3, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.plan_budget(conf, budget=2, bucket=8)          # budget < n
    with pytest.raises(ValueError):
        oracle.plan_budget(conf, budget=8, bucket=7)          # bucket < budget


# --------------------------------------------------------------------------
# Ragged layout and trimming
# --------------------------------------------------------------------------
def _sampling_case(seed, n, K, V):
    from speculative_decoding_verification_rows_gb300 import workloads
    from tests.conftest import np_logits
    w = workloads.random_case(seed, n, K, V, mode="mixed")
    return (np_logits(w.target), np_logits(w.draft), w.draft_tokens.numpy(), w.temperature.numpy(),
            w.top_k.numpy(), w.top_p.numpy())


def test_full_windows_ragged_equals_chain():
    tgt, drf, tok, T, tk, tp = _sampling_case(1, 12, 4, 97)
    n, K = tok.shape
    a = oracle.verify_chain(tgt, drf, tok, T, tk, tp, seed=3)
    qo = np.arange(n + 1, dtype=np.int32) * (K + 1)
    bucket = n * (K + 1) + 3
    packed = np.zeros((bucket, tgt.shape[-1]), tgt.dtype)
    packed[: n * (K + 1)] = tgt.reshape(n * (K + 1), -1)
    b = oracle.verify_ragged(packed, drf, qo, np.full(n, K, np.int32), tok, T, tk, tp, seed=3)
    for key in ("accept_len", "out_tokens", "num_emitted", "pos_status", "flags"):
        assert np.array_equal(a[key], b[key]), key


def test_trimming_keeps_acceptance():
    # accept_len with window v equals min(a_full, v); the tokens up to it agree
    tgt, drf, tok, T, tk, tp = _sampling_case(2, 40, 6, 64)
    n, K = tok.shape
    full = oracle.verify_chain(tgt, drf, tok, T, tk, tp, seed=9)
    rng = np.random.default_rng(0)
    vl = rng.integers(0, K + 1, n).astype(np.int32)
    trim = oracle.verify_chain(tgt, drf, tok, T, tk, tp, verify_len=vl, seed=9)
    for r in range(n):
        if ((full["pos_status"][r] | trim["pos_status"][r]) & oracle.ERROR_MASK).any():
            continue
        if full["flags"][r] or trim["flags"][r]:
            continue
        a_full = full["accept_len"][r]
        assert trim["accept_len"][r] == min(a_full, vl[r])
        if a_full < vl[r]:
            assert trim["out_tokens"][r].tolist() == full["out_tokens"][r].tolist()
        else:
            assert trim["out_tokens"][r, : vl[r]].tolist() == tok[r, : vl[r]].tolist()


def test_ragged_windows_read_their_own_rows_only():
    windows, qo, total = _golden_layouts()[1]                 # [6, 6, 2, 2]
    tgt, drf, tok, T, tk, tp = _sampling_case(3, 4, 5, 50)
    n, K = tok.shape
    vl = np.array(windows, np.int32) - 1
    bucket = total + 2
    packed = np.zeros((bucket, tgt.shape[-1]), np.uint16)
    for r in range(n):
        packed[qo[r]: qo[r] + vl[r] + 1] = tgt[r, : vl[r] + 1]
    packed[total:] = bf16_bits([np.nan] * tgt.shape[-1])     # padding rows: never read
    o = oracle.verify_ragged(packed, drf, np.array(qo, np.int32), vl, tok, T, tk, tp, seed=5)
    # the same windows as a capped uniform call (rows in block layout)
    capped = oracle.verify_chain(tgt, drf, tok, T, tk, tp, verify_len=vl, seed=5)
    for key in ("accept_len", "out_tokens", "num_emitted", "pos_status", "flags"):
        assert np.array_equal(o[key], capped[key]), key
    assert (o["pos_status"] & oracle.ERROR_MASK).sum() == 0
    assert (o["accept_len"] <= vl).all()
    # request 0 as a single-request call (its uniforms are keyed by request 0 either way)
    one = oracle.verify_chain(tgt[:1], drf[:1], tok[:1], T[:1], tk[:1], tp[:1], verify_len=vl[:1], seed=5)
    assert o["out_tokens"][0].tolist() == one["out_tokens"][0].tolist()
    # a window inconsistent with qo_indptr is a layout error, not a misread
    bad = vl.copy()
    bad[1] += 1
    o = oracle.verify_ragged(packed, drf, np.array(qo, np.int32), bad, tok, T, tk, tp, seed=5)
    assert o["pos_status"][1, 0] & oracle.BAD_LAYOUT and o["out_tokens"][1, 0] == -1
