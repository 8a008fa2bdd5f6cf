"""The parity checker's handling of flagged requests (CPU only).

Requests are built whose decisions sit inside the oracle's margins: a ratio
test with |u - p/q| below 1e-6, and a top-p cut whose prefix mass lies within
1e-9 of the threshold.  Results are then handed to the checker as if the GPU
had produced them: the oracle's own outcome and the outcome of the flipped
decision must pass; a token the draw cannot produce, an accepted length the
decisions do not allow, or drafts that are not the request's must fail.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import compare


class Result:
    def __init__(self, acc, tok, nem, st):
        self.accept_len = torch.tensor(acc, dtype=torch.int32)
        self.out_tokens = torch.tensor(tok, dtype=torch.int32)
        self.num_emitted = torch.tensor(nem, dtype=torch.int32)
        self.row_status = torch.tensor(st, dtype=torch.int32)


def _nudge(x: float, steps: int) -> np.float32:
    """x moved by `steps` float32 ulps."""
    v = np.float32(x)
    for _ in range(abs(steps)):
        v = np.nextafter(v, np.float32(np.inf if steps > 0 else -np.inf), dtype=np.float32)
    return v


def ratio_near_tie_case(seed=7):
    """One request, K = 1, vocab 8, T = 1, top-k 2: the test at position 0
    has p/q within 1e-7 of its uniform.  The kept set is {1, 5}; d_0 = 1."""
    V, T, k = 8, 1.0, 2
    u = oracle.uniform(seed, 0, 0, 0)
    drf = np.full((1, 1, V), -4.0, np.float32)
    drf[0, 0, 1], drf[0, 0, 5] = 1.0, 0.5
    q = oracle.row_transform(drf[0, 0], T, k)[1][1]
    tgt = np.full((1, 2, V), -4.0, np.float32)
    tgt[0, :, 5] = 0.5
    # p(1) = u q(1): logit of token 1 against token 5 at fixed mass split
    want = u * q
    base = 0.5 + np.log(want / (1.0 - want))
    best, best_gap = None, np.inf
    for s in range(-200, 201):
        tgt[0, 0, 1] = _nudge(base, s)
        p = oracle.row_transform(tgt[0, 0], T, k)[1][1]
        if abs(u - p / q) < best_gap:
            best, best_gap = tgt[0, 0, 1], abs(u - p / q)
    tgt[0, 0, 1] = best
    tgt[0, 1, 1], tgt[0, 1, 5] = 0.2, 0.1
    assert best_gap < 1e-7
    args = dict(draft_tokens=np.array([[1]], np.int32), temperature=np.array([T], np.float32),
                top_k=np.array([k], np.int32), top_p=np.array([1.0], np.float32), seed=seed)
    return tgt, drf, args


def test_ratio_near_tie_allows_both_outcomes_and_nothing_else():
    tgt, drf, args = ratio_near_tie_case()
    o = oracle.verify_chain(tgt, drf, **args)
    assert o["flags"][0] & oracle.FLAG_RATIO
    assert o["alt_dec"][0, 0] & oracle.ALT_AMBIG
    assert sorted(compare.valid_accepts(o["alt_dec"][0], 1, False)) == [0, 1]
    win, d = np.array([1]), args["draft_tokens"]
    # the oracle's own outcome
    a = int(o["accept_len"][0])
    compare.compare_verify(o, Result(o["accept_len"], o["out_tokens"], o["num_emitted"], o["pos_status"]), d, win, 8)
    # the flipped decision, with the token the oracle draws there
    b = 1 - a
    tok = [[1, int(o["alt_draw"][0, 1])]] if b == 1 else [[int(o["alt_draw"][0, 0]), -1]]
    compare.compare_verify(o, Result([b], tok, [b + 1], o["pos_status"]), d, win, 8)
    # the flipped decision with a token outside the kept set {1, 5}: invalid
    bad = [[1, 3]] if b == 1 else [[3, -1]]
    with pytest.raises(AssertionError):
        compare.compare_verify(o, Result([b], bad, [b + 1], o["pos_status"]), d, win, 8)
    # an accepted draft that is not the request's: invalid
    if b == 1:
        with pytest.raises(AssertionError):
            compare.compare_verify(o, Result([1], [[5, int(o["alt_draw"][0, 1])]], [2], o["pos_status"]), d, win, 8)
    # a token after the emitted one: invalid
    with pytest.raises(AssertionError):
        compare.compare_verify(o, Result([0], [[int(o["alt_draw"][0, 0]), 1]], [1], o["pos_status"]), d, win, 8)


def test_unflagged_request_must_match_exactly():
    tgt, drf, args = ratio_near_tie_case()
    tgt[0, 0, 1] = 3.0   # p/q far from u now: no flag
    o = oracle.verify_chain(tgt, drf, **args)
    assert o["flags"][0] == 0
    a = int(o["accept_len"][0])
    b = 1 - a
    tok = [[1, int(o["alt_draw"][0, 1])]] if b == 1 else [[int(o["alt_draw"][0, 0]), -1]]
    with pytest.raises(AssertionError):
        compare.compare_verify(o, Result([b], tok, [b + 1], o["pos_status"]), args["draft_tokens"], np.array([1]), 8)


def cut_near_tie_row():
    """A vocab-6 fp32 row and a top_p whose top-p prefix after two tokens lies
    within 1e-9 of top_p * Z1 at T = 1 (a small last logit tuned in ulps)."""
    row = np.array([0.0, -0.7, -1.5, -2.5, -3.0, -7.0], np.float32)
    e = np.exp(row.astype(np.float64))
    top_p = float(np.float32((e[0] + e[1]) / (e[:5].sum() + 1e-3)))
    z_tail = (e[0] + e[1]) / top_p - e[:5].sum()
    base = np.log(z_tail)
    best, best_m = None, np.inf
    for s in range(-300, 301):
        row[5] = _nudge(base, s)
        m = oracle.row_transform(row, 1.0, 0, top_p)[0]["cut_margin"]
        if m < best_m:
            best, best_m = row[5], m
    row[5] = best
    assert best_m < 1e-9
    return row, top_p


def test_near_top_p_cut_lets_the_draw_take_the_support():
    row, top_p = cut_near_tie_row()
    d, probs = oracle.row_transform(row, 1.0, 0, top_p)
    assert d["next_index"] >= 0
    V = len(row)
    # one request, K = 1: both target rows and the draft row are this row, so
    # every ratio is 1 and the draft is accepted; the bonus draws from p_1
    tgt = np.stack([row, row])[None]
    drf = row[None, None].copy()
    args = dict(draft_tokens=np.array([[0]], np.int32), temperature=np.array([1.0], np.float32),
                top_k=np.array([0], np.int32), top_p=np.array([top_p], np.float32), seed=3)
    o = oracle.verify_chain(tgt, drf, **args)
    assert o["flags"][0] & oracle.FLAG_CUTOFF and o["accept_len"][0] == 1
    assert o["alt_dec"][0, 1] & oracle.ALT_DRAW_ROW
    win = np.array([1])
    support = set(np.nonzero(probs > 0)[0].tolist()) | {d["next_index"]}
    for t in range(V):
        res = Result([1], [[0, t]], [2], o["pos_status"])
        if t in support:
            compare.compare_verify(o, res, args["draft_tokens"], win, V)
        else:
            with pytest.raises(AssertionError):
                compare.compare_verify(o, res, args["draft_tokens"], win, V)


def test_flag_rate_bound_is_enforced():
    tgt, drf, args = ratio_near_tie_case()
    o = oracle.verify_chain(tgt, drf, **args)
    res = Result(o["accept_len"], o["out_tokens"], o["num_emitted"], o["pos_status"])
    assert o["n_flag"][0] >= 1 and o["n_dec"][0] >= 2
    compare.compare_verify(o, res, args["draft_tokens"], np.array([1]), 8, max_flag_rate=1.0)
    with pytest.raises(AssertionError):
        compare.compare_verify(o, res, args["draft_tokens"], np.array([1]), 8, max_flag_rate=1e-4)


def test_block_alternatives_follow_the_last_stop():
    # block verification of the ratio case: one drafted position, so the stop
    # test at 1 is the chain's test and the same two outcomes are allowed
    tgt, drf, args = ratio_near_tie_case()
    o = oracle.verify_chain(tgt, drf, block=True, **args)
    assert o["flags"][0] & oracle.FLAG_RATIO
    assert sorted(compare.valid_accepts(o["alt_dec"][0], 1, True)) == [0, 1]
    # decisions with no ambiguity: only the last passing stop test counts
    dec = np.array([0, oracle.ALT_ACCEPT, 0, oracle.ALT_ACCEPT, 0])
    assert compare.valid_accepts(dec, 4, True) == [3]
    dec[4] = oracle.ALT_AMBIG
    assert compare.valid_accepts(dec, 4, True) == [3, 4]
    # the chain reading of the same bits: stop at the first rejection
    assert compare.valid_accepts(np.array([oracle.ALT_ACCEPT, 0, oracle.ALT_ACCEPT]), 3, False) == [1]


def test_alternatives_agree_with_the_oracle_path_on_random_cases():
    # on unflagged random requests, the per-position table reproduces the
    # oracle's own outcome: its accepted length is the only one allowed and
    # its emitted token is the draw at that position
    from speculative_decoding_verification_rows_gb300 import workloads
    from tests.conftest import np_logits
    for seed in range(4):
        w = workloads.random_case(seed, 6, 4, 300, mode="mixed")
        for block in (False, True):
            o = oracle.verify_chain(np_logits(w.target), np_logits(w.draft), w.draft_tokens.numpy(),
                                    w.temperature.numpy(), w.top_k.numpy(), w.top_p.numpy(), seed=seed, block=block)
            for r in range(w.n):
                if o["flags"][r] or o["num_emitted"][r] == 0:
                    continue
                a = int(o["accept_len"][r])
                assert compare.valid_accepts(o["alt_dec"][r], w.K, block) == [a], (seed, r, block)
                assert o["alt_draw"][r, a] == o["out_tokens"][r, a], (seed, r, block)
