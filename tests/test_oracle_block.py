"""Pins of the oracle's block verification (local-inference-lab/rtx6kpro
dspark-upstream-consolidation.md, rejection_sample_method "block": joint block
acceptance with residual-mass reweighting; the algorithm of Sun et al.,
"Block Verification Accelerates Speculative Decoding", 2024).

What fixes it: with one drafted position it is the token-by-token test; at
temperature 0 it is the greedy rule (the page: "temp-0 equivalence exact");
when the draft equals the target every draft is accepted; generation by
repeated block steps emits exactly the target distribution (the paper's
theorem, checked by chi-square on whole generated sequences); and its
expected accepted length is at least the token-by-token one.
"""
import numpy as np
import pytest
import scipy.stats

import oracle


def _iid_case(rng, n, K, P, Q, seed_T=1.0):
    """n requests whose every target row is log P and draft row log Q (fp32),
    drafts sampled from Q with the test's own generator."""
    V = len(P)
    tgt = np.broadcast_to(np.log(P).astype(np.float32), (n, K + 1, V)).copy()
    drf = np.broadcast_to(np.log(Q).astype(np.float32), (n, K, V)).copy()
    d = rng.choice(V, size=(n, K), p=Q).astype(np.int32)
    T = np.full(n, seed_T, np.float32)
    return tgt, drf, d, T


def test_one_position_is_the_token_test():
    rng = np.random.default_rng(1)
    for trial in range(5):
        n, V = 400, 7
        tgt = rng.normal(0, 1.5, (n, 2, V)).astype(np.float32)
        drf = rng.normal(0, 1.5, (n, 1, V)).astype(np.float32)
        d = rng.integers(0, V, (n, 1)).astype(np.int32)
        T = rng.choice([0.5, 1.0, 1.3], n).astype(np.float32)
        tk = rng.choice([0, 3], n).astype(np.int32)
        tp = rng.choice([1.0, 0.8], n).astype(np.float32)
        a = oracle.verify_chain(tgt, drf, d, T, tk, tp, seed=trial)
        b = oracle.verify_chain(tgt, drf, d, T, tk, tp, seed=trial, block=True)
        for key in ("accept_len", "out_tokens", "num_emitted", "pos_status"):
            assert np.array_equal(a[key], b[key]), key


def test_greedy_requests_take_the_greedy_rule():
    rng = np.random.default_rng(2)
    n, K, V = 300, 5, 11
    tgt = rng.integers(-3, 4, (n, K + 1, V)).astype(np.float32)   # ties on purpose
    d = rng.integers(0, V, (n, K)).astype(np.int32)
    T = np.zeros(n, np.float32)
    a = oracle.verify_chain(tgt, None, d, T)
    b = oracle.verify_chain(tgt, None, d, T, block=True)
    for key in ("accept_len", "out_tokens", "num_emitted"):
        assert np.array_equal(a[key], b[key]), key


def test_draft_equal_to_target_accepts_everything():
    rng = np.random.default_rng(3)
    n, K, V = 200, 6, 9
    tgt = rng.normal(0, 2, (n, K + 1, V)).astype(np.float32)
    drf = tgt[:, :K].copy()
    d = rng.integers(0, V, (n, K)).astype(np.int32)
    T = np.full(n, 0.8, np.float32)
    # the drafts must lie in the kept set of q for the ratio to be defined: no top-k / top-p here
    o = oracle.verify_chain(tgt, drf, d, T, block=True)
    assert (o["accept_len"] == K).all()
    assert (o["num_emitted"] == K + 1).all()


def _generate(P, Q, K, n, L, seed0, block):
    """n sequences of L tokens by repeated verify steps (fresh drafts each step)."""
    rng = np.random.default_rng(seed0)
    V = len(P)
    seqs = [[] for _ in range(n)]
    step = 0
    while True:
        live = [i for i in range(n) if len(seqs[i]) < L]
        if not live:
            break
        tgt, drf, d, T = _iid_case(rng, len(live), K, P, Q)
        o = oracle.verify_chain(tgt, drf, d, T, seed=1000 + step, block=block)
        for row, i in enumerate(live):
            seqs[i].extend(o["out_tokens"][row, :o["num_emitted"][row]].tolist())
        step += 1
    codes = np.array([sum(s[j] * V ** j for j in range(L)) for s in seqs])
    return codes, seqs


def _chi2_sequences(P, codes, L):
    V = len(P)
    counts = np.bincount(codes, minlength=V ** L)
    expect = np.ones(V ** L)
    for c in range(V ** L):
        x = c
        for j in range(L):
            expect[c] *= P[x % V]
            x //= V
    expect *= len(codes)
    keep = expect >= 5
    stat = ((counts[keep] - expect[keep]) ** 2 / expect[keep]).sum() + \
        (counts[~keep].sum() - expect[~keep].sum()) ** 2 / max(expect[~keep].sum(), 1e-12)
    return scipy.stats.chi2.sf(stat, keep.sum())


PQ = (np.array([0.45, 0.25, 0.2, 0.1]), np.array([0.1, 0.3, 0.25, 0.35]))


def test_generation_by_block_steps_emits_the_target():
    P, Q = PQ
    codes, _ = _generate(P, Q, K=2, n=60_000, L=3, seed0=5, block=True)
    assert _chi2_sequences(P, codes, 3) > 1e-3


def test_block_accepts_at_least_as_much_as_the_token_test():
    P, Q = PQ
    rng = np.random.default_rng(6)
    n, K = 40_000, 4
    tgt, drf, d, T = _iid_case(rng, n, K, P, Q)
    a = oracle.verify_chain(tgt, drf, d, T, seed=77)
    b = oracle.verify_chain(tgt, drf, d, T, seed=77, block=True)
    ma, mb = a["accept_len"].mean(), b["accept_len"].mean()
    sd = np.sqrt((a["accept_len"].var() + b["accept_len"].var()) / n)
    assert mb > ma - 3 * sd
    assert mb > ma            # strictly more on this pair (the paper's gain), by far more than the noise
    assert mb - ma > 5 * sd


def test_block_pin_catches_the_unweighted_residual(tmp_path):
    P, Q = PQ
    with oracle.planted(9, str(tmp_path)):
        codes, _ = _generate(P, Q, K=2, n=60_000, L=3, seed0=5, block=True)
        assert _chi2_sequences(P, codes, 3) < 1e-6
