"""Pins of the oracle's budget choice from a step-cost table and of its
acceptance-against-trimming counters (NVIDIA/TensorRT-LLM PR #17056:
description "What is here / Planner", review commit "Cost model", the
trim_regret_rate commit).

The checks are closed forms (uniform confidence, where the planner's selection
is known in advance), the planner's own selection (pinned separately against a
brute-force sort) as an independent route to tau, special cases the pages
state (no table or a flat one: no trimming), invariances, and hand counts.
"""
import numpy as np
import pytest

import oracle


def _uniform_tau(n, c, m):
    """tau for n requests that each submit m drafted positions of confidence c:
    n * (1 + c + c^2 + ... + c^m) by the geometric series."""
    if c == 1.0:
        return n * (1.0 + m)
    return n * (1.0 + c * (1.0 - c ** m) / (1.0 - c))


def _shelves(n, K, cost_of_m):
    """A table with one shelf per whole-window depth m: n * (m + 1) tokens."""
    toks = [n * (m + 1) for m in range(K + 1)]
    return toks, [cost_of_m(m) for m in range(K + 1)]


@pytest.mark.parametrize("c,a,b", [(0.9, 1.0, 0.2), (0.6, 1.0, 0.2), (0.95, 3.0, 0.1), (0.5, 0.2, 0.4)])
def test_uniform_confidence_closed_form(c, a, b):
    # All survivals of depth i tie; the planner fills whole depths, so the
    # budget lands on a shelf n (m + 1) and tau has the closed form above.
    n, K = 8, 6
    toks, costs = _shelves(n, K, lambda m: a + b * m)
    conf = np.full((n, K), c, np.float32)
    B, th, margin, st = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1))
    thetas = [_uniform_tau(n, c, m) / (a + b * m) for m in range(K + 1)]
    best = max(thetas)
    m_star = max(m for m in range(K + 1) if thetas[m] >= best * (1 - 1e-12))
    assert st == 0
    assert B == n * (m_star + 1)
    assert th == pytest.approx(best, rel=1e-5)     # survivals are fp32 products


def test_not_unimodal_staircase_takes_the_global_argmax():
    # Theta rises to a local maximum at depth 1, falls at depth 2 and 3 (a
    # shelf jump), and rises again to a higher maximum at depth 5.
    n, K, c = 4, 6, 0.95
    costs_m = [1.0, 1.4, 2.6, 2.7, 2.75, 2.8, 4.5]
    toks, costs = _shelves(n, K, lambda m: costs_m[m])
    conf = np.full((n, K), c, np.float32)
    thetas = [_uniform_tau(n, c, m) / costs_m[m] for m in range(K + 1)]
    assert thetas[1] > thetas[2] and thetas[5] > thetas[1]      # the shape this test needs
    B, _, _, _ = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1))
    assert B == n * (int(np.argmax(thetas)) + 1)


def test_tau_through_the_planner_selection():
    # tau(B) from the planner's own selection (windows v_r, survivals by numpy
    # cumprod) must reach the chosen Theta at the chosen B and nowhere exceed it.
    rng = np.random.default_rng(5)
    for trial in range(30):
        n, K = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        conf = rng.uniform(0.0, 1.0, (n, K)).astype(np.float32)
        conf[rng.uniform(size=(n, K)) < 0.2] = 1.0
        bucket = n + int(rng.integers(0, n * K + 2))
        n_sh = int(rng.integers(1, 6))
        toks = np.sort(rng.choice(np.arange(1, n * (K + 1) + 3), n_sh, replace=False)).astype(np.int32)
        costs = np.sort(rng.uniform(0.5, 3.0, n_sh)).astype(np.float32)
        fixed = float(np.float32(rng.uniform(0, 1)))   # the table is fp32
        B, th, margin, st = oracle.choose_budget(conf, toks, costs, bucket, fixed_overhead_ms=fixed)
        surv = np.cumprod(conf, axis=1, dtype=np.float32)
        b_max = n + min(n * K, bucket - n)
        feasible = [b for b in range(n, b_max + 1) if (toks >= b).any()]
        if not feasible:
            assert st & 2 and B == b_max
            continue

        def theta(b):
            vl, _, _, _ = oracle.plan_budget(conf, b, max(bucket, b))
            tau = n + sum(float(surv[r, :vl[r]].astype(np.float64).sum()) for r in range(n))
            shelf = int(np.argmax(toks >= b))
            return tau / (float(costs[shelf]) + fixed)

        vals = {b: theta(b) for b in feasible}
        assert B in vals
        assert vals[B] == pytest.approx(th, rel=1e-9)
        assert all(v <= th * (1 + 1e-9) for v in vals.values())
        # ties go to the larger budget
        assert all(b <= B for b, v in vals.items() if v >= th * (1 - 1e-12) and margin > 1e-9)


def test_no_table_or_flat_table_does_not_trim():
    rng = np.random.default_rng(7)
    conf = rng.uniform(0.2, 1.0, (6, 5)).astype(np.float32)
    n, K = conf.shape
    B, _, _, st = oracle.choose_budget(conf, None, None, bucket=64)
    assert B == n + n * K and st & 2
    B, _, _, st = oracle.choose_budget(conf, [10, 20, 40], [2.0, 2.0, 2.0], bucket=64)
    assert B == n + n * K and st == 0
    # a table none of whose shelves holds even the anchors
    B, _, _, st = oracle.choose_budget(conf, [2, 4], [1.0, 2.0], bucket=64)
    assert B == n + n * K and st & 2
    # the bucket caps the budget
    B, _, _, _ = oracle.choose_budget(conf, [64], [1.0], bucket=20)
    assert B == 20


def test_bad_tables_do_not_trim():
    conf = np.full((4, 3), 0.7, np.float32)
    full = 4 + 4 * 3
    for toks, costs, kw in [([8, 8, 16], [1.0, 1.2, 2.0], {}), ([8, 4], [1.0, 2.0], {}),
                            ([8, 16], [1.0, float("nan")], {}), ([8, 16], [-1.0, 2.0], {}),
                            ([8, 16], [1.0, 2.0], {"fixed_overhead_ms": float("inf")}),
                            ([8, 16], [1.0, 2.0], {"batch_sizes": [4], "batch_overhead_ms": [-0.5]})]:
        B, _, _, st = oracle.choose_budget(conf, toks, costs, bucket=64, **kw)
        assert B == full and st == 4, (toks, costs, kw)


def test_fixed_overheads_move_the_choice_and_scaling_does_not():
    n, K, c = 8, 6, 0.8
    toks, costs = _shelves(n, K, lambda m: 1.0 + 0.5 * m)
    conf = np.full((n, K), c, np.float32)
    b0, _, _, _ = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1))
    b1, _, _, _ = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1), fixed_overhead_ms=1000.0)
    assert b1 == n * (K + 1) and b0 < b1          # a large non-trimmable term: every token counts
    for lam in (0.25, 3.0, 17.0):
        b2, _, _, _ = oracle.choose_budget(conf, toks, (np.array(costs) * lam).tolist(), bucket=n * (K + 1),
                                           fixed_overhead_ms=0.3 * lam, batch_sizes=[4, 16],
                                           batch_overhead_ms=[0.1 * lam, 0.2 * lam])
        b3, _, _, _ = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1), fixed_overhead_ms=0.3,
                                           batch_sizes=[4, 16], batch_overhead_ms=[0.1, 0.2])
        assert b2 == b3
    # the batch staircase: n = 8 takes the entry for 16; above the last, the last
    _, th_a, _, _ = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1), batch_sizes=[4, 16],
                                         batch_overhead_ms=[0.0, 0.7])
    _, th_b, _, _ = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1), fixed_overhead_ms=0.7)
    _, th_c, _, _ = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1), batch_sizes=[2, 4],
                                         batch_overhead_ms=[0.0, 0.7])
    assert th_a == th_b == th_c


def test_shelves_count_the_bonus_token():
    # The review's "Cost model": tokens submitted = bs * (verify_len + 1).  With
    # one shelf per depth at n (m + 1) tokens, depth m costs costs[m]; a lookup
    # without the bonus row would price depth m at a deeper shelf.
    n, K, c = 8, 5, 0.9
    costs_m = [1.0, 1.1, 3.0, 3.1, 3.2, 3.3]
    toks, costs = _shelves(n, K, lambda m: costs_m[m])
    conf = np.full((n, K), c, np.float32)
    B, _, _, _ = oracle.choose_budget(conf, toks, costs, bucket=n * (K + 1))
    thetas = [_uniform_tau(n, c, m) / costs_m[m] for m in range(K + 1)]
    assert B == n * (int(np.argmax(thetas)) + 1)


def test_verify_stats_by_hand():
    # r0 trimmed (v 2 < K 4) and accepted all 2: a regret.  r1 and r5 trimmed,
    # stopped inside their windows.  r2 untrimmed (v = K).  r3 an error
    # (nothing emitted).  r4 K_r = 1 by its own draft length, v 1: untrimmed.
    acc = [2, 0, 3, 0, 1, 1]
    emitted = [3, 1, 4, 0, 2, 2]
    vl = [2, 3, 4, 1, 1, 3]
    dl = [4, 4, 4, 4, 1, 4]
    assert oracle.verify_stats(acc, emitted, vl, 4, dl) == (3 + 1 + 4 + 2 + 2, 3 + 4 + 5 + 2 + 4, 3, 1)
    # no verify lengths: every window is K_r, nothing is trimmed
    assert oracle.verify_stats(acc, emitted, None, 4, dl) == (12, 5 + 5 + 5 + 2 + 5, 0, 0)


def test_budget_pins_catch_planted_mistakes(tmp_path):
    with oracle.planted(6, str(tmp_path)):       # table looked up without the bonus row
        with pytest.raises(AssertionError):
            test_shelves_count_the_bonus_token()
    with oracle.planted(7, str(tmp_path)):       # first descent
        with pytest.raises(AssertionError):
            test_not_unimodal_staircase_takes_the_global_argmax()
    with oracle.planted(8, str(tmp_path)):       # regret counted on the wrong side
        with pytest.raises(AssertionError):
            test_verify_stats_by_hand()
