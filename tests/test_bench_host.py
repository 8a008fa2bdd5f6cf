"""Host logic of bench.py on CPU: the small-top-k promise the bench passes and
the byte accounting of the two row paths agree for every workload."""
import pytest

import bench
from speculative_decoding_verification_rows_gb300 import workloads

SMALL = {"tiny": {}, "medium": dict(n=3, V=2_000), "large": dict(n=3, V=2_000),
         "greedy_wide": dict(n=3, V=2_000), "ragged": dict(n=8, V=2_000, budget=40, bucket=48)}


@pytest.mark.parametrize("name,promise", [("tiny", True), ("medium", False), ("large", True),
                                          ("greedy_wide", True), ("ragged", False)])
def test_promise_matches_the_row_paths(name, promise):
    w = workloads.make(name, device="cpu", scale=SMALL[name])
    assert bench.small_topk(w) is promise
    fast, hist = bench.path_bytes(w)
    # under the promise no row takes the histogram path; without it some do
    assert (hist == 0) is promise
    assert fast + hist > 0


def test_greedy_rows_follow_the_histogram_path_in_mixed_chain_batches():
    # ragged mixes greedy and full-vocabulary requests: chain verification
    # sends the greedy rows to the histogram kernel as argmax scans, block
    # verification keeps them on the one-pass kernel
    w = workloads.make("ragged", device="cpu", scale=SMALL["ragged"])
    fast_c, hist_c = bench.path_bytes(w, None, "chain")
    fast_b, hist_b = bench.path_bytes(w, None, "block")
    assert fast_c == 0 and hist_c == fast_b + hist_b
    assert fast_b > 0 and hist_b > 0
    # a batch with no full-vocabulary request keeps its greedy rows on the one-pass kernel
    w2 = workloads.make("large", device="cpu", scale=SMALL["large"])
    w2.temperature[0] = 0.0
    assert bench.path_bytes(w2, None, "chain")[1] == 0


def test_promise_is_broken_by_one_request():
    w = workloads.make("large", device="cpu", scale=SMALL["large"])
    w.top_k[1] = 33
    assert not bench.small_topk(w)
    w.top_k[1] = 20
    w.temperature[1] = 0.0          # greedy requests keep it whatever their top-k
    w.top_k[1] = 0
    assert bench.small_topk(w)


@pytest.mark.parametrize("name", ["large", "ragged"])
def test_cpu_baseline_times_the_oracle_on_one_pinned_core(name):
    w = workloads.make(name, device="cpu", scale=SMALL[name])
    b = bench.cpu_baseline(w, seconds=0.2)
    assert b["kind"] == "oracle" and b["cores"] == 1 and b["value"] > 0
    assert b["cpu_model"] and b["host_cores"] >= 1
    if name == "ragged":
        # the sample is the plan's packed rows: windows of the planner's lengths
        assert "packed target rows" in b["sample"]


def test_ragged_oracle_sample_follows_the_plan():
    import oracle
    w = workloads.make("ragged", device="cpu", scale=SMALL["ragged"])
    extra = bench.ragged_host_plan(w, None)
    rows, dt = bench.oracle_sample(w, 2, 5, extra)
    vl = extra["verify_lens_host"]
    assert rows == int(sum(vl[2:5]) + 3) and dt >= 0
    # the slice gives what the whole batch gives for those requests
    tgt, drf, qo, v = bench.ragged_slice(w, extra, 0, w.n)
    args = (w.draft_tokens.numpy(), w.temperature.numpy(), w.top_k.numpy(), w.top_p.numpy())
    full = oracle.verify_ragged(tgt, drf, qo, v, *args, seed=w.seed)
    tgt, drf, qo, v = bench.ragged_slice(w, extra, 2, 5)
    part = oracle.verify_ragged(tgt, drf, qo, v, *(a[2:5] for a in args), seed=w.seed, first_req=2)
    assert (part["out_tokens"] == full["out_tokens"][2:5]).all()
