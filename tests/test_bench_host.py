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


def test_promise_is_broken_by_one_request():
    w = workloads.make("large", device="cpu", scale=SMALL["large"])
    w.top_k[1] = 33
    assert not bench.small_topk(w)
    w.top_k[1] = 20
    w.temperature[1] = 0.0          # greedy requests keep it whatever their top-k
    w.top_k[1] = 0
    assert bench.small_topk(w)
