"""Vocabulary-sharded verify (sv_verify_chain_shard_rows / _merge) on one GPU.

The rows of a step are cut along the vocabulary into N contiguous slices
(N in 2, 3, 4; uneven widths), each slice reduced to its records on its own,
the records stacked in a shuffled shard order and merged.  The outputs must
equal sv_verify_chain's on the whole rows bit for bit, and the oracle's
(which knows nothing of shards) on the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_rows_gb300 import build as sv_build
from speculative_decoding_verification_rows_gb300 import shard, sv, workloads
from tests.compare import compare_verify
from tests.conftest import np_logits

pytestmark = pytest.mark.gpu
DEV = "cuda"
FIELDS = ("accept_len", "out_tokens", "num_emitted", "row_status")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv_build.build()
    sv.load()


def sharded(w, n_shards, verify_len=None, seed=0, order_seed=0):
    recs = []
    for r in range(n_shards):
        v0, v1 = shard.shard_bounds(w.V, n_shards, r)
        t = w.target[..., v0:v1].contiguous()
        d = None if w.draft is None else w.draft[..., v0:v1].contiguous()
        recs.append(sv.verify_chain_shard_rows(t, d, w.draft_tokens, w.temperature, w.top_k, w.top_p, v0, w.V,
                                               verify_len=verify_len))
    perm = np.random.default_rng(order_seed).permutation(n_shards)
    stacked = torch.stack([recs[i] for i in perm])
    return sv.verify_chain_shard_merge(stacked, n_shards, w.draft_tokens, w.temperature, w.top_k, w.top_p, w.V,
                                       verify_len=verify_len, seed=seed)


def check(w, n_shards, req_slice=slice(None), verify_len=None, seed=0):
    g = sharded(w, n_shards, verify_len, seed, order_seed=n_shards)
    ref = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p,
                          verify_len=verify_len, seed=seed)
    torch.cuda.synchronize()
    for f in FIELDS:
        assert torch.equal(getattr(g, f), getattr(ref, f)), f
    rs = req_slice
    o = oracle.verify_chain(np_logits(w.target[rs]), None if w.draft is None else np_logits(w.draft[rs]),
                            w.draft_tokens[rs].cpu().numpy(), w.temperature[rs].cpu().numpy(),
                            w.top_k[rs].cpu().numpy(), w.top_p[rs].cpu().numpy(),
                            verify_len=None if verify_len is None else verify_len[rs].cpu().numpy(),
                            seed=seed, first_req=rs.start or 0)

    class S:
        accept_len, out_tokens = g.accept_len[rs], g.out_tokens[rs]
        num_emitted, row_status = g.num_emitted[rs], g.row_status[rs]
    win = np.full(len(o["accept_len"]), w.K) if verify_len is None else verify_len[rs].cpu().numpy()
    compare_verify(o, S, w.draft_tokens[rs].cpu().numpy(), win, w.V)


@pytest.mark.parametrize("n_shards", [2, 3, 4])
@pytest.mark.parametrize("name,scale", [("tiny", None), ("large", dict(n=4)), ("greedy_wide", dict(n=24))])
def test_sharded_workloads_match_whole_rows_and_oracle(name, scale, n_shards):
    w = workloads.make(name, device=DEV, scale=scale)
    check(w, n_shards)


@pytest.mark.parametrize("seed", range(6))
def test_sharded_random_topk(seed):
    rng = np.random.default_rng(700 + seed)
    V = int(rng.choice([7, 16, 100, 1000, 4099, 20000]))
    n, K = int(rng.integers(1, 10)), int(rng.integers(0, 6))
    dtype = torch.float32 if seed % 3 == 2 else torch.bfloat16
    w = workloads.random_case(seed, n, K, V, dtype=dtype, device=DEV, mode="topk")
    w.temperature[::3] = 0.0   # some greedy requests too
    vl = torch.randint(0, K + 1, (n,), dtype=torch.int32, device=DEV) if seed % 2 else None
    check(w, int(rng.integers(2, min(4, V) + 1)), verify_len=vl, seed=seed)


def test_sharded_full_batch_large():
    w = workloads.make("large", device=DEV)   # the benchmark's batch: 128 x 8 rows x 248,320 bf16
    check(w, 2, req_slice=slice(60, 63))


def test_sharded_refuses_full_vocabulary_kept_sets():
    w = workloads.random_case(3, 8, 3, 3000, device=DEV, mode="mixed")
    g = sharded(w, 3)
    ref = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p)
    torch.cuda.synchronize()
    T = w.temperature.cpu()
    tk = w.top_k.cpu()
    listed = (T == 0) | ((tk >= 1) & (tk <= 32) & (tk < w.V))
    assert (~listed).any() and listed.any()
    for r in range(w.n):
        if listed[r]:
            for f in FIELDS:
                assert torch.equal(getattr(g, f)[r], getattr(ref, f)[r]), (r, f)
        else:
            assert int(g.accept_len[r]) == 0 and int(g.num_emitted[r]) == 0
            assert int(g.row_status[r, 0]) & sv.SV_ROW_UNSUPPORTED
            assert (g.out_tokens[r] == -1).all()


def test_shard_record_layout():
    assert sv.shard_record_bytes() == 264
    with pytest.raises(ValueError):
        shard.shard_bounds(3, 4, 0)
