"""The small-top-k promise (SV_SAMPLING_SMALL_TOPK) through the C ABI (needs a GB300).

Under the promise a call launches only its prep, the one-pass row kernel and
the chain (or row output) kernels.  A batch that keeps the promise gives the
same outputs as without it, and the oracle's; a request that breaks it is
refused (SV_ROW_UNSUPPORTED at position 0, nothing accepted or emitted) while
every other request gives the outputs of the call without the promise.
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
FIELDS = ("accept_len", "out_tokens", "num_emitted", "row_status")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv_build.build()
    sv.load()


def _small_case(seed, n, K, V, dtype=torch.bfloat16):
    """Top-k in 1..20 at T > 0 for most requests, greedy for every third."""
    w = workloads.random_case(seed, n, K, V, dtype=dtype, device=DEV, mode="topk")
    w.temperature[::3] = 0.0
    return w


def _keeps_promise(w):
    T = w.temperature.cpu().numpy()
    k = w.top_k.cpu().numpy()
    return (T == 0.0) | ((k >= 1) & (k <= 32))


def _run(w, small, seed):
    o = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=seed,
                        small_topk=small)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("seed,V,dtype", [(0, 30_000, torch.bfloat16), (1, 4_099, torch.bfloat16),
                                          (2, 9_000, torch.float32)])
def test_kept_promise_matches_oracle_and_the_unpromised_call(seed, V, dtype):
    w = _small_case(seed, 24, 4, V, dtype)
    assert _keeps_promise(w).all()
    a = _run(w, True, seed)
    b = _run(w, False, seed)
    for f in FIELDS:
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    o = oracle.verify_chain(np_logits(w.target), np_logits(w.draft), w.draft_tokens.cpu().numpy(),
                            w.temperature.cpu().numpy(), w.top_k.cpu().numpy(), w.top_p.cpu().numpy(), seed=seed)
    compare_verify(o, a, w.draft_tokens.cpu().numpy(), np.full(w.n, w.K), w.V)


@pytest.mark.parametrize("seed", range(2))
def test_broken_promise_refuses_only_those_requests(seed):
    # the mixed menu has top-k off, k = V - 1, V and 64: those sampling
    # requests break the promise
    w = workloads.random_case(10 + seed, 40, 3, 20_000, device=DEV, mode="mixed")
    ok = _keeps_promise(w)
    assert ok.any() and (~ok).any()
    a = _run(w, True, seed)
    b = _run(w, False, seed)
    acc, nem = a.accept_len.cpu().numpy(), a.num_emitted.cpu().numpy()
    tok, st = a.out_tokens.cpu().numpy(), a.row_status.cpu().numpy()
    bad = np.nonzero(~ok)[0]
    assert (st[bad, 0] & sv.ROW_UNSUPPORTED != 0).all()
    assert (acc[bad] == 0).all() and (nem[bad] == 0).all() and (tok[bad] == -1).all()
    good = torch.from_numpy(np.nonzero(ok)[0]).to(DEV)
    for f in FIELDS:
        assert torch.equal(getattr(a, f)[good], getattr(b, f)[good]), f


def test_ragged_with_promise_equals_without():
    w = _small_case(3, 16, 5, 12_345)
    n, K = w.n, w.K
    vl = torch.from_numpy(np.random.default_rng(3).integers(0, K + 1, n).astype(np.int32))
    qo = torch.zeros(n + 1, dtype=torch.int32)
    qo[1:] = torch.cumsum(vl + 1, 0)
    bucket = int(qo[-1]) + 5
    packed = torch.zeros((bucket, w.V), dtype=w.target.dtype, device=DEV)
    for r in range(n):
        packed[int(qo[r]):int(qo[r + 1])] = w.target[r, :int(vl[r]) + 1]
    args = (packed, w.draft, qo.to(DEV), vl.to(DEV), w.draft_tokens, w.temperature, w.top_k, w.top_p)
    a = sv.verify_ragged(*args, seed=4, small_topk=True)
    b = sv.verify_ragged(*args, seed=4)
    torch.cuda.synchronize()
    for f in FIELDS:
        assert torch.equal(getattr(a, f), getattr(b, f)), f


def test_build_target_probs_with_promise():
    w = workloads.random_case(4, 12, 1, 7_001, device=DEV, mode="mixed")
    logits = w.target.reshape(-1, w.V)
    rows = logits.shape[0]
    rr = torch.arange(rows, device=DEV, dtype=torch.int32) // 2
    toks = torch.randint(0, w.V, (rows,), device=DEV, dtype=torch.int32)
    da, pa, _ = sv.build_target_probs(logits, w.temperature, w.top_k, w.top_p, row_to_req=rr, tokens=toks,
                                      small_topk=True)
    db, pb, _ = sv.build_target_probs(logits, w.temperature, w.top_k, w.top_p, row_to_req=rr, tokens=toks)
    torch.cuda.synchronize()
    ok_req = _keeps_promise(w)
    ok = ok_req[rr.cpu().numpy()]
    assert ok.any() and (~ok).any()
    sa = sv.desc_fields(da)["status"]
    assert (sa[~ok] == sv.ROW_UNSUPPORTED).all()
    good = torch.from_numpy(np.nonzero(ok)[0]).to(DEV)
    assert torch.equal(da[good], db[good])
    assert torch.equal(pa[good], pb[good])


class _Rows:
    def __init__(self, o, a, b):
        self.accept_len, self.out_tokens = o.accept_len[a:b], o.out_tokens[a:b]
        self.num_emitted, self.row_status = o.num_emitted[a:b], o.row_status[a:b]


@pytest.mark.parametrize("name,slices", [("large", [(0, 3), (61, 63), (125, 128)]),
                                         ("greedy_wide", [(0, 8), (250, 258), (504, 512)])])
def test_benchmark_step_at_full_size(name, slices):
    # the step exactly as the benchmark times it: its own closure (with the
    # promise), captured once as a CUDA graph and replayed
    import bench
    w = workloads.make(name, device=DEV)
    step, out, extra = bench.make_step(w, sv, torch.device(DEV, torch.cuda.current_device()))
    assert extra is None and bench.small_topk(w)
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for f in FIELDS:
        getattr(out, f).fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    plain = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=w.seed)
    torch.cuda.synchronize()
    for f in FIELDS:
        assert torch.equal(getattr(out, f), getattr(plain, f)), f
    for a, b in slices:
        o = oracle.verify_chain(np_logits(w.target[a:b]), None if w.draft is None else np_logits(w.draft[a:b]),
                                w.draft_tokens[a:b].cpu().numpy(), w.temperature[a:b].cpu().numpy(),
                                w.top_k[a:b].cpu().numpy(), w.top_p[a:b].cpu().numpy(), seed=w.seed, first_req=a)
        compare_verify(o, _Rows(out, a, b), w.draft_tokens[a:b].cpu().numpy(), np.full(b - a, w.K), w.V,
                       max_flag_rate=1e-4)
