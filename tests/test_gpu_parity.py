"""CUDA path against the oracle on the same seeded inputs (needs a GB300).

Every call goes through the C ABI (libsv.so) via the thin binding.  Sizes the
oracle finishes in seconds are compared element by element; the full-size
workloads are compared on requests sampled from the batch (the oracle keys
their uniforms by their index in the full batch), in the same launch
configuration the benchmark uses.
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
# Full-size comparisons: flagged decisions (inside the oracle's margins) must
# stay below this fraction of all decisions compared.
FULL_SIZE_FLAG_RATE = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv_build.build()
    sv.load()


def run_chain(w, verify_len=None, seed=0):
    return sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p,
                           verify_len=verify_len, seed=seed)


def oracle_chain(w, req_slice=slice(None), verify_len=None, seed=0):
    rs = req_slice
    first = rs.start or 0
    return oracle.verify_chain(np_logits(w.target[rs]), None if w.draft is None else np_logits(w.draft[rs]),
                               w.draft_tokens[rs].cpu().numpy(), w.temperature[rs].cpu().numpy(),
                               w.top_k[rs].cpu().numpy(), w.top_p[rs].cpu().numpy(),
                               verify_len=None if verify_len is None else verify_len[rs].cpu().numpy(),
                               seed=seed, first_req=first)


class _Slice:
    def __init__(self, o, rs):
        self.accept_len, self.out_tokens = o.accept_len[rs], o.out_tokens[rs]
        self.num_emitted, self.row_status = o.num_emitted[rs], o.row_status[rs]


def check(w, req_slice=slice(None), verify_len=None, seed=0, max_flag_rate=None):
    g = run_chain(w, verify_len, seed)
    torch.cuda.synchronize()
    o = oracle_chain(w, req_slice, verify_len, seed)
    n = len(o["accept_len"])
    win = np.full(n, w.K) if verify_len is None else verify_len[req_slice].cpu().numpy()
    return compare_verify(o, _Slice(g, req_slice), w.draft_tokens[req_slice].cpu().numpy(), win, w.V,
                          max_flag_rate)


def test_tiny_config_full_size():
    w = workloads.make("tiny", device=DEV)
    check(w)


@pytest.mark.parametrize("name,scale", [("medium", dict(n=6)), ("large", dict(n=4)),
                                        ("greedy_wide", dict(n=64))])
def test_configs_full_vocab_few_requests(name, scale):
    w = workloads.make(name, device=DEV, scale=scale)
    check(w)


def test_large_full_batch_sampled_requests():
    w = workloads.make("large", device=DEV)          # 128 x 8 rows x 248,320 bf16, the benchmark workload
    for rs in (slice(0, 3), slice(61, 63), slice(125, 128)):
        check(w, rs, max_flag_rate=FULL_SIZE_FLAG_RATE)


def test_greedy_wide_full_batch():
    w = workloads.make("greedy_wide", device=DEV)    # 512 x 8 rows x 129,280: greedy is cheap for the oracle
    check(w, max_flag_rate=FULL_SIZE_FLAG_RATE)


def test_medium_full_batch_sampled_requests():
    w = workloads.make("medium", device=DEV)
    check(w, slice(0, 3), max_flag_rate=FULL_SIZE_FLAG_RATE)
    check(w, slice(29, 32), max_flag_rate=FULL_SIZE_FLAG_RATE)


@pytest.mark.parametrize("seed", range(6))
def test_random_mixed_small(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.choice([1, 2, 3, 7, 16, 31, 33, 100, 257, 1000, 4099, 20000]))
    n, K = int(rng.integers(1, 12)), int(rng.integers(0, 6))
    w = workloads.random_case(seed, n, K, V, device=DEV, mode="mixed")
    vl = torch.randint(0, K + 1, (n,), dtype=torch.int32, device=DEV) if seed % 2 else None
    check(w, verify_len=vl, seed=seed)


@pytest.mark.parametrize("seed", range(4))
def test_random_fp32_fast_path(seed):
    rng = np.random.default_rng(100 + seed)
    V = int(rng.choice([5, 64, 999, 9000]))
    w = workloads.random_case(seed, 6, 3, V, dtype=torch.float32, device=DEV, mode="topk")
    check(w, seed=seed)


def test_build_target_probs_matches_oracle():
    for seed, V, mode in [(0, 4099, "mixed"), (1, 151_936, "full"), (2, 248_320, "topk"), (3, 33, "mixed")]:
        w = workloads.random_case(seed, 5, 1, V, device=DEV, mode=mode)
        logits = w.target.reshape(-1, V)
        rows = logits.shape[0]
        rr = torch.arange(rows, device=DEV, dtype=torch.int32) // 2
        toks = torch.randint(0, V, (rows,), device=DEV, dtype=torch.int32)
        desc, ptok, dense = sv.build_target_probs(logits, w.temperature, w.top_k, w.top_p, row_to_req=rr,
                                                  tokens=toks, dense=True)
        torch.cuda.synchronize()
        d = sv.desc_fields(desc)
        host = np_logits(logits)
        for i in range(rows):
            q = int(rr[i])
            od, op = oracle.row_transform(host[i], float(w.temperature[q]), int(w.top_k[q]), float(w.top_p[q]))
            assert d["status"][i] == od["status"], (i, d["status"][i], od)
            assert d["argmax"][i] == od["argmax"]
            if od["cut_margin"] < 1e-9:
                continue
            assert d["kept"][i] == od["kept"] and d["cutoff_ties"][i] == od["cutoff_ties"], (i, V, mode)
            assert d["cutoff_logit"][i] == np.float32(od["cutoff_logit"])
            assert d["max_logit"][i] == np.float32(od["max_logit"])
            assert abs(d["log_norm"][i] - od["log_norm"]) <= 1e-5 * max(1.0, abs(od["log_norm"]))
            g = dense[i].cpu().numpy().astype(np.float64)
            np.testing.assert_allclose(g, op, rtol=1e-5, atol=1e-30)
            t = int(toks[i])
            assert abs(float(ptok[i]) - op[t]) <= 1e-5 * op[t] + 1e-30


def test_emitted_token_follows_p_on_gpu():
    # chi-square over 10^6 draws at vocab 16: draft d ~ q, first emitted token ~ p
    import scipy.stats
    n = 1_000_000
    p = np.arange(1, 17, dtype=np.float64)
    p /= p.sum()
    q = np.arange(16, 0, -1, dtype=np.float64)
    q /= q.sum()
    rng = np.random.default_rng(21)
    d = torch.from_numpy(rng.choice(16, size=n, p=q).astype(np.int32)).view(n, 1).to(DEV)
    tgt = torch.from_numpy(np.log(p).astype(np.float32)).to(DEV).expand(n, 2, 16).contiguous()
    drf = torch.from_numpy(np.log(q).astype(np.float32)).to(DEV).expand(n, 1, 16).contiguous()
    T = torch.ones(n, device=DEV)
    o = sv.verify_chain(tgt, drf, d, T, seed=21)
    first = o.out_tokens[:, 0].cpu().numpy()
    counts = np.bincount(first, minlength=16)
    assert scipy.stats.chisquare(counts, n * p).pvalue > 1e-3
    acc = o.accept_len.float().mean().item()
    ref = np.minimum(p, q).sum()
    assert abs(acc - ref) < 5 * np.sqrt(ref * (1 - ref) / n)


def test_planner_matches_oracle_bit_exact():
    w = workloads.make("ragged", device=DEV, scale=dict(V=64))
    vl, qo, tot, st = sv.plan_budget(w.conf, w.budget, w.bucket)
    ovl, oqo, otot, ost = oracle.plan_budget(w.conf.cpu().numpy(), w.budget, w.bucket)
    assert vl.cpu().numpy().tolist() == ovl.tolist()
    assert qo.cpu().numpy().tolist() == oqo.tolist()
    assert int(tot) == otot == w.budget and int(st) == ost == 0
    rng = np.random.default_rng(3)
    for trial in range(30):
        n, K = int(rng.integers(1, 40)), int(rng.integers(0, 20))
        conf = rng.choice([0.0, 0.25, 0.5, 0.9, 1.0, 1.5, -0.0, np.nan], size=(n, K)).astype(np.float32) \
            if trial % 2 else rng.random((n, K)).astype(np.float32)
        budget = int(rng.integers(n, n * (K + 1) + 4))
        dl = rng.integers(-2, K + 3, n).astype(np.int32) if trial % 3 == 0 else None
        g = sv.plan_budget(torch.from_numpy(conf).to(DEV), budget, budget + 3,
                           None if dl is None else torch.from_numpy(dl).to(DEV))
        o = oracle.plan_budget(conf, budget, budget + 3, dl)
        assert g[0].cpu().numpy().tolist() == o[0].tolist(), trial
        assert g[1].cpu().numpy().tolist() == o[1].tolist()
        assert int(g[2]) == o[2] and int(g[3]) == o[3]


def _ragged_inputs(w, vl, qo):
    packed = workloads.pack_rows(w.target, qo, vl, w.bucket)
    return packed


def test_ragged_scaled_matches_oracle():
    w = workloads.make("ragged", device=DEV, scale=dict(n=24, V=3001, budget=200, bucket=208))
    ovl, oqo, otot, _ = oracle.plan_budget(w.conf.cpu().numpy(), w.budget, w.bucket)
    packed = _ragged_inputs(w, ovl, oqo)
    vl_d = torch.from_numpy(ovl).to(DEV)
    qo_d = torch.from_numpy(oqo).to(DEV)
    g = sv.verify_ragged(packed, w.draft, qo_d, vl_d, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=5)
    torch.cuda.synchronize()
    o = oracle.verify_ragged(np_logits(packed), np_logits(w.draft), oqo, ovl, w.draft_tokens.cpu().numpy(),
                             w.temperature.cpu().numpy(), w.top_k.cpu().numpy(), w.top_p.cpu().numpy(), seed=5)
    compare_verify(o, g, w.draft_tokens.cpu().numpy(), ovl, w.V)
    # full windows: ragged equals the uniform layout bit for bit
    n, K = w.n, w.K
    full_vl = torch.full((n,), K, dtype=torch.int32, device=DEV)
    full_qo = torch.arange(n + 1, dtype=torch.int32, device=DEV) * (K + 1)
    a = sv.verify_ragged(w.target.reshape(n * (K + 1), -1), w.draft, full_qo, full_vl, w.draft_tokens,
                         w.temperature, w.top_k, w.top_p, seed=5)
    b = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=5)
    for f in ("accept_len", "out_tokens", "num_emitted", "row_status"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f


def test_ragged_full_size_sampled():
    w = workloads.make("ragged", device=DEV)         # 256 x 16 drafted, 2048-token budget, 248,320 vocab
    vl, qo, tot, st = sv.plan_budget(w.conf, w.budget, w.bucket)
    ovl, oqo, otot, _ = oracle.plan_budget(w.conf.cpu().numpy(), w.budget, w.bucket)
    assert vl.cpu().numpy().tolist() == ovl.tolist() and otot == w.budget
    packed = _ragged_inputs(w, ovl, oqo)
    g = sv.verify_ragged(packed, w.draft, qo, vl, w.draft_tokens, w.temperature, w.top_k, w.top_p)
    torch.cuda.synchronize()
    for r0, r1 in ((0, 4), (130, 133), (252, 256)):
        qo_local = oqo[r0:r1 + 1] - oqo[r0]
        rows = packed[int(oqo[r0]):int(oqo[r1])]
        o = oracle.verify_ragged(np_logits(rows), np_logits(w.draft[r0:r1]), qo_local, ovl[r0:r1],
                                 w.draft_tokens[r0:r1].cpu().numpy(), w.temperature[r0:r1].cpu().numpy(),
                                 w.top_k[r0:r1].cpu().numpy(), w.top_p[r0:r1].cpu().numpy(), first_req=r0)
        compare_verify(o, _Slice(g, slice(r0, r1)), w.draft_tokens[r0:r1].cpu().numpy(), ovl[r0:r1], w.V,
                       max_flag_rate=FULL_SIZE_FLAG_RATE)
    acc = g.accept_len.cpu().numpy()
    assert (acc <= vl.cpu().numpy()).all()


def test_edge_cases():
    V, n, K = 64, 8, 3
    w = workloads.random_case(7, n, K, V, device=DEV, mode="mixed")
    t = w.target.clone()
    t[0, 1, 5] = float("nan")                     # non-finite logit in a read row
    t[1, 0, :] = float("-inf")                    # an all -inf row
    t[2, 2, 7] = float("inf")
    toks = w.draft_tokens.clone()
    toks[3, 1] = V                                # token out of range
    toks[4, 0] = -3
    T = w.temperature.clone()
    T[5] = -1.0                                   # invalid temperature
    tp = w.top_p.clone()
    tp[6] = 0.0                                   # invalid top-p
    T[6] = 0.5
    w2 = workloads.Workload(w.name, "chain", n, K, V, w.dtype, t.contiguous(), w.draft, toks, T, w.top_k, tp)
    check(w2)
    g = run_chain(w2)
    st = g.row_status.cpu().numpy()
    assert st[5, 0] & sv.ROW_BAD_PARAM and st[6, 0] & sv.ROW_BAD_PARAM
    assert (g.out_tokens[5] == -1).all() and int(g.num_emitted[5]) == 0


def test_graph_capture_and_no_sync():
    w = workloads.make("ragged", device=DEV, scale=dict(n=16, V=1000, budget=150, bucket=160))
    ovl, oqo, _, _ = oracle.plan_budget(w.conf.cpu().numpy(), w.budget, w.bucket)
    packed = _ragged_inputs(w, ovl, oqo)
    ws_p, ws_v = sv.Workspace(DEV), sv.Workspace(DEV)
    outs = {}

    def step():
        vl, qo, tot, st = sv.plan_budget(w.conf, w.budget, w.bucket, ws=ws_p)
        outs["o"] = sv.verify_ragged(packed, w.draft, qo, vl, w.draft_tokens, w.temperature, w.top_k, w.top_p,
                                     seed=1, ws=ws_v)
        return outs["o"]

    eager = step()
    torch.cuda.synchronize()
    ref = [x.clone() for x in (eager.accept_len, eager.out_tokens, eager.num_emitted, eager.row_status)]
    torch.cuda.set_sync_debug_mode("error")
    try:
        step()
    finally:
        torch.cuda.set_sync_debug_mode(0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    o = outs["o"]
    for a, b in zip(ref, (o.accept_len, o.out_tokens, o.num_emitted, o.row_status)):
        assert torch.equal(a, b)


def test_repeated_runs_are_bitwise_identical():
    w = workloads.make("medium", device=DEV, scale=dict(n=4, V=20000))
    first = run_chain(w, seed=3)
    ref = [x.clone() for x in (first.accept_len, first.out_tokens, first.num_emitted, first.row_status)]
    for _ in range(20):
        o = run_chain(w, seed=3)
        for a, b in zip(ref, (o.accept_len, o.out_tokens, o.num_emitted, o.row_status)):
            assert torch.equal(a, b)


@pytest.mark.parametrize("V", [1, 2, 3, 5])
def test_tiny_vocabularies(V):
    n, K = 6, 3
    g = torch.Generator(device=DEV).manual_seed(V)
    tgt = (torch.randn((n, K + 1, V), generator=g, device=DEV) * 2).to(torch.bfloat16)
    drf = (torch.randn((n, K, V), generator=g, device=DEV) * 2).to(torch.bfloat16)
    toks = torch.randint(0, V, (n, K), generator=g, device=DEV, dtype=torch.int32)
    T = torch.tensor([0.0, 0.5, 1.0, 2.0, 0.5, 1.0], device=DEV)
    tk = torch.tensor([0, 0, 1, 2, 5, 0], device=DEV, dtype=torch.int32)
    tp = torch.tensor([1.0, 0.5, 1.0, 0.9, 1.0, 0.2], device=DEV)
    w = workloads.Workload(f"vocab{V}", "chain", n, K, V, torch.bfloat16, tgt, drf, toks, T, tk, tp)
    check(w, seed=V)
