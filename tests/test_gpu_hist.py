"""The exact-histogram row path (rows whose kept set can exceed 32) against the
oracle, through sv_build_target_probs and sv_verify_chain (needs a GB300).

The rows here are built to reach the path's special cases: more occupied
binades than the one-CTA kernel has counters for (those rows are redone by the
cluster kernel), -0 and +0 both present at the maximum, many ties at the top-p
cutoff with the token's rank among them deciding its probability, non-finite
and all -inf rows, and rows that do not start on a 16-byte boundary.
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
ROW_SLOTS = 64   # binades the one-CTA kernel holds per row


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv_build.build()
    sv.load()


def _bits_to_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


def _binades(row_bits: np.ndarray) -> int:
    """Occupied binades (sign + exponent) of a row of bf16 patterns, with -0 and +0 as one."""
    b = row_bits.astype(np.uint32)
    b = np.where((b & 0x7FFF) == 0, 0, b)
    key = np.where(b & 0x8000, ~b & 0xFFFF, b | 0x8000)
    return len(np.unique(key >> 7))


def _check_rows(logits: torch.Tensor, T, tk, tp, toks):
    """build_target_probs on [rows, V] bf16 logits, one request per row, against the oracle."""
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


def test_rows_beyond_the_slot_capacity_match_the_oracle():
    # values spread over ~150 binades of both signs: the one-CTA kernel hands
    # these rows on; rows of ordinary logits in the same launch stay on it
    rng = np.random.default_rng(1)
    V, rows = 20_000, 6
    bits = np.empty((rows, V), np.uint16)
    for r in range(rows):
        if r % 2 == 0:
            e = rng.integers(-70, 8, V)
            s = rng.choice([-1.0, 1.0], V)
            x = (s * rng.uniform(1.0, 2.0, V) * np.exp2(e)).astype(np.float32)
        else:
            x = rng.normal(0.0, 3.0, V).astype(np.float32)
        bits[r] = (torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    spread = [_binades(bits[r]) for r in range(rows)]
    assert all(spread[r] > ROW_SLOTS for r in range(0, rows, 2)), spread
    assert all(spread[r] <= ROW_SLOTS for r in range(1, rows, 2)), spread
    logits = _bits_to_bf16(bits)
    n = _check_rows(logits, [1.0, 0.7, 1.3, 1.0, 0.5, 1.0], [0, 0, 0, 100, 0, 0], [0.9, 0.95, 0.999, 1.0, 0.5, 1.0],
                    rng.integers(0, V, rows))
    assert n >= rows - 1


def test_slot_capacity_boundary():
    # exactly ROW_SLOTS and ROW_SLOTS + 1 occupied binades
    rng = np.random.default_rng(2)
    V = 9_000
    rows = []
    for nb in (ROW_SLOTS - 1, ROW_SLOTS, ROW_SLOTS + 1):
        exps = np.arange(-nb + 4, 4)              # nb positive binades
        e = exps[rng.integers(0, nb, V)]
        e[:nb] = exps                             # every one occupied
        x = (rng.uniform(1.0, 2.0, V) * np.exp2(e)).astype(np.float32)
        b = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert _binades(b) == nb
        rows.append(b)
    logits = _bits_to_bf16(np.stack(rows))
    assert _check_rows(logits, [1.0, 1.0, 1.0], [0, 0, 0], [0.9, 0.9, 0.9], rng.integers(0, V, 3)) == 3


def test_signed_zeros_at_the_maximum():
    V = 1000
    neg_inf = 0xFF80
    bits = np.full((4, V), neg_inf, np.uint16)
    bits[0, [17, 400, 800]] = [0x8000, 0x0000, 0x8000]   # -0 first: the argmax is 17
    bits[1, [5, 6, 900]] = [0x0000, 0x8000, 0x0000]      # +0 first
    bits[2, [300, 301]] = [0x8000, 0x8000]               # only -0
    bits[3, :] = 0x8000                                  # all -0, top-p cuts inside the tie group
    bits[3, ::2] = 0x0000
    logits = _bits_to_bf16(bits)
    toks = [800, 900, 301, 700]
    n = _check_rows(logits, [1.0, 0.5, 1.0, 1.0], [0, 0, 0, 0], [0.9, 1.0, 0.6, 0.3005], toks)
    assert n >= 3


def test_ties_at_the_cutoff_and_the_token_rank():
    # few distinct values: the top-p cutoff falls inside a large tie group,
    # and the token is taken before, at and after the kept part of it
    rng = np.random.default_rng(3)
    V, rows = 50_000, 12
    x = rng.choice(np.array([0.0, 0.5, 1.0, 1.5], np.float32), (rows, V), p=[0.4, 0.3, 0.2, 0.1])
    logits = torch.from_numpy(x).to(torch.bfloat16)
    host = np_logits(logits)
    vals = logits.float().numpy()
    T = [1.0] * rows
    tp = list(np.linspace(0.15, 0.95, rows))
    toks = []
    for i in range(rows):
        od, _ = oracle.row_transform(host[i], 1.0, 0, float(tp[i]))
        cut = np.flatnonzero(vals[i] == od["cutoff_logit"])
        toks.append(int(cut[[0, len(cut) // 2, -1][i % 3]]) if od["cutoff_ties"] < len(cut) else int(cut[0]))
    assert _check_rows(logits, T, [0] * rows, tp, toks) >= rows - 1


def test_nonfinite_and_empty_rows():
    rng = np.random.default_rng(4)
    V = 4_000
    x = rng.normal(0, 3, (5, V)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    bits[0, 123] = 0xFFC1          # NaN with the sign bit set
    bits[1, 77] = 0x7FC0           # NaN
    bits[2, 3999] = 0x7F80         # +inf
    bits[3, :] = 0xFF80            # all -inf
    bits[4, 10] = 0xFF80           # one -inf among finite values: fine
    logits = _bits_to_bf16(bits)
    _check_rows(logits, [1.0] * 5, [0] * 5, [0.9] * 5, [0, 1, 2, 3, 10])
    d = sv.desc_fields(sv.build_target_probs(logits.to(DEV), torch.ones(5, device=DEV),
                                             top_p=torch.full((5,), 0.9, device=DEV))[0])
    assert (d["status"][:3] == sv.ROW_NONFINITE).all() and d["status"][3] == sv.ROW_EMPTY and d["status"][4] == 0


@pytest.mark.parametrize("V", [4099, 151_937, 9])
def test_unaligned_rows(V):
    # consecutive rows of an odd vocabulary start at every 2-byte offset
    w = workloads.random_case(5, 4, 3, V, device=DEV, mode="full")
    logits = w.target.reshape(-1, V)
    rows = logits.shape[0]
    rng = np.random.default_rng(V)
    T = rng.choice([0.6, 1.0, 1.4], rows).tolist()
    tp = rng.choice([0.5, 0.9, 1.0], rows).tolist()
    assert _check_rows(logits.cpu(), T, [0] * rows, tp, rng.integers(0, V, rows)) >= rows - 1


def test_verify_with_handed_on_rows_in_the_batch():
    # a medium-shaped batch where some requests' rows need the cluster kernel
    w = workloads.make("medium", device=DEV, scale=dict(n=8, V=30_000))
    rng = np.random.default_rng(6)
    t = w.target.clone()
    for r in (1, 5):
        e = rng.integers(-70, 6, (w.K + 1, w.V))
        x = (rng.uniform(1.0, 2.0, e.shape) * np.exp2(e) * rng.choice([-1.0, 1.0], e.shape)).astype(np.float32)
        t[r] = torch.from_numpy(x).to(t.dtype).to(DEV)
    w2 = workloads.Workload(w.name, "chain", w.n, w.K, w.V, w.dtype, t.contiguous(), w.draft, w.draft_tokens,
                            w.temperature, w.top_k, w.top_p)
    g = sv.verify_chain(w2.target, w2.draft, w2.draft_tokens, w2.temperature, w2.top_k, w2.top_p, seed=4)
    torch.cuda.synchronize()
    o = oracle.verify_chain(np_logits(w2.target), np_logits(w2.draft), w2.draft_tokens.cpu().numpy(),
                            w2.temperature.cpu().numpy(), w2.top_k.cpu().numpy(), w2.top_p.cpu().numpy(), seed=4)
    compare_verify(o, g, w2.draft_tokens.cpu().numpy(), np.full(w2.n, w2.K), w2.V)


def test_rows_past_a_known_rejection_keep_their_status():
    # Every request rejects at position 0 (its first draft token has target
    # logit -inf, so p = 0), and the rows outnumber one wave of CTAs: rows of
    # later positions taken after that test is decided get the status scan
    # only.  Non-finite and all -inf rows planted there must still fail
    # their requests exactly as the oracle says, and the others must draw
    # their token from the residual of the full rows at position 0.
    rng = np.random.default_rng(7)
    n, K, V = 384, 6, 4_096
    x = rng.normal(0, 3, (n, K + 1, V)).astype(np.float32)
    y = (0.8 * x[:, :K] + 0.6 * rng.normal(0, 3, (n, K, V))).astype(np.float32)
    toks = rng.integers(0, V, (n, K)).astype(np.int32)
    x[np.arange(n), 0, toks[:, 0]] = -np.inf
    tbits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    dbits = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    planted = {}
    for r in range(0, n, 7):
        j = int(rng.integers(2, K + 1))
        kind = r // 7 % 5
        bits = tbits if kind < 4 or j == K else dbits
        if kind == 0:
            bits[r, j, 5] = 0x7FC0        # NaN
        elif kind == 1:
            bits[r, j, 6] = 0xFFC1        # NaN with the sign bit set
        elif kind == 2:
            bits[r, j, V - 1] = 0x7F80    # +inf
        elif kind == 3:
            bits[r, j, :] = 0xFF80        # all -inf
        else:
            bits[r, j, 9] = 0x7FC0        # NaN in the draft row (the target row where j = K)
        planted[r] = j
    tgt = _bits_to_bf16(tbits).reshape(n, K + 1, V)
    drf = _bits_to_bf16(dbits).reshape(n, K, V)
    T = np.where(np.arange(n) % 3 == 0, 0.7, 1.0).astype(np.float32)
    tp = np.where(np.arange(n) % 2 == 0, 0.9, 1.0).astype(np.float32)
    tk = np.zeros(n, np.int32)
    g = sv.verify_chain(tgt.to(DEV), drf.to(DEV), torch.from_numpy(toks).to(DEV), torch.from_numpy(T).to(DEV),
                        torch.from_numpy(tk).to(DEV), torch.from_numpy(tp).to(DEV), seed=11)
    torch.cuda.synchronize()
    o = oracle.verify_chain(np_logits(tgt), np_logits(drf), toks, T, tk, tp, seed=11)
    assert (o["accept_len"] == 0).all()
    failed = o["num_emitted"] == 0
    assert failed[list(planted)].all() and failed.sum() == len(planted)
    compare_verify(o, g, toks, np.full(n, K), V)


def test_every_row_in_full_when_every_test_accepts():
    # Draft rows equal to the target rows (q = p: every test accepts), more
    # rows than one wave of CTAs: the rows are taken position by position
    # while the early tests are decided, none is ever past a known rejection,
    # and every one needs its full pass.
    rng = np.random.default_rng(8)
    n, K, V = 320, 6, 4_096
    x = rng.normal(0, 3, (n, K + 1, V)).astype(np.float32)
    tgt = torch.from_numpy(x).to(torch.bfloat16)
    drf = tgt[:, :K].contiguous()
    T = np.where(np.arange(n) % 2 == 0, 0.8, 1.0).astype(np.float32)
    tp = np.where(np.arange(n) % 3 == 0, 0.95, 1.0).astype(np.float32)
    tk = np.zeros(n, np.int32)
    # each draft token drawn from its own row's kept set (so q > 0 there)
    toks = np.empty((n, K), np.int32)
    host = np_logits(tgt)
    for r in range(n):
        for j in range(K):
            _, op = oracle.row_transform(host[r, j], float(T[r]), 0, float(tp[r]))
            toks[r, j] = rng.choice(V, p=op / op.sum())
    g = sv.verify_chain(tgt.to(DEV), drf.to(DEV), torch.from_numpy(toks).to(DEV), torch.from_numpy(T).to(DEV),
                        torch.from_numpy(tk).to(DEV), torch.from_numpy(tp).to(DEV), seed=12)
    torch.cuda.synchronize()
    o = oracle.verify_chain(host, np_logits(drf), toks, T, tk, tp, seed=12)
    assert (o["accept_len"] == K).all()
    compare_verify(o, g, toks, np.full(n, K), V)
