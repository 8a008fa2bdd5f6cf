"""CPU oracle of the speculative-decoding verify step (test infrastructure).

This package is the checker the CUDA library is compared against: a plain,
single-threaded, double-precision C implementation of the definition
(``oracle.c``), loaded here through ctypes.  Only the tests, the package smoke
check and the benchmark's CPU-baseline leg use it; the product path never
imports it, and it shares no code with the CUDA sources.

The numpy wrappers below only marshal arguments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

# Status bits (same values as the library's public ones: they are an
# interface, restated here rather than shared).
NONFINITE, EMPTY, BAD_TOKEN, BAD_PARAM, BAD_LAYOUT, Q_ZERO, RESID_ZERO = 1, 2, 4, 8, 16, 32, 64
ERROR_MASK = NONFINITE | EMPTY | BAD_TOKEN | BAD_PARAM | BAD_LAYOUT
FLAG_RATIO, FLAG_CUTOFF, FLAG_INVCDF, FLAG_RESID = 1, 2, 4, 8
# Per-position bits of the alternative outcomes (ORC_ALT_* in oracle.c).
ALT_ACCEPT, ALT_AMBIG, ALT_DRAW_NEAR, ALT_DRAW_ROW = 1, 2, 4, 8


def build(force: bool = False, plant: int = 0, out_dir: str | None = None) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, no fast-math).

    plant != 0 builds a library with one deliberate mistake (see ORC_PLANT in
    oracle.c) into out_dir, for the tests that show the pins catch it."""
    path = _LIB_PATH if plant == 0 else os.path.join(out_dir, f"liboracle_plant{plant}.so")
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               f"-DORC_PLANT={plant}", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, path)
    return path


_lib = None
# ORACLE_LIB: load another build of oracle.c (for instance one compiled with
# -fsanitize=address or -fsanitize=undefined) instead of liboracle.so.
_lib_path = os.environ.get("ORACLE_LIB") or None


class planted:
    """Context manager: route every wrapper below through a library built
    with mistake number `plant` (test use only)."""

    def __init__(self, plant: int, out_dir: str):
        self.path = build(plant=plant, out_dir=out_dir)

    def __enter__(self):
        global _lib, _lib_path
        self._saved = (_lib, _lib_path)
        _lib, _lib_path = None, self.path
        return self

    def __exit__(self, *exc):
        global _lib, _lib_path
        _lib, _lib_path = self._saved


class RowOut(ctypes.Structure):
    _fields_ = [("max_logit", ctypes.c_double), ("log_norm", ctypes.c_double),
                ("cutoff_logit", ctypes.c_double), ("cutoff_ties", ctypes.c_int32),
                ("kept", ctypes.c_int32), ("argmax", ctypes.c_int32), ("status", ctypes.c_int32),
                ("cut_margin", ctypes.c_double), ("z_rest", ctypes.c_double), ("next_index", ctypes.c_int64)]


class AltOut(ctypes.Structure):
    _fields_ = [("dec", ctypes.c_void_p), ("draw", ctypes.c_void_p), ("draw_alt", ctypes.c_void_p),
                ("n_flag", ctypes.c_void_p), ("n_dec", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(_lib_path or build())
        P = ctypes.c_void_p
        _lib.orc_philox4x32_10.argtypes = [P, P, P]
        _lib.orc_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        _lib.orc_uniform.restype = ctypes.c_double
        _lib.orc_row_transform.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_int32,
                                           ctypes.c_float, ctypes.POINTER(RowOut), P]
        _lib.orc_row_transform.restype = ctypes.c_int
        A = ctypes.POINTER(AltOut)
        _lib.orc_verify_chain.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                          P, P, P, P, P, ctypes.c_uint64, ctypes.c_int, P, P, P, P, P, P, P, A]
        _lib.orc_verify_block.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                          P, P, P, P, P, ctypes.c_uint64, ctypes.c_int, P, P, P, P, P, P, P, A]
        _lib.orc_verify_ragged.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                           ctypes.c_int64, P, P, P, P, P, P, ctypes.c_uint64, ctypes.c_int,
                                           P, P, P, P, P, P, P, A]
        _lib.orc_plan_budget.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, P, P, P, P]
        _lib.orc_plan_budget.restype = ctypes.c_int
        _lib.orc_choose_budget.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
                                           ctypes.c_float, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P]
        _lib.orc_choose_budget.restype = ctypes.c_int
        _lib.orc_verify_stats.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, P]
        _lib.orc_est_init.argtypes = [P, ctypes.c_int]
        _lib.orc_est_features.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, P, P, P, P]
        _lib.orc_est_predict.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P]
        _lib.orc_est_observe.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """(contiguous array, dtype code): bf16 arrives as uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, 0
    if a.dtype == np.float32:
        return a, 1
    raise TypeError(f"logits must be float32 or bf16 bits as uint16, got {a.dtype}")


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, req: int, pos: int, draw: int) -> float:
    return lib().orc_uniform(seed, req, pos, draw)


def row_transform(row, T: float, top_k: int = 0, top_p: float = 1.0, want_probs: bool = True):
    """One row's distribution: (RowOut as dict, dense p or None)."""
    row, dt = _logits(row)
    out = RowOut()
    probs = np.zeros(row.shape[-1], dtype=np.float64) if want_probs else None
    lib().orc_row_transform(_ptr(row), dt, row.shape[-1], T, top_k, top_p, ctypes.byref(out), _ptr(probs))
    d = {f: getattr(out, f) for f, _ in RowOut._fields_}
    return d, probs


def _verify_outputs(n, width):
    return dict(accept_len=np.zeros(n, np.int32), out_tokens=np.zeros((n, width), np.int32),
                num_emitted=np.zeros(n, np.int32), pos_status=np.zeros((n, width), np.int32),
                flags=np.zeros(n, np.int32), p_tok=np.zeros((n, width), np.float64),
                q_tok=np.zeros((n, width), np.float64),
                alt_dec=np.zeros((n, width), np.int32), alt_draw=np.zeros((n, width), np.int32),
                alt_tokens=np.zeros((n, width, 2), np.int32), n_flag=np.zeros(n, np.int32),
                n_dec=np.zeros(n, np.int32))


def _alt(o):
    """Pointers of the alternative-outcome arrays of an output dict (kept
    alive by the dict itself)."""
    return ctypes.byref(AltOut(_ptr(o["alt_dec"]), _ptr(o["alt_draw"]), _ptr(o["alt_tokens"]), _ptr(o["n_flag"]),
                               _ptr(o["n_dec"])))


def _support_fn(row_of, T, tk, tp):
    """support(r, j): tokens a draw at position j of request r may emit when
    the distribution it draws from is uncertain (a near top-p cut or a
    near-empty residual): the support of the target row's p plus the token
    its cut leaves out next.  row_of(r, j) gives the row's logits."""
    def support(r, j):
        d, probs = row_transform(row_of(r, j), float(T[r]), 0 if tk is None else int(tk[r]),
                                 1.0 if tp is None else float(tp[r]))
        mask = probs > 0.0
        if d["next_index"] >= 0:
            mask[d["next_index"]] = True
        return mask
    return support


def verify_chain(target, draft, draft_tokens, temperature, top_k=None, top_p=None, verify_len=None, seed=0,
                 first_req=0, block=False):
    """Uniform layout: target [n, K+1, V], draft [n, K, V] (None if all greedy).
    The requests are requests first_req.. of a larger batch (uniform keys).
    block=True runs block verification (joint block acceptance) instead of
    the token-by-token chain."""
    target, dt = _logits(target)
    n, k1, V = target.shape
    K = k1 - 1
    if draft is not None:
        draft, dt2 = _logits(draft)
        assert dt2 == dt and draft.shape == (n, K, V)
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(n, K)
    T = np.ascontiguousarray(temperature, dtype=np.float32)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32)
    tp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32)
    vl = None if verify_len is None else np.ascontiguousarray(verify_len, dtype=np.int32)
    o = _verify_outputs(n, K + 1)
    fn = lib().orc_verify_block if block else lib().orc_verify_chain
    fn(_ptr(target), _ptr(draft), dt, n, K, V, _ptr(tok), _ptr(vl), _ptr(T), _ptr(tk), _ptr(tp), seed, first_req,
       _ptr(o["accept_len"]), _ptr(o["out_tokens"]), _ptr(o["num_emitted"]), _ptr(o["pos_status"]),
       _ptr(o["flags"]), _ptr(o["p_tok"]), _ptr(o["q_tok"]), _alt(o))
    o["block"] = bool(block)
    o["support"] = _support_fn(lambda r, j: target[r, j], T, tk, tp)
    return o


def verify_ragged(target, draft, qo_indptr, verify_lens, draft_tokens, temperature, top_k=None, top_p=None,
                  seed=0, first_req=0):
    """Packed target [bucket, V] by qo_indptr; draft in block layout [n, K_max, V]."""
    target, dt = _logits(target)
    bucket, V = target.shape
    tok = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    n, K = tok.shape
    if draft is not None:
        draft, dt2 = _logits(draft)
        assert dt2 == dt and draft.shape == (n, K, V)
    qo = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    vl = np.ascontiguousarray(verify_lens, dtype=np.int32)
    T = np.ascontiguousarray(temperature, dtype=np.float32)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32)
    tp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32)
    o = _verify_outputs(n, K + 1)
    lib().orc_verify_ragged(_ptr(target), _ptr(draft), dt, n, K, V, bucket, _ptr(qo), _ptr(vl), _ptr(tok),
                            _ptr(T), _ptr(tk), _ptr(tp), seed, first_req, _ptr(o["accept_len"]), _ptr(o["out_tokens"]),
                            _ptr(o["num_emitted"]), _ptr(o["pos_status"]), _ptr(o["flags"]),
                            _ptr(o["p_tok"]), _ptr(o["q_tok"]), _alt(o))
    o["block"] = False
    o["support"] = _support_fn(lambda r, j: target[int(qo[r]) + j], T, tk, tp)
    return o


def plan_budget(conf, budget: int, bucket: int, draft_len=None):
    """Planner: returns (verify_lens [n], qo_indptr [n+1], total, status)."""
    c = np.ascontiguousarray(conf, dtype=np.float32)
    n, K = c.shape
    dl = None if draft_len is None else np.ascontiguousarray(draft_len, dtype=np.int32)
    vl = np.zeros(n, np.int32)
    qo = np.zeros(n + 1, np.int32)
    tot = np.zeros(1, np.int32)
    st = np.zeros(1, np.int32)
    rc = lib().orc_plan_budget(_ptr(c), K, _ptr(dl), n, K, budget, bucket, _ptr(vl), _ptr(qo), _ptr(tot), _ptr(st))
    if rc != 0:
        raise ValueError("invalid planner arguments")
    return vl, qo, int(tot[0]), int(st[0])


def choose_budget(conf, cost_tokens, cost_ms, bucket: int, fixed_overhead_ms: float = 0.0,
                  batch_sizes=None, batch_overhead_ms=None, draft_len=None):
    """Budget from a step-cost table: returns (budget, theta_best, margin, status)."""
    c = np.ascontiguousarray(conf, dtype=np.float32)
    n, K = c.shape
    dl = None if draft_len is None else np.ascontiguousarray(draft_len, dtype=np.int32)
    ct = np.ascontiguousarray(cost_tokens if cost_tokens is not None else [], dtype=np.int32)
    cm = np.ascontiguousarray(cost_ms if cost_ms is not None else [], dtype=np.float32)
    bs = np.ascontiguousarray(batch_sizes if batch_sizes is not None else [], dtype=np.int32)
    bo = np.ascontiguousarray(batch_overhead_ms if batch_overhead_ms is not None else [], dtype=np.float32)
    if len(ct) != len(cm) or len(bs) != len(bo):
        raise ValueError("table arrays differ in length")
    b = np.zeros(1, np.int32)
    th = np.zeros(1, np.float64)
    mg = np.zeros(1, np.float64)
    st = np.zeros(1, np.int32)
    rc = lib().orc_choose_budget(_ptr(c), K, _ptr(dl), n, K, _ptr(ct), _ptr(cm), len(ct), fixed_overhead_ms,
                                 _ptr(bs), _ptr(bo), len(bs), bucket, _ptr(b), _ptr(th), _ptr(mg), _ptr(st))
    if rc != 0:
        raise ValueError("invalid budget arguments")
    return int(b[0]), float(th[0]), float(mg[0]), int(st[0])


def verify_stats(accept_len, num_emitted, verify_lens, K: int, draft_len=None):
    """(tokens emitted, tokens submitted, requests trimmed, trimmed requests that accepted their whole window)."""
    al = np.ascontiguousarray(accept_len, dtype=np.int32)
    ne = np.ascontiguousarray(num_emitted, dtype=np.int32)
    vl = None if verify_lens is None else np.ascontiguousarray(verify_lens, dtype=np.int32)
    dl = None if draft_len is None else np.ascontiguousarray(draft_len, dtype=np.int32)
    out = np.zeros(4, np.int64)
    lib().orc_verify_stats(_ptr(al), _ptr(ne), _ptr(vl), _ptr(dl), len(al), K, _ptr(out))
    return tuple(int(x) for x in out)


class Estimator:
    """The oracle's online acceptance estimator (state as the C side lays it out)."""

    def __init__(self, K: int):
        self.K = K
        self.state = np.zeros(4 * K + 5, np.float64)
        lib().orc_est_init(_ptr(self.state), K)

    @property
    def slope(self) -> float:
        return float(self.state[0])

    @property
    def bias(self) -> np.ndarray:
        return self.state[1:1 + self.K].copy()

    def predict(self, x) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        n = x.shape[0]
        p = np.zeros((n, self.K), np.float64)
        lib().orc_est_predict(_ptr(self.state), _ptr(x), n, self.K, _ptr(p))
        return p

    def observe(self, x, accept_len, num_emitted, verify_lens=None, refit_every: int = 100):
        x = np.ascontiguousarray(x, dtype=np.float64)
        al = np.ascontiguousarray(accept_len, dtype=np.int32)
        ne = np.ascontiguousarray(num_emitted, dtype=np.int32)
        vl = None if verify_lens is None else np.ascontiguousarray(verify_lens, dtype=np.int32)
        lib().orc_est_observe(_ptr(self.state), _ptr(x), _ptr(al), _ptr(ne), _ptr(vl), len(al), self.K, refit_every)


def est_features(draft, temperature, top_k=None, top_p=None) -> np.ndarray:
    """x [n, K] = clamp(logit(q_max), +-40) of every draft row (T = 1 for greedy requests)."""
    draft, dt = _logits(draft)
    n, K, V = draft.shape
    T = np.ascontiguousarray(temperature, dtype=np.float32)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32)
    tp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32)
    x = np.zeros((n, K), np.float64)
    lib().orc_est_features(_ptr(draft), dt, n, K, V, _ptr(T), _ptr(tk), _ptr(tp), _ptr(x))
    return x
