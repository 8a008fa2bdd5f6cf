"""Thin Python binding of libsv (include/sv.h): argument marshalling only.

Every step of the verify path runs in the CUDA library; this module passes
tensor data pointers, sizes and the current CUDA stream through ctypes and
allocates the output and workspace tensors with PyTorch.  There is no CPU
fallback: if the library is missing or no GPU is present the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_WORKSPACE, SV_ERR_CUDA, SV_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
# per-position status bits (SV_ROW_* in sv.h)
SV_ROW_NONFINITE, SV_ROW_EMPTY, SV_ROW_BAD_TOKEN, SV_ROW_BAD_PARAM, SV_ROW_BAD_LAYOUT = 1, 2, 4, 8, 16
SV_ROW_Q_ZERO, SV_ROW_RESID_ZERO, SV_ROW_UNSUPPORTED, SV_ROW_TIMEOUT = 32, 64, 128, 256
DTYPE_BF16, DTYPE_F32 = 0, 1
ROW_NONFINITE, ROW_EMPTY, ROW_BAD_TOKEN, ROW_BAD_PARAM, ROW_BAD_LAYOUT = 1, 2, 4, 8, 16
ROW_Q_ZERO, ROW_RESID_ZERO, ROW_UNSUPPORTED, ROW_TIMEOUT = 32, 64, 128, 256
ROW_ERROR_MASK = (ROW_NONFINITE | ROW_EMPTY | ROW_BAD_TOKEN | ROW_BAD_PARAM | ROW_BAD_LAYOUT | ROW_UNSUPPORTED
                  | ROW_TIMEOUT)

EXPORTED = ("sv_workspace_size", "sv_workspace_size_block", "sv_status_string", "sv_plan_budget",
            "sv_build_target_probs", "sv_verify_chain", "sv_verify_ragged", "sv_set_timing_events",
            "sv_set_hist_timing_events", "sv_verify_chain_noalloc", "sv_plan_budget_cost", "sv_verify_stats",
            "sv_verify_block", "sv_estimator_state_bytes", "sv_estimator_init", "sv_estimator_predict",
            "sv_estimator_observe", "sv_shard_record_bytes", "sv_verify_chain_shard_rows",
            "sv_verify_chain_shard_merge", "sv_q_rows_bytes", "sv_estimator_predict_q", "sv_verify_chain_q")


class SVError(RuntimeError):
    pass


class Sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_void_p), ("top_k", ctypes.c_void_p), ("top_p", ctypes.c_void_p),
                ("flags", ctypes.c_int32)]


# sv_sampling_t.flags: every request is greedy or keeps at most 32 tokens by
# top-k, so the full-vocabulary kernels are not launched (a request that
# breaks the promise is refused with ROW_UNSUPPORTED)
SAMPLING_SMALL_TOPK = 1


class RowDesc(ctypes.Structure):
    _fields_ = [("max_logit", ctypes.c_float), ("log_norm", ctypes.c_float), ("cutoff_logit", ctypes.c_float),
                ("cutoff_ties", ctypes.c_int32), ("kept", ctypes.c_int32), ("argmax", ctypes.c_int32),
                ("status", ctypes.c_int32), ("temperature", ctypes.c_float)]


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libsv.so (building it first only if asked)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB_PATH):
        if not build_if_missing:
            raise SVError(f"CUDA library not built: {_build.LIB_PATH} is missing (run build())")
        _build.build()
    L = ctypes.CDLL(_build.LIB_PATH)
    P, I, I64, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    L.sv_workspace_size.argtypes = [I, I, I]
    L.sv_workspace_size.restype = SZ
    L.sv_workspace_size_block.argtypes = [I, I, I]
    L.sv_workspace_size_block.restype = SZ
    L.sv_status_string.argtypes = [I]
    L.sv_status_string.restype = ctypes.c_char_p
    L.sv_plan_budget.argtypes = [P, I, P, I, I, I, I, P, P, P, P, P, SZ, P]
    L.sv_plan_budget.restype = I
    L.sv_build_target_probs.argtypes = [P, I, I64, I, I, P, I, Sampling, P, P, P, P, P, SZ, P]
    L.sv_build_target_probs.restype = I
    L.sv_verify_chain.argtypes = [P, P, I, I, I, I, P, P, Sampling, U64, P, P, P, P, P, SZ, P]
    L.sv_verify_chain.restype = I
    L.sv_verify_block.argtypes = [P, P, I, I, I, I, P, P, Sampling, U64, P, P, P, P, P, SZ, P]
    L.sv_verify_block.restype = I
    L.sv_verify_ragged.argtypes = [P, P, I, I, I, I, I, P, P, P, Sampling, U64, P, P, P, P, P, SZ, P]
    L.sv_verify_ragged.restype = I
    L.sv_verify_chain_noalloc.argtypes = [P, P, I, I, I, I, P, P, Sampling, U64, P, P, P, P, P]
    L.sv_verify_chain_noalloc.restype = I
    L.sv_plan_budget_cost.argtypes = [P, I, P, I, I, P, P, I, ctypes.c_float, P, P, I, I, P, P, P, P, P, P, P, SZ, P]
    L.sv_plan_budget_cost.restype = I
    L.sv_verify_stats.argtypes = [P, P, P, P, I, I, P, P]
    L.sv_verify_stats.restype = I
    L.sv_estimator_state_bytes.argtypes = [I]
    L.sv_estimator_state_bytes.restype = SZ
    L.sv_estimator_init.argtypes = [P, I, P]
    L.sv_estimator_init.restype = I
    L.sv_estimator_predict.argtypes = [P, I, I, I, I, Sampling, P, P, P, P, SZ, P]
    L.sv_estimator_predict.restype = I
    L.sv_estimator_observe.argtypes = [P, P, P, P, P, I, I, I, P]
    L.sv_estimator_observe.restype = I
    L.sv_q_rows_bytes.argtypes = [I, I]
    L.sv_q_rows_bytes.restype = SZ
    L.sv_estimator_predict_q.argtypes = [P, I, I, I, I, Sampling, P, P, P, P, P, P, SZ, P]
    L.sv_estimator_predict_q.restype = I
    L.sv_verify_chain_q.argtypes = [P, P, I, I, I, I, P, P, Sampling, U64, P, P, P, P, P, P, SZ, P]
    L.sv_verify_chain_q.restype = I
    L.sv_shard_record_bytes.argtypes = []
    L.sv_shard_record_bytes.restype = SZ
    L.sv_verify_chain_shard_rows.argtypes = [P, P, I, I, I, I, I, I, P, P, Sampling, P, P, SZ, P]
    L.sv_verify_chain_shard_rows.restype = I
    L.sv_verify_chain_shard_merge.argtypes = [P, I, I, I, I, P, P, Sampling, U64, P, P, P, P, P, SZ, P]
    L.sv_verify_chain_shard_merge.restype = I
    L.sv_set_timing_events.argtypes = [P, P]
    L.sv_set_timing_events.restype = I
    L.sv_set_hist_timing_events.argtypes = [P, P]
    L.sv_set_hist_timing_events.restype = I
    _lib = L
    return L


def _check(rc: int):
    if rc != SV_OK:
        raise SVError(load().sv_status_string(rc).decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise SVError(f"logits must be bf16 or fp32, got {t.dtype}")


def _dev(t: torch.Tensor, dtype=None) -> torch.Tensor:
    if not t.is_cuda:
        raise SVError("tensors must live on the GPU (the library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise SVError(f"expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise SVError("tensors must be contiguous")
    return t


def _sampling(temperature, top_k, top_p, small_topk: bool = False) -> Sampling:
    return Sampling(temperature.data_ptr(), None if top_k is None else top_k.data_ptr(),
                    None if top_p is None else top_p.data_ptr(), SAMPLING_SMALL_TOPK if small_topk else 0)


def set_timing_events(start: Optional["torch.cuda.Event"], stop: Optional["torch.cuda.Event"]):
    """Have later calls record these events around the one-pass row kernel."""
    if start is None or stop is None:
        load().sv_set_timing_events(None, None)
    else:
        load().sv_set_timing_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event))


def set_hist_timing_events(start: Optional["torch.cuda.Event"], stop: Optional["torch.cuda.Event"]):
    """Have later bf16 calls record these events around the exact-histogram row kernels."""
    if start is None or stop is None:
        load().sv_set_hist_timing_events(None, None)
    else:
        load().sv_set_hist_timing_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event))


def workspace_size(n_req: int, k_max: int, vocab: int) -> int:
    size = load().sv_workspace_size(n_req, k_max, vocab)
    if size == 0:
        raise SVError("sizes beyond what the library supports")
    return size


def workspace_size_block(n_req: int, k_max: int, vocab: int) -> int:
    size = load().sv_workspace_size_block(n_req, k_max, vocab)
    if size == 0:
        raise SVError("sizes beyond what the library supports")
    return size


class Workspace:
    """A reusable device workspace (grows on demand, 256-byte aligned)."""

    def __init__(self, device="cuda"):
        self.device = torch.device(device)
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.buf.data_ptr()) % 256
        return self.buf[off:off + nbytes]


def _ws(ws: Optional[Workspace], device, nbytes) -> torch.Tensor:
    if ws is None:
        ws = Workspace(device)
    return ws.get(nbytes)


@dataclass
class VerifyOut:
    accept_len: torch.Tensor     # [n] int32
    out_tokens: torch.Tensor     # [n, K+1] int32, -1 filled
    num_emitted: torch.Tensor    # [n] int32
    row_status: torch.Tensor     # [n, K+1] int32


def plan_budget(conf: torch.Tensor, budget: int, bucket: int, draft_len: Optional[torch.Tensor] = None,
                ws: Optional[Workspace] = None):
    """sv_plan_budget: (verify_lens [n], qo_indptr [n+1], total [1], status [1]) on the device."""
    conf = _dev(conf, torch.float32)
    n, K = conf.shape
    dev = conf.device
    vl = torch.empty(n, dtype=torch.int32, device=dev)
    qo = torch.empty(n + 1, dtype=torch.int32, device=dev)
    tot = torch.empty(1, dtype=torch.int32, device=dev)
    st = torch.empty(1, dtype=torch.int32, device=dev)
    w = _ws(ws, dev, workspace_size(n, K, 0))
    _check(load().sv_plan_budget(_ptr(conf), K, _ptr(draft_len), n, K, budget, bucket, _ptr(vl), _ptr(qo),
                                 _ptr(tot), _ptr(st), _ptr(w), w.numel(), _stream(dev)))
    return vl, qo, tot, st


def plan_budget_cost(conf: torch.Tensor, cost_tokens: Optional[torch.Tensor], cost_ms: Optional[torch.Tensor],
                     bucket: int, fixed_overhead_ms: float = 0.0, batch_sizes: Optional[torch.Tensor] = None,
                     batch_overhead_ms: Optional[torch.Tensor] = None, draft_len: Optional[torch.Tensor] = None,
                     ws: Optional[Workspace] = None):
    """sv_plan_budget_cost: (budget [1], budget_status [1], verify_lens [n], qo_indptr [n+1], total [1],
    status [1]) on the device; the table arrays are device tensors (int32 tokens, fp32 ms) or None."""
    conf = _dev(conf, torch.float32)
    n, K = conf.shape
    dev = conf.device
    ct = None if cost_tokens is None else _dev(cost_tokens, torch.int32)
    cm = None if cost_ms is None else _dev(cost_ms, torch.float32)
    bs = None if batch_sizes is None else _dev(batch_sizes, torch.int32)
    bo = None if batch_overhead_ms is None else _dev(batch_overhead_ms, torch.float32)
    n_cost = 0 if ct is None else ct.numel()
    n_batch = 0 if bs is None else bs.numel()
    if (cm is None and n_cost) or (cm is not None and cm.numel() != n_cost):
        raise SVError("cost_tokens and cost_ms differ in length")
    if (bo is None and n_batch) or (bo is not None and bo.numel() != n_batch):
        raise SVError("batch_sizes and batch_overhead_ms differ in length")
    b = torch.empty(1, dtype=torch.int32, device=dev)
    bst = torch.empty(1, dtype=torch.int32, device=dev)
    vl = torch.empty(n, dtype=torch.int32, device=dev)
    qo = torch.empty(n + 1, dtype=torch.int32, device=dev)
    tot = torch.empty(1, dtype=torch.int32, device=dev)
    st = torch.empty(1, dtype=torch.int32, device=dev)
    w = _ws(ws, dev, workspace_size(n, K, 0))
    _check(load().sv_plan_budget_cost(_ptr(conf), K, _ptr(draft_len), n, K, _ptr(ct), _ptr(cm), n_cost,
                                      float(fixed_overhead_ms), _ptr(bs), _ptr(bo), n_batch, bucket, _ptr(b),
                                      _ptr(bst), _ptr(vl), _ptr(qo), _ptr(tot), _ptr(st), _ptr(w), w.numel(),
                                      _stream(dev)))
    return b, bst, vl, qo, tot, st


def verify_stats(accept_len: torch.Tensor, num_emitted: torch.Tensor, verify_lens: Optional[torch.Tensor], K: int,
                 draft_len: Optional[torch.Tensor] = None) -> torch.Tensor:
    """sv_verify_stats: int64 [4] on the device (tokens emitted, tokens submitted, requests trimmed,
    trimmed requests that accepted their whole window)."""
    accept_len = _dev(accept_len, torch.int32)
    num_emitted = _dev(num_emitted, torch.int32)
    dev = accept_len.device
    out = torch.empty(4, dtype=torch.int64, device=dev)
    _check(load().sv_verify_stats(_ptr(accept_len), _ptr(num_emitted), _ptr(verify_lens), _ptr(draft_len),
                                  accept_len.numel(), K, _ptr(out), _stream(dev)))
    return out


class Estimator:
    """The online acceptance estimator: a device state and its three calls."""

    def __init__(self, K: int, device="cuda"):
        self.K = K
        self.state = torch.empty(4 * K + 5, dtype=torch.float64, device=device)
        _check(load().sv_estimator_init(_ptr(self.state), K, _stream(self.state.device)))
        self.ws = Workspace(self.state.device)

    @property
    def slope(self) -> torch.Tensor:
        return self.state[0]

    @property
    def bias(self) -> torch.Tensor:
        return self.state[1:1 + self.K]

    def predict(self, draft: torch.Tensor, temperature: torch.Tensor, top_k: Optional[torch.Tensor] = None,
                top_p: Optional[torch.Tensor] = None):
        """(x [n, K], p [n, K]) fp32 on the device for draft logits [n, K, V]."""
        draft = _dev(draft)
        n, K, V = draft.shape
        assert K == self.K
        dev = draft.device
        x = torch.empty((n, K), dtype=torch.float32, device=dev)
        p = torch.empty((n, K), dtype=torch.float32, device=dev)
        w = _ws(self.ws, dev, workspace_size(n * K, 0, V))
        _check(load().sv_estimator_predict(_ptr(draft), _dtype_code(draft), n, K, V,
                                           _sampling(temperature, top_k, top_p), _ptr(self.state), _ptr(x), _ptr(p),
                                           _ptr(w), w.numel(), _stream(dev)))
        return x, p

    def predict_q(self, draft: torch.Tensor, draft_tokens: torch.Tensor, temperature: torch.Tensor,
                  top_k: Optional[torch.Tensor] = None, top_p: Optional[torch.Tensor] = None,
                  q_rows: Optional[torch.Tensor] = None):
        """sv_estimator_predict_q: (x, p, q_rows) -- q_rows (uint8 on the device) carries every draft
        row's distribution for verify_chain_q over the same batch."""
        draft = _dev(draft)
        n, K, V = draft.shape
        assert K == self.K
        dev = draft.device
        x = torch.empty((n, K), dtype=torch.float32, device=dev)
        p = torch.empty((n, K), dtype=torch.float32, device=dev)
        nbytes = int(load().sv_q_rows_bytes(n, K))
        if q_rows is None:
            q_rows = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        assert q_rows.numel() >= nbytes and q_rows.is_cuda
        w = _ws(self.ws, dev, workspace_size(n * K, 0, V))
        _check(load().sv_estimator_predict_q(_ptr(draft), _dtype_code(draft), n, K, V,
                                             _sampling(temperature, top_k, top_p), _ptr(self.state),
                                             _ptr(_dev(draft_tokens, torch.int32)), _ptr(x), _ptr(p), _ptr(q_rows),
                                             _ptr(w), w.numel(), _stream(dev)))
        return x, p, q_rows

    def observe(self, x: torch.Tensor, accept_len: torch.Tensor, num_emitted: torch.Tensor,
                verify_lens: Optional[torch.Tensor] = None, refit_every: int = 100):
        x = _dev(x, torch.float32)
        n = x.shape[0]
        _check(load().sv_estimator_observe(_ptr(self.state), _ptr(x), _ptr(_dev(accept_len, torch.int32)),
                                           _ptr(_dev(num_emitted, torch.int32)), _ptr(verify_lens), n, self.K,
                                           refit_every, _stream(x.device)))


def build_target_probs(logits: torch.Tensor, temperature: torch.Tensor, top_k: Optional[torch.Tensor] = None,
                       top_p: Optional[torch.Tensor] = None, row_to_req: Optional[torch.Tensor] = None,
                       tokens: Optional[torch.Tensor] = None, dense: bool = False,
                       ws: Optional[Workspace] = None, small_topk: bool = False):
    """sv_build_target_probs over [rows, vocab] logits (small_topk: the
    SAMPLING_SMALL_TOPK promise).

    Returns (desc [rows, 8] int32 view of sv_row_desc_t, prob_of_token [rows]
    or None, dense [rows, vocab] or None)."""
    logits = _dev(logits)
    rows, V = logits.shape
    dev = logits.device
    n_req = temperature.numel()
    desc = torch.empty((rows, 8), dtype=torch.int32, device=dev)
    ptok = torch.empty(rows, dtype=torch.float32, device=dev) if tokens is not None else None
    dn = torch.empty((rows, V), dtype=torch.float32, device=dev) if dense else None
    w = _ws(ws, dev, workspace_size(rows, 0, V))
    _check(load().sv_build_target_probs(_ptr(logits), _dtype_code(logits), V, rows, V, _ptr(row_to_req), n_req,
                                        _sampling(temperature, top_k, top_p, small_topk), _ptr(tokens), _ptr(ptok),
                                        _ptr(desc), _ptr(dn), _ptr(w), w.numel(), _stream(dev)))
    return desc, ptok, dn


def desc_fields(desc: torch.Tensor) -> dict:
    """Split the [rows, 8] int32 descriptor view into named host arrays."""
    d = desc.cpu()
    f = d.view(torch.float32)
    return dict(max_logit=f[:, 0].numpy(), log_norm=f[:, 1].numpy(), cutoff_logit=f[:, 2].numpy(),
                cutoff_ties=d[:, 3].numpy(), kept=d[:, 4].numpy(), argmax=d[:, 5].numpy(),
                status=d[:, 6].numpy(), temperature=f[:, 7].numpy())


def _outs(n, K, dev):
    return VerifyOut(torch.empty(n, dtype=torch.int32, device=dev),
                     torch.empty((n, K + 1), dtype=torch.int32, device=dev),
                     torch.empty(n, dtype=torch.int32, device=dev),
                     torch.empty((n, K + 1), dtype=torch.int32, device=dev))


def verify_chain(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                 temperature: torch.Tensor, top_k: Optional[torch.Tensor] = None,
                 top_p: Optional[torch.Tensor] = None, verify_len: Optional[torch.Tensor] = None, seed: int = 0,
                 ws: Optional[Workspace] = None, out: Optional[VerifyOut] = None, block: bool = False,
                 small_topk: bool = False) -> VerifyOut:
    """sv_verify_chain (or, with block=True, sv_verify_block): target [n, K+1, V], draft [n, K, V]
    (or None if all greedy); small_topk: the SAMPLING_SMALL_TOPK promise."""
    target = _dev(target)
    n, k1, V = target.shape
    K = k1 - 1
    dev = target.device
    if draft is not None:
        _dev(draft, target.dtype)
        assert draft.shape == (n, K, V)
    o = out or _outs(n, K, dev)
    w = _ws(ws, dev, workspace_size_block(n, K, V) if block else workspace_size(n, K, V))
    fn = load().sv_verify_block if block else load().sv_verify_chain
    _check(fn(_ptr(target), _ptr(draft), _dtype_code(target), n, K, V, _ptr(draft_tokens), _ptr(verify_len),
              _sampling(temperature, top_k, top_p, small_topk), seed, _ptr(o.accept_len), _ptr(o.out_tokens),
              _ptr(o.num_emitted), _ptr(o.row_status), _ptr(w), w.numel(), _stream(dev)))
    return o


def verify_chain_noalloc(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                         temperature: torch.Tensor, top_k: Optional[torch.Tensor] = None,
                         top_p: Optional[torch.Tensor] = None, verify_len: Optional[torch.Tensor] = None,
                         seed: int = 0, out: Optional[VerifyOut] = None, small_topk: bool = False) -> VerifyOut:
    """sv_verify_chain_noalloc: sv_verify_chain with the library's static scratch
    (no workspace).  The outputs are allocated here unless `out` is given."""
    target = _dev(target)
    n, k1, V = target.shape
    K = k1 - 1
    dev = target.device
    if draft is not None:
        _dev(draft, target.dtype)
        assert draft.shape == (n, K, V)
    o = out or _outs(n, K, dev)
    _check(load().sv_verify_chain_noalloc(_ptr(target), _ptr(draft), _dtype_code(target), n, K, V,
                                          _ptr(draft_tokens), _ptr(verify_len),
                                          _sampling(temperature, top_k, top_p, small_topk),
                                          seed, _ptr(o.accept_len), _ptr(o.out_tokens), _ptr(o.num_emitted),
                                          _ptr(o.row_status), _stream(dev)))
    return o


def verify_ragged(target: torch.Tensor, draft: Optional[torch.Tensor], qo_indptr: torch.Tensor,
                  verify_lens: torch.Tensor, draft_tokens: torch.Tensor, temperature: torch.Tensor,
                  top_k: Optional[torch.Tensor] = None, top_p: Optional[torch.Tensor] = None, seed: int = 0,
                  ws: Optional[Workspace] = None, out: Optional[VerifyOut] = None,
                  small_topk: bool = False) -> VerifyOut:
    """sv_verify_ragged: packed target [bucket, V], draft [n, K_max, V] block layout; small_topk: the
    SAMPLING_SMALL_TOPK promise."""
    target = _dev(target)
    bucket, V = target.shape
    n, K = draft_tokens.shape
    dev = target.device
    if draft is not None:
        _dev(draft, target.dtype)
        assert draft.shape == (n, K, V)
    o = out or _outs(n, K, dev)
    w = _ws(ws, dev, workspace_size(n, K, V))
    _check(load().sv_verify_ragged(_ptr(target), _ptr(draft), _dtype_code(target), n, K, V, bucket,
                                   _ptr(qo_indptr), _ptr(verify_lens), _ptr(draft_tokens),
                                   _sampling(temperature, top_k, top_p, small_topk), seed, _ptr(o.accept_len),
                                   _ptr(o.out_tokens), _ptr(o.num_emitted), _ptr(o.row_status), _ptr(w),
                                   w.numel(), _stream(dev)))
    return o


def shard_record_bytes() -> int:
    return int(load().sv_shard_record_bytes())


def verify_chain_shard_rows(target_shard: torch.Tensor, draft_shard: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                            temperature: torch.Tensor, top_k: Optional[torch.Tensor], top_p: Optional[torch.Tensor],
                            v0: int, vocab: int, verify_len: Optional[torch.Tensor] = None,
                            ws: Optional[Workspace] = None, records: Optional[torch.Tensor] = None) -> torch.Tensor:
    """sv_verify_chain_shard_rows: one vocabulary shard's records (uint8 [n * (2K+1) * record bytes]).
    target_shard [n, K+1, Vs] holds columns v0 .. v0 + Vs - 1 of the target rows, draft_shard [n, K, Vs]
    the same of the draft rows (None if all greedy)."""
    target_shard = _dev(target_shard)
    n, k1, Vs = target_shard.shape
    K = k1 - 1
    dev = target_shard.device
    if draft_shard is not None:
        _dev(draft_shard, target_shard.dtype)
        assert draft_shard.shape == (n, K, Vs)
    nbytes = n * (2 * K + 1) * shard_record_bytes()
    if records is None:
        records = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    assert records.numel() >= nbytes and records.is_cuda
    w = _ws(ws, dev, workspace_size(n, K, Vs))
    _check(load().sv_verify_chain_shard_rows(_ptr(target_shard), _ptr(draft_shard), _dtype_code(target_shard), n, K,
                                             vocab, v0, v0 + Vs, _ptr(draft_tokens), _ptr(verify_len),
                                             _sampling(temperature, top_k, top_p), _ptr(records), _ptr(w), w.numel(),
                                             _stream(dev)))
    return records


def verify_chain_shard_merge(records: torch.Tensor, n_shards: int, draft_tokens: torch.Tensor,
                             temperature: torch.Tensor, top_k: Optional[torch.Tensor], top_p: Optional[torch.Tensor],
                             vocab: int, verify_len: Optional[torch.Tensor] = None, seed: int = 0,
                             ws: Optional[Workspace] = None, out: Optional[VerifyOut] = None) -> VerifyOut:
    """sv_verify_chain_shard_merge: the step's outputs from every shard's records (device
    [n_shards, n * (2K+1) * record bytes], any shard order)."""
    records = _dev(records)
    n, K = draft_tokens.shape
    dev = records.device
    assert records.numel() >= n_shards * n * (2 * K + 1) * shard_record_bytes()
    o = out or _outs(n, K, dev)
    w = _ws(ws, dev, workspace_size(n, K, 1))
    _check(load().sv_verify_chain_shard_merge(_ptr(records), n_shards, n, K, vocab, _ptr(draft_tokens),
                                              _ptr(verify_len), _sampling(temperature, top_k, top_p), seed,
                                              _ptr(o.accept_len), _ptr(o.out_tokens), _ptr(o.num_emitted),
                                              _ptr(o.row_status), _ptr(w), w.numel(), _stream(dev)))
    return o


def verify_chain_q(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                   temperature: torch.Tensor, top_k: Optional[torch.Tensor], top_p: Optional[torch.Tensor],
                   q_rows: torch.Tensor, verify_len: Optional[torch.Tensor] = None, seed: int = 0,
                   ws: Optional[Workspace] = None, out: Optional[VerifyOut] = None,
                   small_topk: bool = False) -> VerifyOut:
    """sv_verify_chain_q: sv_verify_chain with the draft rows' distributions from Estimator.predict_q."""
    target = _dev(target)
    n, k1, V = target.shape
    K = k1 - 1
    dev = target.device
    if draft is not None:
        _dev(draft, target.dtype)
        assert draft.shape == (n, K, V)
    o = out or _outs(n, K, dev)
    w = _ws(ws, dev, workspace_size(n, K, V))
    _check(load().sv_verify_chain_q(_ptr(target), _ptr(draft), _dtype_code(target), n, K, V, _ptr(draft_tokens),
                                    _ptr(verify_len), _sampling(temperature, top_k, top_p, small_topk), seed,
                                    _ptr(_dev(q_rows)),
                                    _ptr(o.accept_len), _ptr(o.out_tokens), _ptr(o.num_emitted), _ptr(o.row_status),
                                    _ptr(w), w.numel(), _stream(dev)))
    return o
