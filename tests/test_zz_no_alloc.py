"""sv_verify_chain_noalloc (static scratch, no workspace) against sv_verify_chain.

Kept in a file of its own that pytest collects last: the entry point's first
call on a device looks up its static scratch, and this must work both in a
fresh process and after every other test has run.
"""
import ctypes

import pytest
import torch

from speculative_decoding_verification_rows_gb300 import build as sv_build
from speculative_decoding_verification_rows_gb300 import sv, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv_build.build()
    sv.load()


def _same(a: sv.VerifyOut, b: sv.VerifyOut):
    for f in ("accept_len", "out_tokens", "num_emitted", "row_status"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    # call 1: bf16 top-p rows (histogram and resample kernels); call 2: the
    # benchmark's top-k rows.  The second call must not see the first's leftovers.
    cases = [(workloads.make("medium", device=DEV, scale=dict(n=4, V=30000)), 11),
             (workloads.make("large", device=DEV, scale=dict(n=16)), 12)]
    for w, seed in cases:
        got = sv.verify_chain_noalloc(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=seed)
        ref = sv.verify_chain(w.target, w.draft, w.draft_tokens, w.temperature, w.top_k, w.top_p, seed=seed)
        torch.cuda.synchronize()
        _same(got, ref)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    lib = sv.load()
    assert lib.sv_workspace_size(4096, 7, 248_320) > (32 << 20)
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check comes first
    rc = lib.sv_verify_chain_noalloc(fake, fake, 0, 4096, 7, 248_320, fake, None,
                                     sv.Sampling(0x1000, None, None), 0, fake, fake, fake, None, None)
    assert rc == sv.SV_ERR_UNSUPPORTED
