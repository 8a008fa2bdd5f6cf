"""The C-ABI library loads and exports what include/sv.h declares (no GPU).

Only host-side entry behaviour is exercised here: the size function, the
status strings and argument checks that must fail before any launch.
"""
import ctypes
import os
import re
import subprocess

import pytest

from speculative_decoding_verification_rows_gb300 import build as sv_build
from speculative_decoding_verification_rows_gb300 import sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sv_build.build()
    return sv.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "sv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_symbols() == sorted(sv.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sv_build.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (sv_\w+)", out))
    for name in declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)


def test_workspace_size_and_status_strings(lib):
    assert lib.sv_workspace_size(128, 7, 248_320) > 0
    assert lib.sv_workspace_size(128, 7, 248_320) >= lib.sv_workspace_size(4, 4, 1024)
    assert lib.sv_workspace_size(256, 16, 0) >= 256 * 16 * 8           # planner keys
    assert lib.sv_workspace_size(-1, 4, 10) == 0
    assert lib.sv_workspace_size(4, 64, 10) == 0                         # K beyond the bit masks
    assert lib.sv_workspace_size(4, 4, 10_000_000) == 0                  # vocab beyond one cluster per row
    for code, name in [(0, b"SV_OK"), (1, b"SV_ERR_INVALID_ARG"), (2, b"SV_ERR_WORKSPACE"), (3, b"SV_ERR_CUDA"),
                       (4, b"SV_ERR_UNSUPPORTED")]:
        assert lib.sv_status_string(code) == name


def test_argument_errors_return_before_any_launch(lib):
    S = sv.Sampling(None, None, None)
    null = None
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the checks fail first
    rc = lib.sv_verify_chain(null, null, 0, 4, 4, 1024, fake, null, sv.Sampling(0x1000, None, None), 0,
                             fake, fake, fake, null, fake, 1 << 20, null)
    assert rc == sv.SV_ERR_INVALID_ARG                                   # target missing
    rc = lib.sv_verify_chain(fake, null, 0, 4, 4, 1024, fake, null, S, 0, fake, fake, fake, null, fake, 1 << 20, null)
    assert rc == sv.SV_ERR_INVALID_ARG                                   # temperature missing
    rc = lib.sv_verify_chain(fake, null, 7, 4, 4, 1024, fake, null, sv.Sampling(0x1000, None, None), 0,
                             fake, fake, fake, null, fake, 1 << 20, null)
    assert rc == sv.SV_ERR_INVALID_ARG                                   # dtype
    rc = lib.sv_verify_chain(fake, null, 0, 4, 4, 1024, fake, null, sv.Sampling(0x1000, None, None), 0,
                             fake, fake, fake, null, fake, 16, null)
    assert rc == sv.SV_ERR_WORKSPACE                                     # workspace too small
    rc = lib.sv_verify_chain(fake, null, 0, 4, 4, 1024, fake, null, sv.Sampling(0x1000, None, None), 0,
                             fake, fake, fake, null, ctypes.c_void_p(0x1001), 1 << 30, null)
    assert rc == sv.SV_ERR_WORKSPACE                                     # misaligned workspace
    rc = lib.sv_verify_chain(fake, null, 0, 4, 70, 1024, fake, null, sv.Sampling(0x1000, None, None), 0,
                             fake, fake, fake, null, fake, 1 << 30, null)
    assert rc == sv.SV_ERR_UNSUPPORTED                                   # K beyond 63
    rc = lib.sv_verify_ragged(fake, null, 0, 4, 4, 1024, 20, null, fake, fake, sv.Sampling(0x1000, None, None),
                              0, fake, fake, fake, null, fake, 1 << 30, null)
    assert rc == sv.SV_ERR_INVALID_ARG                                   # qo_indptr missing
    out = (ctypes.c_int32 * 8)()
    rc = lib.sv_plan_budget(fake, 4, null, 4, 4, 3, 8, out, out, out, null, fake, 1 << 20, null)
    assert rc == sv.SV_ERR_INVALID_ARG                                   # budget < n_req
    rc = lib.sv_plan_budget(fake, 4, null, 4, 4, 8, 7, out, out, out, null, fake, 1 << 20, null)
    assert rc == sv.SV_ERR_INVALID_ARG                                   # bucket < budget
    rc = lib.sv_plan_budget(fake, 3, null, 4, 4, 8, 8, out, out, out, null, fake, 1 << 20, null)
    assert rc == sv.SV_ERR_INVALID_ARG                                   # ld_conf < K
    rc = lib.sv_build_target_probs(fake, 0, 100, 4, 1024, null, 4, sv.Sampling(0x1000, None, None), null, null,
                                   null, null, fake, 1 << 30, null)
    assert rc == sv.SV_ERR_INVALID_ARG                                   # row stride < vocab


def test_product_path_has_no_cpu_fallback():
    # the binding refuses host tensors instead of computing anything on the CPU
    import torch
    with pytest.raises(sv.SVError):
        sv.verify_chain(torch.zeros((1, 2, 8)), None, torch.zeros((1, 1), dtype=torch.int32), torch.zeros(1))
    src = open(os.path.join(ROOT, "speculative_decoding_verification_rows_gb300", "sv.py")).read()
    assert "oracle" not in src.replace("no CPU fallback", "")


def test_struct_layouts_match_the_header(tmp_path):
    # the binding's ctypes structs against the C compiler's view of sv.h
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "sv.h"\n'
                   "int main(void) {\n"
                   '  printf("%zu %zu %zu\\n", sizeof(sv_sampling_t), offsetof(sv_sampling_t, top_p),\n'
                   "         offsetof(sv_sampling_t, flags));\n"
                   '  printf("%zu %zu\\n", sizeof(sv_row_desc_t), offsetof(sv_row_desc_t, temperature));\n'
                   '  printf("%d\\n", (int)SV_SAMPLING_SMALL_TOPK);\n'
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    assert [int(x) for x in lines[0].split()] == [ctypes.sizeof(sv.Sampling), sv.Sampling.top_p.offset,
                                                  sv.Sampling.flags.offset]
    assert [int(x) for x in lines[1].split()] == [ctypes.sizeof(sv.RowDesc), sv.RowDesc.temperature.offset]
    assert int(lines[2]) == sv.SAMPLING_SMALL_TOPK
