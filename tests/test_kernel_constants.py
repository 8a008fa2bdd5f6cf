"""Constant tables the CUDA sources carry, checked against their
definitions on the host (no GPU).

The double-float exp of the kernels takes 2^(j / 64), j = 0 .. 63, from a
table of (hi, lo) float pairs: hi must be the value rounded to fp32 and
hi + lo must lie within 2^-47 of the value (computed here to 50 digits).
"""
import os
import re
from decimal import Decimal, getcontext

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "speculative_decoding_verification_rows_gb300", "csrc", "sv_internal.cuh")


def _exp2_table():
    text = open(HEADER).read()
    body = text[text.index("c_exp2_64[64] = {"):]
    body = body[body.index("{") + 1:body.index("};")]
    pairs = re.findall(r"\{\s*([^,{}]+?)\s*,\s*([^,{}]+?)\s*\}", body)
    return [(float.fromhex(h.rstrip("f")) if "0x" in h else float(h.rstrip("f")),
             float.fromhex(l.rstrip("f")) if "0x" in l else float(l.rstrip("f"))) for h, l in pairs]


def test_exp2_table_is_two_to_the_j_over_64():
    getcontext().prec = 50
    tab = _exp2_table()
    assert len(tab) == 64
    ln2 = Decimal(2).ln()
    for j, (hi, lo) in enumerate(tab):
        exact = (ln2 * j / 64).exp()
        assert np.float32(hi) == hi and np.float32(lo) == lo, j        # both parts are floats
        assert hi == float(np.float32(float(exact))), j                 # hi: the value rounded to fp32
        err = abs(Decimal(hi) + Decimal(lo) - exact) / exact
        assert err < Decimal(2) ** -47, (j, err)
