"""Comparison of the CUDA path's verify outputs with the oracle's (test helper).

Bit-exact on accept_len, out_tokens, num_emitted and the per-position status
for every request the oracle did not flag.  A flagged request (a decision
within its margin: ratio test |u - p/q| < 1e-6, top-p prefix within 1e-9 of
the threshold, inverse-CDF draw within 1e-9 of a boundary, residual mass below
1e-9) is only checked for validity: it accepts a prefix of its own drafts, no
longer than its window, and emits one token in range after it.
"""
import numpy as np

import oracle


def compare_verify(orc: dict, gpu, draft_tokens, windows, vocab, max_flag_rate=None):
    acc = gpu.accept_len.cpu().numpy()
    tok = gpu.out_tokens.cpu().numpy()
    nem = gpu.num_emitted.cpu().numpy()
    st = gpu.row_status.cpu().numpy()
    toks = np.asarray(draft_tokens)
    n = len(acc)
    flagged = orc["flags"] != 0
    bad = []
    for r in range(n):
        if flagged[r]:
            a = acc[r]
            ok = 0 <= a <= windows[r] and nem[r] == a + 1 and (tok[r, :a] == toks[r, :a]).all() \
                and 0 <= tok[r, a] < vocab and (tok[r, a + 1:] == -1).all()
            if not ok:
                bad.append((r, "flagged request invalid", acc[r], tok[r].tolist()))
            continue
        if acc[r] != orc["accept_len"][r] or nem[r] != orc["num_emitted"][r] \
                or not np.array_equal(tok[r], orc["out_tokens"][r]) or not np.array_equal(st[r], orc["pos_status"][r]):
            bad.append((r, "gpu", acc[r], tok[r].tolist(), st[r].tolist(), "oracle", int(orc["accept_len"][r]),
                        orc["out_tokens"][r].tolist(), orc["pos_status"][r].tolist()))
    assert not bad, bad[:5]
    if max_flag_rate is not None:
        assert flagged.mean() <= max_flag_rate, flagged.mean()
    return flagged.sum()
