"""Comparison of the CUDA path's verify outputs with the oracle's (test helper).

Bit-exact on accept_len, out_tokens, num_emitted and the per-position status
for every request the oracle did not flag.  A flagged request holds a
decision inside its margin (ratio test |u - p/q| < 1e-6, top-p prefix within
1e-9 of the threshold, inverse-CDF draw within 1e-9 of a boundary, residual
mass below 1e-9); such a decision may go either way, and the result must be
one of the outcomes the oracle's decisions allow:

* every position before the accepted length accepts, or its decision is
  ambiguous; the position at the accepted length rejects, or is ambiguous
  (block verification: the accepted length is the last position whose stop
  test passes, each test taken either way where it is ambiguous);
* the accepted tokens are the request's drafts and nothing follows the
  emitted token;
* the emitted token is the one the oracle draws when the chain stops there,
  or a token across a near boundary of that draw, or -- when the distribution
  drawn from is itself uncertain (a near top-p cut, a near-empty residual) --
  a token of the target row's support (with the token its cut leaves out
  next);
* the error bits of every position are the oracle's.

Every comparison adds its flagged and total decisions to a session tally,
which the test session prints at its end.
"""
import numpy as np

import oracle

# flagged decisions, decisions (on the oracle's own paths), flagged requests,
# requests; summed over the session and printed by tests/conftest.py
TALLY = {"flagged": 0, "decisions": 0, "flagged_requests": 0, "requests": 0}


def valid_accepts(dec_row, v: int, block: bool) -> list:
    """The accepted lengths the per-position decisions allow."""
    acc = [(int(x) & oracle.ALT_ACCEPT) != 0 for x in dec_row]
    amb = [(int(x) & oracle.ALT_AMBIG) != 0 for x in dec_row]
    out = []
    for a in range(v + 1):
        if block:
            # a = the last j in 1..v with eta_j < h_j (0 if none)
            ok = all((not acc[i]) or amb[i] for i in range(a + 1, v + 1)) and (a == 0 or acc[a] or amb[a])
        else:
            ok = all(acc[j] or amb[j] for j in range(a)) and (a == v or (not acc[a]) or amb[a])
        if ok:
            out.append(a)
    return out


def valid_token(orc: dict, r: int, a: int, t: int) -> bool:
    """Whether t may be the token emitted after a accepted drafts."""
    bits = int(orc["alt_dec"][r, a])
    if t == int(orc["alt_draw"][r, a]):
        return True
    if bits & oracle.ALT_DRAW_NEAR and t in [int(x) for x in orc["alt_tokens"][r, a] if x >= 0]:
        return True
    if bits & oracle.ALT_DRAW_ROW and 0 <= t < len(orc["support"](r, a)):
        return bool(orc["support"](r, a)[t])
    return False


def check_flagged(orc: dict, r: int, acc, tok, nem, st, drafts, v: int) -> str:
    """'' if request r's result is one of the outcomes its decisions allow,
    else the reason it is not."""
    a = int(acc)
    if a not in valid_accepts(orc["alt_dec"][r], v, orc.get("block", False)):
        return f"accept_len {a} not allowed (oracle {int(orc['accept_len'][r])})"
    if int(nem) != a + 1:
        return f"num_emitted {int(nem)} != accept_len + 1"
    if not (tok[:a] == drafts[:a]).all() or not (tok[a + 1:] == -1).all():
        return "accepted tokens are not the drafts, or tokens follow the emitted one"
    if not valid_token(orc, r, a, int(tok[a])):
        return f"token {int(tok[a])} is not an outcome of the draw at {a}"
    if not np.array_equal(st & oracle.ERROR_MASK, orc["pos_status"][r] & oracle.ERROR_MASK):
        return "error bits differ"
    return ""


def compare_verify(orc: dict, gpu, draft_tokens, windows, vocab, max_flag_rate=None):
    """Compare a verify call's outputs with the oracle's; returns the number of
    flagged requests.  max_flag_rate bounds the flagged decisions over all
    decisions of this comparison (the oracle's own path)."""
    acc = gpu.accept_len.cpu().numpy()
    tok = gpu.out_tokens.cpu().numpy()
    nem = gpu.num_emitted.cpu().numpy()
    st = gpu.row_status.cpu().numpy()
    toks = np.asarray(draft_tokens)
    n = len(acc)
    flagged = orc["flags"] != 0
    bad = []
    for r in range(n):
        exact = acc[r] == orc["accept_len"][r] and nem[r] == orc["num_emitted"][r] \
            and np.array_equal(tok[r], orc["out_tokens"][r]) and np.array_equal(st[r], orc["pos_status"][r])
        if exact:
            continue
        if flagged[r] and orc["num_emitted"][r] > 0:
            why = check_flagged(orc, r, acc[r], tok[r], nem[r], st[r], toks[r], int(windows[r]))
            if why:
                bad.append((r, "flagged request: " + why, acc[r], tok[r].tolist(), "oracle",
                            int(orc["accept_len"][r]), orc["out_tokens"][r].tolist()))
            continue
        bad.append((r, "gpu", acc[r], tok[r].tolist(), st[r].tolist(), "oracle", int(orc["accept_len"][r]),
                    orc["out_tokens"][r].tolist(), orc["pos_status"][r].tolist()))
    assert not bad, bad[:5]
    n_flag, n_dec = int(orc["n_flag"].sum()), int(orc["n_dec"].sum())
    TALLY["flagged"] += n_flag
    TALLY["decisions"] += n_dec
    TALLY["flagged_requests"] += int(flagged.sum())
    TALLY["requests"] += n
    if max_flag_rate is not None:
        assert n_flag <= max_flag_rate * max(n_dec, 1), (n_flag, n_dec)
    return int(flagged.sum())
