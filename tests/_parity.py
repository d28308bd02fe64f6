"""GPU-vs-oracle comparison rules.

Tokens and tau must be identical, except where the oracle flagged the
deciding uniform as lying within 1e-6 of the accept threshold or of a CDF
boundary (a "tie"); after such a decision the rest of that chain is excluded
from token comparison.  p(x), q(x) must agree to 1e-5 relative (1e-12
absolute floor); TV to 1e-5 relative plus 1e-6 absolute (fp32 sums over
151,552 terms).
"""
from __future__ import annotations

import numpy as np

P_RTOL, P_ATOL = 1e-5, 1e-12
TV_RTOL, TV_ATOL = 1e-5, 1e-6


def token_parity(got: dict, ref: dict, k: int) -> dict:
    """Per-chain comparison of tokens and tau; returns counts, raises on a real mismatch."""
    gt, gtau = got["tokens"], got["tau"]
    rt, rtau = ref["tokens"], ref["tau"]
    B = rtau.shape[0]
    exact = ties_flagged = tie_mismatch = 0
    bad = []
    for b in range(B):
        flagged = bool(ref["accept_tie"][b].any() or ref["cdf_tie"][b])
        ties_flagged += flagged
        if gtau[b] == rtau[b] and np.array_equal(gt[b], rt[b]):
            exact += 1
            continue
        if rtau[b] < 0 or gtau[b] < 0:
            bad.append((b, "validity", int(gtau[b]), int(rtau[b])))
            continue
        d = min(int(gtau[b]), int(rtau[b]))
        if not np.array_equal(gt[b, :d], rt[b, :d]):
            bad.append((b, "prefix", gt[b].tolist(), rt[b].tolist()))
            continue
        if gtau[b] != rtau[b]:
            ok = bool(ref["accept_tie"][b, d])
        else:
            ok = bool(ref["cdf_tie"][b])
        if ok:
            tie_mismatch += 1
        else:
            bad.append((b, "decision", gt[b].tolist(), rt[b].tolist(), int(gtau[b]), int(rtau[b])))
    assert not bad, f"{len(bad)} chains disagree beyond the tie band, first: {bad[:3]}"
    return {"chains": B, "exact": exact, "ties_flagged": ties_flagged, "tie_mismatch": tie_mismatch}


def prob_parity(got: dict, ref: dict) -> dict:
    stats = {}
    valid = ref["tau"] >= 0
    for key in ("p_draft", "q_draft"):
        if key in got:
            g = got[key][valid].astype(np.float64)
            o = ref[key][valid]
            err = np.abs(g - o)
            assert np.all(err <= P_RTOL * np.abs(o) + P_ATOL), (key, float(np.max(err / (np.abs(o) + 1e-30))))
            stats[f"{key}_max_rel"] = float(np.max(err / np.maximum(np.abs(o), 1e-30))) if err.size else 0.0
    if "tv" in got:
        g = got["tv"][valid].astype(np.float64)
        o = ref["tv"][valid]
        err = np.abs(g - o)
        assert np.all(err <= TV_RTOL * o + TV_ATOL), ("tv", float(err.max()))
        stats["tv_max_abs"] = float(err.max()) if err.size else 0.0
    return stats


def assert_parity(got: dict, ref: dict, k: int) -> dict:
    s = token_parity(got, ref, k)
    s.update(prob_parity(got, ref))
    return s
