"""GPU-versus-oracle comparison rules (test infrastructure, like the rest of
this package: only the tests, ``__graft_entry__.smoke()`` and the CPU leg of
``bench.py`` import it).

Tokens and tau must be identical, except where the oracle flagged the
deciding uniform as lying within 1e-6 of the accept threshold or of a CDF
boundary (a "tie", page "Optimizing speculative decoding", section "Rejection
sampling and a loss that optimizes acceptance directly": the accept test and
the residual draw); after such a decision the rest of that chain is excluded
from token comparison.  Flagged decisions are counted whether or not the two
sides differ there.  p(x), q(x) must agree to 1e-5 relative (1e-12 absolute
floor); TV to 1e-5 relative plus 1e-6 absolute (fp32 sums over 151,552
terms).  ``compare`` returns the counts and the largest errors seen;
``assert_parity`` also raises on a violation.
"""
from __future__ import annotations

import numpy as np

P_RTOL, P_ATOL = 1e-5, 1e-12
TV_RTOL, TV_ATOL = 1e-5, 1e-6


def token_counts(got: dict, ref: dict) -> dict:
    """Per-chain comparison of tokens and tau.  Returns the counts and the
    list of chains that differ outside the tie band (``beyond_band``)."""
    gt, gtau = np.asarray(got["tokens"]), np.asarray(got["tau"])
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
    return {"chains": int(B), "exact": exact, "ties_flagged": ties_flagged, "tie_mismatch": tie_mismatch,
            "invalid": int((rtau < 0).sum()), "beyond_band": bad}


def prob_errors(got: dict, ref: dict) -> dict:
    """Largest errors of p(x), q(x) (relative) and TV (absolute) over the valid
    chains, and how many entries break the tolerances."""
    stats = {}
    valid = ref["tau"] >= 0
    for key in ("p_draft", "q_draft"):
        if key in got and got[key] is not None:
            g = np.asarray(got[key])[valid].astype(np.float64)
            o = ref[key][valid]
            err = np.abs(g - o)
            stats[f"{key}_max_rel"] = float(np.max(err / np.maximum(np.abs(o), 1e-30))) if err.size else 0.0
            stats[f"{key}_violations"] = int((~(err <= P_RTOL * np.abs(o) + P_ATOL)).sum())
    if "tv" in got and got["tv"] is not None:
        g = np.asarray(got["tv"])[valid].astype(np.float64)
        o = ref["tv"][valid]
        err = np.abs(g - o)
        stats["tv_max_abs"] = float(err.max()) if err.size else 0.0
        stats["tv_max_rel"] = float(np.max(err / np.maximum(np.abs(o), 1e-30))) if err.size else 0.0
        stats["tv_violations"] = int((~(err <= TV_RTOL * o + TV_ATOL)).sum())
    return stats


def compare(got: dict, ref: dict) -> dict:
    """Counts and largest errors of one GPU result against the oracle's
    (no exception; ``ok`` is False on any violation)."""
    s = token_counts(got, ref)
    s.update(prob_errors(got, ref))
    bad = s.pop("beyond_band")
    s["beyond_band"] = len(bad)
    s["first_beyond_band"] = [list(map(str, x)) for x in bad[:3]]
    s["ok"] = not bad and all(v == 0 for key, v in s.items() if key.endswith("_violations"))
    return s


def assert_parity(got: dict, ref: dict, k: int | None = None) -> dict:
    """compare(), raising AssertionError on a chain that differs outside the
    tie band or a probability / TV beyond its tolerance."""
    s = token_counts(got, ref)
    bad = s.pop("beyond_band")
    assert not bad, f"{len(bad)} chains disagree beyond the tie band, first: {bad[:3]}"
    valid = ref["tau"] >= 0
    for key in ("p_draft", "q_draft"):
        if key in got and got[key] is not None:
            g = np.asarray(got[key])[valid].astype(np.float64)
            o = ref[key][valid]
            err = np.abs(g - o)
            assert np.all(err <= P_RTOL * np.abs(o) + P_ATOL), (key, float(np.max(err / (np.abs(o) + 1e-30))))
    if "tv" in got and got["tv"] is not None:
        g = np.asarray(got["tv"])[valid].astype(np.float64)
        o = ref["tv"][valid]
        err = np.abs(g - o)
        assert np.all(err <= TV_RTOL * o + TV_ATOL), ("tv", float(err.max()))
    s.update(prob_errors(got, ref))
    return s
