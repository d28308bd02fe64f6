"""The GPU-versus-oracle comparison rules on hand-made results (no GPU): a
token mismatch is allowed only at a decision the oracle flagged as a tie, and
every flagged decision is counted."""
import numpy as np

from oracle import parity


def _ref(B=4, k=3):
    tokens = np.arange(B * (k + 1), dtype=np.int32).reshape(B, k + 1)
    tau = np.array([3, 1, 0, 2], np.int32)[:B]
    for b in range(B):
        tokens[b, tau[b] + 1:] = -1
    return {"tokens": tokens, "tau": tau, "accept_tie": np.zeros((B, k), np.int32), "cdf_tie": np.zeros(B, np.int32),
            "p_draft": np.full((B, k), 0.25), "q_draft": np.full((B, k), 0.5), "tv": np.full((B, k), 0.3)}


def _got(ref):
    return {"tokens": ref["tokens"].copy(), "tau": ref["tau"].copy(), "p_draft": ref["p_draft"].astype(np.float32),
            "q_draft": ref["q_draft"].astype(np.float32), "tv": ref["tv"].astype(np.float32)}


def test_identical_results_are_exact():
    ref = _ref()
    s = parity.compare(_got(ref), ref)
    assert s["ok"] and s["exact"] == 4 and s["ties_flagged"] == 0 and s["tie_mismatch"] == 0
    assert s["p_draft_max_rel"] == 0.0 and s["tv_max_abs"] < 1e-7


def test_mismatch_at_flagged_accept_tie_is_allowed_and_counted():
    ref = _ref()
    ref["accept_tie"][1, 1] = 1          # chain 1 rejected at position 2 within the band
    got = _got(ref)
    got["tau"][1] = 2                    # the GPU accepted it instead
    got["tokens"][1] = [4, 5, 77, -1]
    s = parity.compare(got, ref)
    assert s["ok"] and s["ties_flagged"] == 1 and s["tie_mismatch"] == 1 and s["exact"] == 3
    parity.assert_parity(got, ref)


def test_unflagged_mismatch_fails():
    ref = _ref()
    got = _got(ref)
    got["tokens"][2, 0] = 99             # a different final draw with no CDF tie flagged
    s = parity.compare(got, ref)
    assert not s["ok"] and s["beyond_band"] == 1
    try:
        parity.assert_parity(got, ref)
    except AssertionError:
        pass
    else:
        raise AssertionError("an unflagged mismatch passed")
    ref["cdf_tie"][2] = 1                # flagged: now allowed
    assert parity.compare(got, ref)["ok"]


def test_flag_counted_without_mismatch_and_prefix_mismatch_fails():
    ref = _ref()
    ref["cdf_tie"][0] = 1
    got = _got(ref)
    s = parity.compare(got, ref)
    assert s["ok"] and s["ties_flagged"] == 1 and s["tie_mismatch"] == 0
    got["tokens"][0, 0] = 5              # an accepted draft differs: never a tie
    assert not parity.compare(got, ref)["ok"]


def test_probability_and_tv_tolerances():
    ref = _ref()
    got = _got(ref)
    got["p_draft"][0, 0] = np.float32(0.25 * (1 + 2e-5))
    got["tv"][3, 2] = np.float32(0.3 + 5e-6)
    s = parity.compare(got, ref)
    assert not s["ok"] and s["p_draft_violations"] == 1 and s["tv_violations"] == 1
    assert abs(s["p_draft_max_rel"] - 2e-5) < 1e-6
