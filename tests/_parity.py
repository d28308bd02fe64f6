"""GPU-vs-oracle comparison rules, shared by the GPU tests (the rules live in
``oracle/parity.py`` so that the bench's CPU leg reports the same counts)."""
from __future__ import annotations

from oracle.parity import P_ATOL, P_RTOL, TV_ATOL, TV_RTOL, assert_parity, compare, prob_errors, token_counts  # noqa: F401


def token_parity(got: dict, ref: dict, k: int | None = None) -> dict:
    """Token and tau comparison only, raising on a chain that differs outside the tie band."""
    s = token_counts(got, ref)
    bad = s.pop("beyond_band")
    assert not bad, f"{len(bad)} chains disagree beyond the tie band, first: {bad[:3]}"
    return s
