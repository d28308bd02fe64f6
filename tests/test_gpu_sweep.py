"""A seeded sweep over shapes, dtypes, temperatures, draft recipes and masked
vocabulary entries (-inf logits), each checked end to end through the C ABI:
verification against the oracle, lazy verification and the TV-only call
against verification, and the entropies against the oracle."""
import numpy as np
import pytest

import spec_inputs as si
from tests import _parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _cases(n=12, seed=2026):
    rng = np.random.default_rng(seed)
    vocabs = [2, 3, 17, 100, 1003, 4096, 30011, 65536, 151552]
    out = []
    while len(out) < n:
        V = int(rng.choice(vocabs))
        k = int(rng.choice([1, 2, 3, 5, 7, 9, 15, 31]))
        B = int(rng.integers(1, 25))
        if B * (2 * k + 1) * V > 40_000_000:
            continue
        dtype = si.BF16 if rng.random() < 0.6 or V > 81920 else si.FP32
        temp_mode = int(rng.integers(0, 2))
        lo = float(rng.choice([0.0, 0.5, 1.0])) if temp_mode == 0 else 0.2
        w = si.Workload(f"sweep{len(out)}_B{B}_k{k}_V{V}", B, k, V, dtype, float(rng.uniform(0.5, 4.0)),
                        draft_mode=int(rng.random() < 0.3), draft_sigma=float(rng.uniform(0.1, 2.0)),
                        temp_mode=temp_mode, temp_lo=lo, temp_hi=1.5 if temp_mode else lo, seed=len(out) + 7)
        mask = float(rng.choice([0.0, 0.0, 0.2])) if V > 3 else 0.0
        out.append((w, mask))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_68_gb300 as sv
    sv.build()
    return sv


def _masked(w, frac):
    """The workload's batch with the same random vocabulary entries set to -inf in
    every target and draft row (a vocabulary mask); drafted tokens stay unmasked."""
    b = si.generate(w)
    if frac > 0.0:
        rng = np.random.default_rng(w.seed)
        ids = rng.choice(w.vocab, size=int(frac * w.vocab), replace=False)
        ids = np.setdiff1d(ids, np.unique(b.tokens))
        neg_inf = np.uint16(0xFF80) if w.dtype == si.BF16 else np.float32(-np.inf)
        b.target[:, :, ids] = neg_inf
        b.draft[:, :, ids] = neg_inf
    return b


def _dev(b):
    dev = torch.device("cuda")
    if b.workload.dtype == si.BF16:
        tgt = torch.from_numpy(b.target.view(np.int16)).to(dev).view(torch.bfloat16)
        dft = torch.from_numpy(b.draft.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        tgt = torch.from_numpy(b.target).to(dev)
        dft = torch.from_numpy(b.draft).to(dev)
    return (tgt, dft, torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.temperature).to(dev),
            torch.from_numpy(b.uniforms).to(dev))


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}_mask{c[1]}")
def test_sweep(lib, oracle, case):
    w, frac = case
    b = _masked(w, frac)
    ins = _dev(b)
    v = lib.SpecVerifier(w.batch, w.k, w.vocab, torch.float32 if w.dtype == si.FP32 else torch.bfloat16)
    full = v.verify(*ins, want_tv=True, want_entropy=True)
    lazy = v.verify_lazy(*ins)
    tv = v.verify_tv(ins[0], ins[1], ins[3])
    torch.cuda.synchronize()
    rc, n_bad = v.get_error()
    v.close()
    got = {key: t.cpu().numpy() for key, t in full.items()}
    ref = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, nthreads=16)
    stats = _parity.assert_parity({key: got[key] for key in ("tokens", "tau", "p_draft", "q_draft", "tv")}, ref, w.k)
    assert n_bad == int((ref["tau"] < 0).sum())
    for key in ("tokens", "tau"):
        assert np.array_equal(lazy[key].cpu().numpy(), got[key]), key
    assert np.array_equal(tv.cpu().numpy(), got["tv"], equal_nan=True)
    h_t, h_d = oracle.entropy_batch(b.target, b.draft, b.temperature, w.dtype, nthreads=16)
    for g_h, r_h in ((got["entropy_target"], h_t), (got["entropy_draft"], h_d)):
        g_h = g_h.astype(np.float64)
        assert np.array_equal(np.isnan(g_h), np.isnan(r_h))
        ok = np.isnan(r_h) | (np.abs(g_h - r_h) <= 2e-5 + 2e-6 * np.abs(r_h))
        assert ok.all(), float(np.nanmax(np.abs(g_h - r_h)))
    print(w.name, frac, stats)


@pytest.mark.parametrize("T", [0.6, 1.0])
def test_masked_warp_ranges(lib, oracle, T):
    """Whole warp ranges of -inf in one row of a pair: at V = 151,552 bf16 a warp owns 2,304 or
    2,560 consecutive logits of a CTA's 18,944, so a masked block of 6,000 covers at least one
    range, whose part then has no reference.  Chains 0-3 mask the target row, 4-7 the draft row,
    8-11 both, at every position (the bonus row too), in both the rounds whose exponentials wait
    in tensor memory and the rounds that are recomputed."""
    w = si.Workload(f"maskedwarps_T{T}", 12, 7, 151552, si.BF16, 2.0, draft_sigma=0.8, temp_lo=T, temp_hi=T)
    b = si.generate(w)
    neg_inf = np.uint16(0xFF80)
    rng = np.random.default_rng(31)
    for c in range(w.batch):
        lo = int(rng.integers(0, 8)) * (w.vocab // 8) + int(rng.integers(0, 12000))
        hi = lo + 6000
        if c < 4 or c >= 8:
            b.target[c, :, lo:hi] = neg_inf
        if c >= 4:
            b.draft[c, :, lo:hi] = neg_inf
        inside = (b.tokens[c] >= lo) & (b.tokens[c] < hi)
        b.tokens[c, inside] = (b.tokens[c, inside] + 7000) % w.vocab   # drafted tokens stay unmasked
    ins = _dev(b)
    v = lib.SpecVerifier(w.batch, w.k, w.vocab, torch.bfloat16)
    full = v.verify(*ins, want_tv=True, want_entropy=True)
    lazy = v.verify_lazy(*ins)
    torch.cuda.synchronize()
    rc, n_bad = v.get_error()
    v.close()
    got = {key: t.cpu().numpy() for key, t in full.items()}
    ref = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, nthreads=16)
    assert int((ref["tau"] < 0).sum()) == 0 and n_bad == 0
    _parity.assert_parity({key: got[key] for key in ("tokens", "tau", "p_draft", "q_draft", "tv")}, ref, w.k)
    for key in ("tokens", "tau"):
        assert np.array_equal(lazy[key].cpu().numpy(), got[key]), key
    h_t, h_d = oracle.entropy_batch(b.target, b.draft, b.temperature, w.dtype, nthreads=16)
    for g_h, r_h in ((got["entropy_target"], h_t), (got["entropy_draft"], h_d)):
        g_h = g_h.astype(np.float64)
        assert np.all(np.abs(g_h - r_h) <= 2e-5 + 2e-6 * np.abs(r_h)), float(np.max(np.abs(g_h - r_h)))
