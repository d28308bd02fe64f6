"""spec_verify_lazy (CUDA, through the C ABI): tokens and tau bit-identical to
spec_verify's and in parity with the oracle, while reading no row past a
chain's first rejection."""
import numpy as np
import pytest

import spec_inputs as si
from tests import _parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_68_gb300 as sv
    sv.build()
    return sv


def to_dev(b):
    dev = torch.device("cuda")
    if b.workload.dtype == si.BF16:
        tgt = torch.from_numpy(b.target.view(np.int16)).to(dev).view(torch.bfloat16)
        dft = torch.from_numpy(b.draft.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        tgt = torch.from_numpy(b.target).to(dev)
        dft = torch.from_numpy(b.draft).to(dev)
    return (tgt, dft, torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.temperature).to(dev),
            torch.from_numpy(b.uniforms).to(dev))


def run(lib, w, b):
    v = lib.SpecVerifier(max(1, b.nb), w.k, w.vocab, torch.float32 if w.dtype == si.FP32 else torch.bfloat16)
    ins = to_dev(b)
    full = v.verify(*ins, want_pq=False)
    lazy = v.verify_lazy(*ins)
    lazy2 = v.verify_lazy(*ins)   # a second call runs on the first call's workspace
    torch.cuda.synchronize()
    v.close()
    c = lambda o: {k: t.cpu().numpy() for k, t in o.items()}
    return c(full), c(lazy), c(lazy2)


@pytest.mark.parametrize("w", [si.TINY, si.C2, si.C3_T0, si.C3_T06, si.C3_T1, si.C4, si.C5.scaled(batch=96)],
                         ids=lambda w: w.name)
def test_lazy_matches_full_and_oracle(lib, oracle, w):
    b = si.generate(w)
    full, lazy, lazy2 = run(lib, w, b)
    for key in ("tokens", "tau"):
        assert np.array_equal(full[key], lazy[key]), key
        assert np.array_equal(lazy[key], lazy2[key]), key
    ref = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, want_tv=False, nthreads=16)
    stats = _parity.token_parity(lazy, ref, w.k)
    print(w.name, stats, "mean tau", float(lazy["tau"].mean()))


@pytest.mark.parametrize("V,dtype", [(37, si.FP32), (2050, si.BF16), (32001, si.BF16), (262144, si.BF16), (151552, si.FP32)])
def test_lazy_ragged(lib, oracle, V, dtype):
    w = si.Workload(f"lazy_V{V}", 9, 5, V, dtype, 2.0, draft_sigma=0.4, temp_mode=1, temp_lo=0.0, temp_hi=1.5)
    b = si.generate(w)
    full, lazy, _ = run(lib, w, b)
    assert np.array_equal(full["tokens"], lazy["tokens"]) and np.array_equal(full["tau"], lazy["tau"])


def test_lazy_reads_only_up_to_the_stop(lib):
    """A NaN row after a chain's stop leaves the lazy result valid (the full
    path reads it and flags the chain); before the stop both flag the chain."""
    w = si.Workload("lazy_nan", 6, 6, 3000, si.FP32, 2.0, draft_sigma=3.0, temp_lo=1.0, temp_hi=1.0)
    b = si.generate(w)
    full, lazy, _ = run(lib, w, b)
    tau = lazy["tau"]
    late = [i for i in range(w.batch) if tau[i] < w.k - 1]
    assert late, "expected early rejections with these drafts"
    c1 = late[0]
    c2 = next(i for i in range(w.batch) if i != c1)
    b.draft[c1, w.k - 1, 3] = np.nan          # after c1's stop: never read by the lazy path
    b.target[c2, 0, 5] = np.nan               # position 0 is always read
    full2, lazy2, _ = run(lib, w, b)
    assert lazy2["tau"][c1] == tau[c1] and np.array_equal(lazy2["tokens"][c1], lazy["tokens"][c1])
    assert full2["tau"][c1] == -1
    assert lazy2["tau"][c2] == -1 and full2["tau"][c2] == -1


def test_lazy_all_accepted_walks_to_the_bonus(lib, oracle):
    """Identical draft and target rows accept every draft: every chain walks
    all k positions and draws its bonus token from target row k."""
    w = si.Workload("lazy_same", 50, 5, 4099, si.BF16, 2.0, draft_sigma=0.0)
    b = si.generate(w)
    assert np.array_equal(b.draft, b.target[:, :w.k])
    full, lazy, lazy2 = run(lib, w, b)
    assert np.all(lazy["tau"] == w.k)
    for key in ("tokens", "tau"):
        assert np.array_equal(full[key], lazy[key]) and np.array_equal(lazy[key], lazy2[key]), key
    ref = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, want_tv=False, nthreads=16)
    _parity.token_parity(lazy, ref, w.k)


@pytest.mark.parametrize("B", [1, 2, 5, 37, 73])
def test_lazy_chain_counts(lib, oracle, B):
    """Fewer chains than clusters, one or two per cluster, and more: each
    cluster walks its share of the chains two at a time."""
    w = si.Workload(f"lazy_b{B}", B, 3, 151552, si.BF16, 2.0, draft_sigma=0.6, temp_mode=1, temp_lo=0.5,
                    temp_hi=1.2)
    b = si.generate(w)
    full, lazy, lazy2 = run(lib, w, b)
    for key in ("tokens", "tau"):
        assert np.array_equal(full[key], lazy[key]) and np.array_equal(lazy[key], lazy2[key]), key
    ref = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, want_tv=False, nthreads=16)
    _parity.token_parity(lazy, ref, w.k)
    if B >= 2:   # with these seeds chain 1 accepts all three drafts
        assert lazy["tau"].max() == w.k
