"""Per-row entropy from spec_verify_ex (CUDA, through the C ABI) against the
fp64 oracle, and the verification outputs of spec_verify_ex bit-identical to
those of spec_verify on the same inputs.

Tolerance.  The kernel forms H = ln S - ln2 * A / S from two fp32 sums over the
row, S = sum e and A = sum e*a with e = 2^a, a = z*c - R (R the row's integer
reference, so |a| <= |z*c - R| and e <= 1).  Each e carries the relative error
of ex2.approx (below 2^-22) and the sums the rounding of fp32 accumulation
(about log2(V) * 2^-24 relative).  |A| / S is the mean of |a| under p, at most
(ln S - H) / ln 2 + 1 <= log2(V) + 1, so the error of H stays below about
(1 + ln 2 * (log2 V + 1)) * 2^-21 ~ 6e-6 at V = 151,552; the tests allow
2e-5 + 2e-6 * H."""
import numpy as np
import pytest

import spec_inputs as si

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-5, 2e-6


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


def run_both(lib, w, b):
    v = lib.SpecVerifier(max(1, b.nb), w.k, w.vocab, torch.float32 if w.dtype == si.FP32 else torch.bfloat16)
    ins = to_dev(b)
    plain = v.verify(*ins, want_tv=True)
    ex = v.verify(*ins, want_tv=True, want_entropy=True)
    torch.cuda.synchronize()
    v.close()
    return ({k: t.cpu().numpy() for k, t in plain.items()}, {k: t.cpu().numpy() for k, t in ex.items()})


def check(lib, oracle, w, b=None):
    b = b if b is not None else si.generate(w)
    plain, ex = run_both(lib, w, b)
    for key in plain:   # the extra statistic changes nothing else
        assert np.array_equal(plain[key], ex[key], equal_nan=True), key
    want_t, want_d = oracle.entropy_batch(b.target, b.draft, b.temperature, w.dtype, nthreads=16)
    worst = 0.0
    for got, want in ((ex["entropy_target"], want_t), (ex["entropy_draft"], want_d)):
        assert np.array_equal(np.isnan(got), np.isnan(want)), "NaN pattern differs"
        ok = ~np.isnan(want)
        err = np.abs(got[ok].astype(np.float64) - want[ok])
        assert np.all(err <= ATOL + RTOL * want[ok]), float(err.max())
        worst = max(worst, float(err.max()) if err.size else 0.0)
    print(w.name, "max |dH|", worst)
    return ex, want_t, want_d


@pytest.mark.parametrize("w", [si.TINY, si.C2, si.C3_T0, si.C3_T06, si.C3_T1, si.C4.scaled(batch=32), si.C5.scaled(batch=48)],
                         ids=lambda w: w.name)
def test_entropy_workloads(lib, oracle, w):
    check(lib, oracle, w)


@pytest.mark.parametrize("V,dtype", [(16, si.FP32), (1001, si.FP32), (2050, si.BF16), (32001, si.BF16), (163840, si.BF16),
                                     (262144, si.BF16), (151552, si.FP32)])
def test_entropy_ragged(lib, oracle, V, dtype):
    w = si.Workload(f"ent_V{V}", 5, 4, V, dtype, 2.0, draft_sigma=0.8, temp_mode=1, temp_lo=0.3, temp_hi=1.5)
    check(lib, oracle, w)


def test_entropy_special_rows(lib, oracle):
    """Greedy and invalid chains, masked tokens, a constant row (H = ln V)."""
    w = si.Workload("ent_special", 8, 3, 4096, si.FP32, 2.0, draft_sigma=0.5, temp_lo=1.0, temp_hi=1.0)
    b = si.generate(w)
    b.temperature[0] = 0.0             # greedy: H = 0 for every row
    b.temperature[1] = -1.0            # invalid temperature: NaN
    b.target[2, 1, 7] = np.nan         # one invalid row: NaN there only
    b.draft[3, 0, :] = -np.inf         # no finite logit: NaN
    b.target[4, 2, 100:] = -np.inf     # masked tokens: the entropy of the first 100
    b.draft[5, 1, :] = 3.5             # constant row: ln V
    ex, want_t, want_d = check(lib, oracle, w, b)
    assert np.all(ex["entropy_target"][0] == 0.0) and np.all(ex["entropy_draft"][0] == 0.0)
    assert np.all(np.isnan(ex["entropy_target"][1])) and np.isnan(ex["entropy_target"][2, 1])
    assert not np.isnan(ex["entropy_target"][2, 0]) and np.isnan(ex["entropy_draft"][3, 0])
    assert abs(float(ex["entropy_draft"][5, 1]) - np.log(4096)) <= ATOL + RTOL * np.log(4096)


def test_entropy_bonus_pairs(lib, oracle):
    """Bonus rows two chains to a unit, each at its own temperature (greedy next
    to sampling, two temperatures, an invalid one, the odd last chain alone)."""
    temps = [0.0, 1.0, 0.7, 0.0, 1.3, 0.5, -1.0, 0.9, 0.0]
    w = si.Workload("ent_bonus_pairs", len(temps), 2, 32001, si.BF16, 2.0, draft_sigma=0.8)
    b = si.generate(w)
    b.temperature[:] = temps
    ex, want_t, want_d = check(lib, oracle, w, b)
    assert ex["entropy_target"][0, w.k] == 0.0 and ex["entropy_target"][3, w.k] == 0.0
    assert np.isnan(ex["entropy_target"][6, w.k]) and not np.isnan(ex["entropy_target"][7, w.k])
