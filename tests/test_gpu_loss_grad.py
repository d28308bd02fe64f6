"""spec_verify_loss_grad (CUDA, through the C ABI) against the fp64 oracle:
per-position losses (TV = 1 - alpha, overlap = -ln alpha, alpha = sum
min(p, q)) and the gradient of the weighted loss with respect to the draft
logits.

Tolerances.  alpha and beta are fp32 sums of ex2.approx values (relative
error below 2^-22 each, fp32 accumulation about log2(V) * 2^-24), so both
carry a relative error of a few 1e-7: the losses are compared to 2e-6
(TV) and 2e-6 / alpha (overlap).  Each gradient entry K e_d ([q < p] - beta)
is formed in fp32 and rounded once to the logit dtype, so a bf16 entry may
sit one bf16 step (2^-7 relative) from the rounded fp64 value, and an fp32
entry within 2e-5 relative (plus 1e-7 of the row's largest entry, for
entries near beta's cancellation).  Entries with |p - q| <= 1e-6 max(p, q),
where the subgradient [q < p] is arbitrary, are left out; positions whose
near-tie draft mass could move beta by more than 1e-6 are skipped whole."""
import numpy as np
import pytest

import spec_inputs as si

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_68_gb300 as sv
    sv.build()
    return sv


def bf16_round(x):
    """fp64 -> bf16 (round to nearest even) -> fp64."""
    f = np.asarray(x, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def to_dev(b):
    dev = torch.device("cuda")
    if b.workload.dtype == si.BF16:
        tgt = torch.from_numpy(b.target.view(np.int16)).to(dev).view(torch.bfloat16)
        dft = torch.from_numpy(b.draft.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        tgt = torch.from_numpy(b.target).to(dev)
        dft = torch.from_numpy(b.draft).to(dev)
    return tgt, dft, torch.from_numpy(b.temperature).to(dev)


def check(lib, oracle, w, kind, b=None, weights=None):
    b = b if b is not None else si.generate(w)
    tgt, dft, tmp = to_dev(b)
    v = lib.SpecVerifier(max(1, b.nb), w.k, w.vocab, torch.float32 if w.dtype == si.FP32 else torch.bfloat16)
    wt = None if weights is None else torch.from_numpy(weights).cuda()
    out = v.loss_grad(tgt, dft, tmp, kind=kind, weights=wt)
    torch.cuda.synchronize()
    v.close()
    loss = out["loss"].cpu().numpy().astype(np.float64)
    if w.dtype == si.BF16:
        grad = out["grad"].view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
        grad = grad.view(np.float32).astype(np.float64)
    else:
        grad = out["grad"].cpu().numpy().astype(np.float64)
    ref = oracle.overlap_grad_batch(b.target, b.draft, b.temperature, 0 if kind == "tv" else 1, weights,
                                    w.dtype, nthreads=16)
    assert np.array_equal(np.isnan(loss), np.isnan(ref["loss"]))
    B, k, V = grad.shape
    checked = skipped = 0
    for bi in range(B):
        for i in range(k):
            if np.isnan(ref["loss"][bi, i]):
                assert not np.any(grad[bi, i]), "invalid position must have a zero gradient"
                continue
            alpha = ref["alpha"][bi, i]
            tol = 2e-6 if kind == "tv" else 2e-6 / alpha
            assert abs(loss[bi, i] - ref["loss"][bi, i]) <= tol, (bi, i, loss[bi, i], ref["loss"][bi, i])
            if ref["tie"][bi, i] > 1e-6:
                skipped += 1
                continue
            T = float(b.temperature[bi])
            p = oracle.probs(b.target[bi, i], T, w.dtype)
            q = oracle.probs(b.draft[bi, i], T, w.dtype)
            keep = ~(np.abs(p - q) <= 1e-6 * np.maximum(p, q))
            gr = ref["grad"][bi, i]
            gg = grad[bi, i]
            if w.dtype == si.BF16:
                want = bf16_round(gr)
                ok = np.abs(gg - want) <= 2.0 ** -7 * np.abs(want) + 1e-30
            else:
                ok = np.abs(gg - gr) <= 2e-5 * np.abs(gr) + 1e-7 * np.abs(gr).max()
            assert np.all(ok | ~keep), (bi, i, int((~ok & keep).sum()))
            # softmax gradients sum to zero; after rounding each entry to the logit dtype
            # the sum is bounded by the rounding (half a bf16 step, 2^-8 relative, per entry)
            bound = (2.0 ** -8 if w.dtype == si.BF16 else 1e-4) * np.abs(gg).sum()
            assert abs(gg.sum()) <= bound + 1e-30
            checked += 1
    print(w.name, kind, "positions checked", checked, "skipped (near-ties)", skipped)
    assert checked > 0 and skipped <= max(1, checked // 10)
    return loss, grad, ref


@pytest.mark.parametrize("kind", ["tv", "overlap"])
@pytest.mark.parametrize("w", [si.TINY, si.C2, si.C3_T1.scaled(batch=6), si.C4.scaled(batch=4), si.C5.scaled(batch=6)],
                         ids=lambda w: w.name)
def test_loss_grad_workloads(lib, oracle, w, kind):
    check(lib, oracle, w, kind)


@pytest.mark.parametrize("V,dtype", [(37, si.FP32), (1001, si.FP32), (2050, si.BF16), (32001, si.BF16)])
def test_loss_grad_ragged_and_weights(lib, oracle, V, dtype):
    w = si.Workload(f"lg_V{V}", 4, 3, V, dtype, 2.0, draft_sigma=0.8, temp_mode=1, temp_lo=0.4, temp_hi=1.5)
    wts = np.random.default_rng(V).uniform(0.2, 3.0, (4, 3)).astype(np.float32)
    check(lib, oracle, w, "overlap", weights=wts)


@pytest.mark.parametrize("kind", ["tv", "overlap"])
@pytest.mark.parametrize("V,dtype", [(262144, si.BF16), (151552, si.FP32)])
def test_loss_grad_large_vocab(lib, oracle, V, dtype, kind):
    """Vocabularies past 163,840 (bf16) or 81,920 (fp32): one CTA per SM.  The
    draft noise keeps near-tie positions (left out of the comparison) rare."""
    w = si.Workload(f"lg_big_V{V}", 4, 3, V, dtype, 2.0, draft_sigma=1.5, temp_mode=1, temp_lo=0.4, temp_hi=1.5)
    wts = np.random.default_rng(V).uniform(0.2, 3.0, (4, 3)).astype(np.float32)
    check(lib, oracle, w, kind, weights=wts)


def test_loss_grad_invalid_and_identical(lib, oracle):
    w = si.Workload("lg_special", 6, 3, 4096, si.BF16, 2.0, draft_sigma=0.5, temp_lo=1.0, temp_hi=1.0)
    b = si.generate(w)
    b.temperature[0] = 0.0            # greedy chain: no sampling distribution, invalid for the losses
    b.draft[1, 2, 5] = 0x7FC0         # a NaN logit (bf16 bits): that position is invalid
    b.draft[2, 1] = b.target[2, 1]    # identical rows: alpha = 1, loss 0, gradient 0
    loss, grad, ref = check(lib, oracle, w, "overlap", b=b)
    assert np.all(np.isnan(loss[0])) and not np.any(grad[0])
    assert np.isnan(loss[1, 2]) and not np.any(grad[1, 2]) and not np.isnan(loss[1, 1])
    assert loss[2, 1] == 0.0 and not np.any(grad[2, 1])
