"""CUDA library (through the C ABI) against the CPU oracle, on the same seeded inputs."""
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


def to_dev(b: si.Batch):
    dev = torch.device("cuda")
    if b.workload.dtype == si.BF16:
        tgt = torch.from_numpy(b.target.view(np.int16)).to(dev).view(torch.bfloat16)
        dft = torch.from_numpy(b.draft.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        tgt = torch.from_numpy(b.target).to(dev)
        dft = torch.from_numpy(b.draft).to(dev)
    return (tgt, dft, torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.temperature).to(dev),
            torch.from_numpy(b.uniforms).to(dev))


def run_gpu(lib, w, b, flags=0, want_tv=True):
    v = lib.SpecVerifier(max(1, b.nb), w.k, w.vocab, torch.float32 if w.dtype == si.FP32 else torch.bfloat16, flags)
    out = v.verify(*to_dev(b), want_tv=want_tv)
    torch.cuda.synchronize()
    res = {k: t.cpu().numpy() for k, t in out.items()}
    rc, n_bad = v.get_error()
    v.close()
    return res, rc, n_bad


def check(lib, oracle, w, b=None, flags=0):
    b = b if b is not None else si.generate(w)
    got, rc, n_bad = run_gpu(lib, w, b, flags)
    ref = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, nthreads=16)
    stats = _parity.assert_parity(got, ref, w.k)
    n_invalid = int((ref["tau"] < 0).sum())
    assert n_bad == n_invalid and (rc == 0) == (n_invalid == 0), (rc, n_bad, n_invalid)
    print(w.name, stats)
    return got, ref, stats


# -------- the five workloads at full size (every chain compared)
@pytest.mark.parametrize("w", [si.TINY, si.C2, si.C3_T0, si.C3_T06, si.C3_T1, si.C4, si.C5], ids=lambda w: w.name)
def test_workload_full(lib, oracle, w):
    check(lib, oracle, w)


# -------- smaller cases spanning tiles and ragged tails
@pytest.mark.parametrize("V,dtype", [(16, si.FP32), (37, si.FP32), (1000, si.FP32), (1001, si.FP32), (4096, si.BF16),
                                     (2050, si.BF16), (20000, si.BF16), (32001, si.BF16), (81920, si.FP32),
                                     (163840, si.BF16)])
@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_ragged_vocab(lib, oracle, V, dtype, T):
    w = si.Workload(f"ragged_V{V}", 6, 5, V, dtype, 2.0, draft_sigma=0.8, temp_lo=T, temp_hi=T)
    check(lib, oracle, w)


# -------- vocabularies past 163,840 (bf16) or 81,920 (fp32): twice the register rounds, one CTA per SM
@pytest.mark.parametrize("V,dtype", [(163848, si.BF16), (200003, si.BF16), (262144, si.BF16), (327680, si.BF16),
                                     (81928, si.FP32), (151552, si.FP32), (163840, si.FP32)])
def test_large_vocab(lib, oracle, V, dtype):
    w = si.Workload(f"bigV{V}", 5, 3, V, dtype, 2.0, draft_sigma=0.6, temp_mode=1, temp_lo=0.0, temp_hi=1.3)
    check(lib, oracle, w)


@pytest.mark.parametrize("k", [1, 2, 15, 31])
def test_draft_lengths(lib, oracle, k):
    w = si.Workload(f"k{k}", 5, k, 3000, si.BF16, 1.0, draft_sigma=0.3, temp_mode=1, temp_lo=0.5, temp_hi=1.5)
    check(lib, oracle, w)


def test_no_tma_path_bit_identical(lib):
    w = si.C3_T06.scaled(batch=6)
    b = si.generate(w)
    a, _, _ = run_gpu(lib, w, b)
    c, _, _ = run_gpu(lib, w, b, flags=lib.SV_FLAG_NO_TMA)
    for key in a:
        assert np.array_equal(a[key], c[key]), key


def test_deterministic(lib):
    w = si.C4.scaled(batch=16)
    b = si.generate(w)
    a, _, _ = run_gpu(lib, w, b)
    c, _, _ = run_gpu(lib, w, b)
    for key in a:
        assert np.array_equal(a[key], c[key], equal_nan=True), key


def test_identical_rows_accept_all(lib, oracle):
    w = si.C3_T06.scaled(batch=8, vocab=151552)
    b = si.generate(w)
    b.draft[:] = b.target[:, :w.k]
    got, ref, _ = check(lib, oracle, w, b)
    assert np.all(got["tau"] == w.k) and np.all(got["tv"] == 0.0)


def test_greedy_ties_lowest_index(lib, oracle):
    rng = np.random.default_rng(4)
    w = si.Workload("greedy_ties", 32, 7, 5000, si.FP32, 1.0, temp_lo=0.0, temp_hi=0.0)
    b = si.generate(w)
    b.target[:] = rng.integers(-3, 4, b.target.shape).astype(np.float32)
    b.draft[:] = rng.integers(-3, 4, b.draft.shape).astype(np.float32)
    am = np.argmax(b.target, -1)
    b.tokens[:] = np.where(rng.random((32, 7)) < 0.8, am[:, :7], np.argmax(b.draft, -1)).astype(np.int32)
    check(lib, oracle, w, b)


def test_invalid_chains_flagged(lib, oracle):
    w = si.C2.scaled(batch=8, vocab=2048)
    b = si.generate(w)
    b.tokens[1, 3] = w.vocab          # out of range
    b.tokens[2, 0] = -5
    b.temperature[3] = -1.0
    b.temperature[4] = np.nan
    b.target[5, 7, 11] = np.nan       # bonus row
    b.draft[6, 2, :] = -np.inf        # no finite logit
    b.draft[7, 2, 5] = -np.inf        # a masked token: still valid
    got, ref, _ = check(lib, oracle, w, b)
    assert list(np.nonzero(got["tau"] < 0)[0]) == [1, 2, 3, 4, 5, 6]


# The bonus rows of chains 2j and 2j + 1 share one unit; each row keeps its own
# chain's temperature and status.  Pairs here: greedy next to sampling (both
# orders), two greedy, two temperatures, an invalid temperature next to a NaN
# bonus row, a fully masked bonus row next to a valid one, and the odd last
# chain alone.
BONUS_TEMPS = [0.0, 1.0, 0.7, 0.0, 0.0, 0.0, 1.3, 0.5, -1.0, 0.9, 0.8, 1.1, 0.6]


@pytest.mark.parametrize("V,dtype", [(5000, si.FP32), (151552, si.BF16)])
def test_bonus_pairs_mixed_chains(lib, oracle, V, dtype):
    w = si.Workload(f"bonus_pairs_V{V}", len(BONUS_TEMPS), 3, V, dtype, 2.0, draft_sigma=0.6)
    b = si.generate(w)
    b.temperature[:] = BONUS_TEMPS
    nan = np.uint16(0x7FC0) if dtype == si.BF16 else np.float32(np.nan)
    neg_inf = np.uint16(0xFF80) if dtype == si.BF16 else np.float32(-np.inf)
    b.target[9, w.k, 17] = nan
    b.target[11, w.k, :] = neg_inf
    got, ref, _ = check(lib, oracle, w, b)
    assert list(np.nonzero(got["tau"] < 0)[0]) == [8, 9, 11]


def test_spec_verify_tv(lib, oracle):
    w = si.C5.scaled(batch=24)
    b = si.generate(w)
    v = lib.SpecVerifier(24, w.k, w.vocab, torch.bfloat16)
    tgt, dft, _, tmp, _ = to_dev(b)
    tv = v.verify_tv(tgt, dft, tmp).cpu().numpy()
    ref = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, nthreads=16)
    err = np.abs(tv - ref["tv"])
    assert np.all(err <= _parity.TV_RTOL * ref["tv"] + _parity.TV_ATOL)
    v.close()


def test_host_entry_point(lib):
    w = si.C3_T1.scaled(batch=8)
    b = si.generate(w)
    dev, _, _ = run_gpu(lib, w, b)
    v = lib.SpecVerifier(8, w.k, w.vocab, torch.bfloat16, flags=lib.SV_FLAG_HOST_STAGING)
    tg = torch.from_numpy(b.target.view(np.int16)).view(torch.bfloat16).pin_memory()
    dr = torch.from_numpy(b.draft.view(np.int16)).view(torch.bfloat16).pin_memory()
    host_out = v.alloc_outputs(8, want_pq=True, want_tv=True, device="cpu")
    host_out = {k: t.pin_memory() for k, t in host_out.items()}
    v.verify_host(tg, dr, torch.from_numpy(b.tokens), torch.from_numpy(b.temperature), torch.from_numpy(b.uniforms),
                  host_out)
    torch.cuda.synchronize()
    for key in dev:
        assert np.array_equal(dev[key], host_out[key].numpy()), key
    v.close()


def test_host_entry_point_larger_batch(lib):
    """300 chains through spec_verify_host, twice on the same staging buffers:
    the outputs equal those of the device-pointer path."""
    w = si.Workload("host_chunks", 300, 5, 4096, si.BF16, 2.0, draft_sigma=0.6, temp_mode=1, temp_lo=0.0, temp_hi=1.2)
    b = si.generate(w)
    dev, _, _ = run_gpu(lib, w, b)
    v = lib.SpecVerifier(w.batch, w.k, w.vocab, torch.bfloat16, flags=lib.SV_FLAG_HOST_STAGING)
    tg = torch.from_numpy(b.target.view(np.int16)).view(torch.bfloat16).pin_memory()
    dr = torch.from_numpy(b.draft.view(np.int16)).view(torch.bfloat16).pin_memory()
    host_out = {k: t.pin_memory() for k, t in v.alloc_outputs(w.batch, want_pq=True, want_tv=True, device="cpu").items()}
    for _ in range(2):   # the second call reuses the staging buffers
        v.verify_host(tg, dr, torch.from_numpy(b.tokens), torch.from_numpy(b.temperature),
                      torch.from_numpy(b.uniforms), host_out)
        torch.cuda.synchronize()
        for key in dev:
            assert np.array_equal(dev[key], host_out[key].numpy(), equal_nan=True), key
    v.close()


def test_host_entry_point_pageable(lib):
    """Pageable host logits go through the device staging copy; page-locked
    ones are read in place by the kernels.  Both equal the device path."""
    w = si.C3_T06.scaled(batch=6)
    b = si.generate(w)
    dev, _, _ = run_gpu(lib, w, b)
    v = lib.SpecVerifier(w.batch, w.k, w.vocab, torch.bfloat16, flags=lib.SV_FLAG_HOST_STAGING)
    tg = torch.from_numpy(b.target.view(np.int16)).view(torch.bfloat16)
    dr = torch.from_numpy(b.draft.view(np.int16)).view(torch.bfloat16)
    assert not tg.is_pinned() and not dr.is_pinned()
    for pinned in (False, True):
        host_out = v.alloc_outputs(w.batch, want_pq=True, want_tv=True, device="cpu")
        args = (tg.pin_memory(), dr.pin_memory()) if pinned else (tg, dr)
        v.verify_host(*args, torch.from_numpy(b.tokens), torch.from_numpy(b.temperature),
                      torch.from_numpy(b.uniforms), host_out)
        torch.cuda.synchronize()
        for key in dev:
            assert np.array_equal(dev[key], host_out[key].numpy(), equal_nan=True), (pinned, key)
    v.close()


def test_empty_batch_and_bad_args(lib):
    v = lib.SpecVerifier(4, 3, 64, torch.float32)
    e = torch.empty((0, 4, 64), device="cuda")
    out = v.verify(e, torch.empty((0, 3, 64), device="cuda"), torch.empty((0, 3), dtype=torch.int32, device="cuda"),
                   torch.empty((0,), device="cuda"), torch.empty((0, 4), device="cuda"))
    assert out["tokens"].shape == (0, 4)
    with pytest.raises(lib.SpecVerifyError):
        lib.SpecVerifier(4, 32, 64, torch.float32)     # k above the limit
    with pytest.raises(lib.SpecVerifyError):
        lib.SpecVerifier(4, 7, 327681, torch.bfloat16)  # V above the limit
    v.close()


def test_target_preservation_sampled_gpu(lib, oracle):
    """The GPU passes the same chi-squared test as the oracle (tiny rows, 200,000 chains)."""
    import scipy.stats
    from tests import _pins
    n = 200_000
    base = si.generate(si.TINY)
    k, V = si.TINY.k, si.TINY.vocab
    t = np.ascontiguousarray(np.broadcast_to(base.target[0], (n, k + 1, V)))
    d = np.ascontiguousarray(np.broadcast_to(base.draft[0], (n, k, V)))
    x = si.gumbel_argmax(303, d, si.FP32, np.ones(n * k, np.float32)).astype(np.int32)
    u = si.uniforms(303, si.STREAM_VERIFY, 0, n, k + 1)
    b = si.Batch(si.TINY.scaled(batch=n), 0, t, d, x, np.ones(n, np.float32), u)
    got, _, _ = run_gpu(lib, b.workload, b)
    ref = oracle.verify(t, d, x, np.ones(n, np.float32), u, si.FP32, nthreads=16)
    _parity.assert_parity(got, ref, k)
    p = _pins.softmax_rows(t[0], 1.0)
    emitted = got["tau"] + 1
    for j in range(k + 1):
        sel = emitted >= j + 1
        counts = np.bincount(got["tokens"][sel, j], minlength=V)
        exp = p[j] * sel.sum()
        keep = exp > 5
        assert scipy.stats.chisquare(counts[keep], exp[keep] * counts[keep].sum() / exp[keep].sum()).pvalue > 1e-4


def _noalloc(lib, w, ins, out):
    import ctypes
    from speculative_decoding_verification_68_gb300 import _native
    c = _native.load()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    B = ins[0].shape[0]
    dt = lib.SV_BF16 if w.dtype == si.BF16 else lib.SV_FP32
    return c.spec_verify_noalloc(B, w.k, w.vocab, dt, *[p(t) for t in ins], p(out["tokens"]), p(out["tau"]),
                                 p(out["p_draft"]), p(out["q_draft"]), p(out["tv"]),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_staged_and_plain_handles_coexist(lib):
    """The kernels' shared-memory limit is shared by every handle of the same
    shape: opening a handle with plain loads (SV_FLAG_NO_TMA) while a staging
    handle is live must not lower it under the live handle, nor under the
    allocation-free entry point's cached launch plan."""
    w = si.C3_T06.scaled(batch=6)
    b = si.generate(w)
    ins = to_dev(b)
    dt = torch.bfloat16
    staged = lib.SpecVerifier(6, w.k, w.vocab, dt)
    first = {k: t.cpu().numpy() for k, t in staged.verify(*ins, want_tv=True).items()}
    na = staged.alloc_outputs(6, want_pq=True, want_tv=True)
    assert _noalloc(lib, w, ins, na) == lib.SV_OK
    plain = lib.SpecVerifier(6, w.k, w.vocab, dt, lib.SV_FLAG_NO_TMA)
    again = staged.verify(*ins, want_tv=True)          # failed to launch when the limit was lowered
    p_out = plain.verify(*ins, want_tv=True)
    na2 = staged.alloc_outputs(6, want_pq=True, want_tv=True)
    assert _noalloc(lib, w, ins, na2) == lib.SV_OK
    torch.cuda.synchronize()
    for res in (again, p_out, na, na2):
        for key in first:
            assert np.array_equal(first[key], res[key].cpu().numpy()), key
    assert staged.get_error() == (lib.SV_OK, 0) and plain.get_error() == (lib.SV_OK, 0)
    staged.close()
    plain.close()


def test_concurrent_handles_on_streams(lib):
    """Three handles whose kernels may share SMs, launched on three streams without waiting for
    each other: V = 151,552 (256 tensor-memory columns per CTA), V = 262,144 (512 columns, one
    CTA per SM) and V = 20,000 (no tensor memory).  Each result is bit-identical to the same
    handle's result alone."""
    ws = [si.C3_T1.scaled(batch=48), si.Workload("conc_v262144", 16, 7, 262144, si.BF16, 2.0, draft_sigma=0.8,
                                                  temp_lo=1.0, temp_hi=1.0),
          si.Workload("conc_v20000", 64, 7, 20000, si.BF16, 2.0, draft_sigma=0.8, temp_lo=0.7, temp_hi=0.7)]
    handles, inputs, alone = [], [], []
    for w in ws:
        b = si.generate(w)
        v = lib.SpecVerifier(w.batch, w.k, w.vocab, torch.bfloat16)
        ins = to_dev(b)
        out = v.verify(*ins, want_tv=True)
        torch.cuda.synchronize()
        handles.append(v); inputs.append(ins); alone.append({k: t.cpu().numpy() for k, t in out.items()})
    streams = [torch.cuda.Stream() for _ in ws]
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        for v, ins, s in zip(handles, inputs, streams):
            outs.append(v.verify(*ins, want_tv=True, stream=s))
    torch.cuda.synchronize()
    for i, out in enumerate(outs):
        ref = alone[i % len(ws)]
        for key, t in out.items():
            assert np.array_equal(t.cpu().numpy(), ref[key], equal_nan=True), (ws[i % len(ws)].name, key)
    for v in handles:
        assert v.get_error()[0] == 0
        v.close()
