"""Seeded input generator: Philox known answers, lattice uniforms, bf16 rounding,
determinism, and the distributions the workloads ask for."""
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import spec_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(t, 16) for t in line.split()])
    assert len(rows) == 3
    for r in rows:
        out = si.philox4x32_10(r[0:4], r[4:6])
        assert out.tolist() == r[6:10]


def test_uniforms_on_lattice():
    u = si.uniforms(7, si.STREAM_VERIFY, 0, 64, 33)
    assert u.min() >= 0.0 and u.max() < 1.0
    n = u.astype(np.float64) * 2 ** 24
    assert np.all(n == np.floor(n))
    # counter-based: any row can be generated on its own
    assert np.array_equal(si.uniforms(7, si.STREAM_VERIFY, 10, 1, 33)[0], u[10])
    assert si.uniform(7, si.STREAM_VERIFY, 3, 5) == u[3, 5]
    # loose uniformity check (KS)
    assert scipy.stats.kstest(u.ravel(), "uniform").pvalue > 1e-4


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 3, 4000), rng.normal(0, 1e-3, 500), rng.normal(0, 1e4, 500)]).astype(np.float32)
    # exact ties between two bf16 neighbours round to even
    ties = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(2.0 + 2 ** -7)], np.float32)
    x = np.concatenate([x, ties])
    ours = si.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(si.bf16_to_f32(ours[-3:]), np.array([1.0, 1.0 + 2 ** -6, -2.0], np.float32))


def test_generation_deterministic_and_thread_independent():
    w = si.C3_T1.scaled(batch=3, vocab=4096)
    a = si.generate(w, nthreads=1)
    b = si.generate(w, nthreads=3)
    for f in ("target", "draft", "tokens", "temperature", "uniforms"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    # a sub-range of chains equals the same chains of the full batch
    c = si.generate(w, b0=1, nb=2)
    assert np.array_equal(c.target, a.target[1:]) and np.array_equal(c.tokens, a.tokens[1:])


def test_workload_distributions():
    w = si.C3_T1.scaled(batch=2, vocab=151552)
    b = si.generate(w)
    t = si.bf16_to_f32(b.target).astype(np.float64)
    d = si.bf16_to_f32(b.draft).astype(np.float64)
    # 20 distinct boosted ids per target row, +8 on an N(0, 3^2) background
    for row in t.reshape(-1, w.vocab):
        big = np.sort(row)[-20:]
        assert big.min() > 8.0 - 1.0
    q1, q3 = np.percentile(t, [25, 75])
    assert abs(np.median(t)) < 0.05 and abs((q3 - q1) / 1.3489795 - 3.0) < 0.05
    # draft = target + N(0, 1)
    noise = d - t[:, :w.k]
    assert abs(noise.mean()) < 0.01 and abs(noise.std() - 1.0) < 0.02
    # config with per-chain temperatures in [0.3, 1.2] and two regimes
    w4 = si.C4.scaled(batch=8, vocab=2048)
    b4 = si.generate(w4)
    assert np.all((b4.temperature >= 0.3) & (b4.temperature <= 1.2))
    t4 = si.bf16_to_f32(b4.target).astype(np.float64)
    assert abs(t4[:4].std() - 6.0) < 0.3 and abs(t4[4:].std() - 0.5) < 0.03
    # independent drafts
    w5 = si.C5.scaled(batch=2, vocab=8192)
    b5 = si.generate(w5)
    t5 = si.bf16_to_f32(b5.target)[:, :w5.k].astype(np.float64).ravel()
    d5 = si.bf16_to_f32(b5.draft).astype(np.float64).ravel()
    assert abs(np.corrcoef(t5, d5)[0, 1]) < 0.02 and abs(d5.std() - 2.0) < 0.05


def test_gumbel_draft_sampling_follows_softmax():
    """Draft tokens drawn with Gumbel-max follow softmax(z/T) (chi-squared, scipy softmax)."""
    rng = np.random.default_rng(1)
    z = rng.normal(0, 1.5, 8).astype(np.float32)
    n = 60000
    for T in (1.0, 0.5):
        zz = np.broadcast_to(z, (n, 8)).copy()
        toks = si.gumbel_argmax(11, zz, si.FP32, np.full(n, T, np.float32))
        counts = np.bincount(toks, minlength=8)
        p = scipy.special.softmax(z.astype(np.float64) / T)
        assert scipy.stats.chisquare(counts, p * n).pvalue > 1e-4
    toks0 = si.gumbel_argmax(11, np.array([[1, 3, 3, 2]], np.float32), si.FP32, np.zeros(1, np.float32))
    assert toks0[0] == 1
