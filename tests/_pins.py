"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, written without the oracle's own formulas.

Each pin takes an ``oracle.Oracle`` (the real one, or a build with a planted
mistake) and raises AssertionError when the oracle disagrees with:
  - hand-worked examples (tests/golden/worked_examples.json);
  - library routines (scipy softmax / log_softmax, numpy argmax);
  - the acceptance identity sum_x q(x) P(accept | x) = sum_x min(p(x), q(x))
    = 1 - TV (page "Optimizing speculative decoding", section "Kimi K3");
  - target preservation: the emitted token at every position is distributed
    as the target row, measured exactly on the 2^-24 uniform lattice
    (same page, section "Rejection sampling and a loss that optimizes
    acceptance directly", first bullet);
  - greedy verification = argmax match (same bullet: greedy drafting).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special

import spec_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LATTICE = 1 << 24


def softmax_rows(z, T):
    z = np.asarray(z, np.float64)
    if T == 0:
        out = np.zeros_like(z)
        idx = np.argmax(z, axis=-1)
        np.put_along_axis(out, idx[..., None], 1.0, axis=-1)
        return out
    return scipy.special.softmax(z / T, axis=-1)


def _example_arrays(ex):
    if "target_probs" in ex:
        t = np.log(np.array(ex["target_probs"], np.float64)).astype(np.float32)
        d = np.log(np.array(ex["draft_probs"], np.float64)).astype(np.float32)
    else:
        t = np.array(ex["target_logits"], np.float32)
        d = np.array(ex["draft_logits"], np.float32)
    return t, d


def pin_worked_examples(orc):
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        exs = json.load(f)["examples"]
    for ex in exs:
        t, d = _example_arrays(ex)
        k = d.shape[0]
        r = orc.verify(t[None], d[None], np.array([ex["x"]], np.int32), np.array([ex["T"]], np.float32),
                       np.array([ex["u"]], np.float32), si.FP32, want_tv=True)
        assert r["tokens"][0].tolist() == ex["tokens"], (ex["name"], r["tokens"][0])
        assert int(r["tau"][0]) == ex["tau"], ex["name"]
        np.testing.assert_allclose(r["p_draft"][0], ex["p_draft"], atol=1e-6, err_msg=ex["name"])
        np.testing.assert_allclose(r["q_draft"][0], ex["q_draft"], atol=1e-6, err_msg=ex["name"])
        np.testing.assert_allclose(r["tv"][0], ex["tv"], atol=1e-6, err_msg=ex["name"])
        assert k == len(ex["x"])


def pin_softmax_library(orc):
    rng = np.random.default_rng(5)
    for V, T, s in ((16, 1.0, 2.0), (1000, 0.6, 3.0), (4096, 1.7, 0.5), (300, 0.3, 6.0)):
        z = rng.normal(0, s, V).astype(np.float32)
        lp, lse = orc.log_softmax(z, T)
        ref = scipy.special.log_softmax(z.astype(np.float64) / T)
        np.testing.assert_allclose(lp, ref, rtol=0, atol=1e-12)
        assert abs(lse - scipy.special.logsumexp(z.astype(np.float64) / T)) < 1e-12
    # closed form: constant logits c give lse = log V + c / T
    for V, c, T in ((7, 1.5, 1.0), (151552, -2.25, 0.6)):
        lp, lse = orc.log_softmax(np.full(V, c, np.float32), T)
        assert abs(lse - (np.log(V) + c / T)) < 1e-9
        assert np.allclose(lp, -np.log(V), atol=1e-12)
    # one dominant logit: p(max) = 1 / (1 + (V-1) e^{-delta/T})
    V, delta, T = 100, 12.0, 0.8
    z = np.zeros(V, np.float32)
    z[37] = delta
    p = orc.probs(z, T)
    assert abs(p[37] - 1.0 / (1.0 + (V - 1) * np.exp(-delta / T))) < 1e-14
    # bf16 rows convert exactly
    zb = si.f32_to_bf16(rng.normal(0, 2, 64).astype(np.float32))
    lpb, _ = orc.log_softmax(zb, 1.0, si.BF16)
    np.testing.assert_allclose(lpb, scipy.special.log_softmax(si.bf16_to_f32(zb).astype(np.float64)), atol=1e-12)


def pin_argmax_library(orc):
    rng = np.random.default_rng(9)
    for _ in range(50):
        z = rng.integers(-3, 4, 40).astype(np.float32)   # many exact ties
        assert orc.argmax(z) == int(np.argmax(z))       # numpy returns the first maximum
    zb = si.f32_to_bf16(np.array([0.5, 2.0, 2.0, 1.0], np.float32))
    assert orc.argmax(zb, si.BF16) == 1


def pin_tv_identities(orc):
    """TV = 1/2 sum|p - q| = sum max(0, p - q) = 1 - sum min(p, q), from scipy's softmax."""
    rng = np.random.default_rng(3)
    B, k, V = 6, 3, 512
    t = rng.normal(0, 2, (B, k + 1, V)).astype(np.float32)
    d = (t[:, :k] + rng.normal(0, 0.7, (B, k, V))).astype(np.float32)
    x = rng.integers(0, V, (B, k)).astype(np.int32)
    for T in (1.0, float(np.float32(0.6))):   # temperatures enter as fp32
        r = orc.verify(t, d, x, np.full(B, T, np.float32), np.full((B, k + 1), 0.5, np.float32), si.FP32)
        p = softmax_rows(t[:, :k], T)
        q = softmax_rows(d, T)
        np.testing.assert_allclose(r["tv"], 1.0 - np.minimum(p, q).sum(-1), atol=1e-12)
        np.testing.assert_allclose(r["tv"], np.maximum(p - q, 0).sum(-1), atol=1e-12)
        np.testing.assert_allclose(r["p_draft"], np.take_along_axis(p, x[..., None], -1)[..., 0], rtol=1e-12)
        np.testing.assert_allclose(r["q_draft"], np.take_along_axis(q, x[..., None], -1)[..., 0], rtol=1e-12)
    # identical rows: TV 0; disjoint one-hots (greedy, different argmax): TV 1
    r = orc.verify(t, t[:, :k].copy(), x, np.ones(B, np.float32), np.full((B, k + 1), 0.5, np.float32), si.FP32)
    assert np.all(np.abs(r["tv"]) < 1e-15)
    d2 = np.zeros_like(d)
    d2[..., 0] = 100.0
    t2 = np.zeros_like(t)
    t2[..., 1] = 100.0
    r = orc.verify(t2, d2, x, np.zeros(B, np.float32), np.full((B, k + 1), 0.5, np.float32), si.FP32)
    assert np.all(r["tv"] == 1.0)


def lattice_boundary(pred, n_queries: int) -> np.ndarray:
    """For monotone predicates (True below a threshold N*, False from N* on) over
    n in [0, 2^24], return N* per query by bisection.  pred(ns) -> bool array."""
    lo = np.zeros(n_queries, np.int64)          # pred(lo) True or lo == 0
    hi = np.full(n_queries, LATTICE, np.int64)  # first n with pred False is <= hi
    while True:
        active = hi > lo
        if not active.any():
            return lo
        mid = (lo + hi) // 2
        ok = pred(mid)
        lo = np.where(active & ok, mid + 1, lo)
        hi = np.where(active & ~ok, mid, hi)


def acceptance_masses(orc, lp, lq):
    """Exact lattice measure of {u : oracle accepts} for arrays of (log p, log q)."""
    lp = np.asarray(lp, np.float64).ravel()
    lq = np.asarray(lq, np.float64).ravel()

    def pred(ns):
        return np.array([orc.accept(a, b, n / LATTICE)[0] for a, b, n in zip(lp, lq, ns)])
    return lattice_boundary(pred, lp.size) / LATTICE


def pin_acceptance_is_overlap(orc):
    """sum_x q(x) P(accept | x) = sum_x min(p, q) = 1 - TV (exact, on the lattice)."""
    rng = np.random.default_rng(13)
    V = 12
    for T in (1.0, float(np.float32(0.7))):
        zt = rng.normal(0, 2, V).astype(np.float32)
        zd = (zt + rng.normal(0, 0.8, V)).astype(np.float32)
        p = softmax_rows(zt, T)
        q = softmax_rows(zd, T)
        lp, _ = orc.log_softmax(zt, T)
        lq, _ = orc.log_softmax(zd, T)
        A = acceptance_masses(orc, lp, lq)
        # lattice measure is within one lattice step of min(1, p/q)
        np.testing.assert_allclose(A, np.minimum(1.0, p / q), atol=1.0 / LATTICE + 1e-12)
        assert abs((q * A).sum() - np.minimum(p, q).sum()) < 2.0 / LATTICE
        assert abs((q * A).sum() - (1.0 - 0.5 * np.abs(p - q).sum())) < 2.0 / LATTICE


def _tiny_rows(seed=0, T=1.0):
    w = si.TINY if seed == 0 else si.TINY.scaled(seed=seed)
    b = si.generate(w)
    return b.target[0], b.draft[0], w


def pin_target_preservation_exact(orc, seed=0):
    """Exact output distribution of the chain driver on the tiny workload
    (V = 16, k = 3): for every draft tuple x (16^3, weight prod q_i(x_i)), the
    accept decisions and the final draw are measured on the 2^-24 uniform
    lattice by bisection over the oracle's own verify call.  Then
        P(y_j = a, n >= j) = p_j(a) * prod_{i<j} (1 - TV_i)   for j = 1..k+1
    (the emitted token at each position follows the target; n = tau + 1)."""
    t, d, w = _tiny_rows(seed)
    k, V, T = w.k, w.vocab, 1.0
    p = softmax_rows(t, T)          # [k+1, V]
    q = softmax_rows(d, T)          # [k, V]
    tv = 0.5 * np.abs(p[:k] - q).sum(-1)

    tuples = np.stack(np.meshgrid(*[np.arange(V)] * k, indexing="ij"), -1).reshape(-1, k).astype(np.int32)
    nT = tuples.shape[0]

    def run(x, u):
        n = x.shape[0]
        return orc.verify(np.broadcast_to(t, (n,) + t.shape), np.broadcast_to(d, (n,) + d.shape), x,
                          np.full(n, T, np.float32), u, si.FP32, want_tv=False, nthreads=8)

    # A[tuple, i]: lattice measure of acceptance at position i, earlier positions
    # accepted with u = 0 (p > 0 everywhere at T = 1), later uniforms arbitrary.
    A = np.zeros((nT, k))
    for i in range(k):
        def pred(ns, i=i):
            u = np.zeros((nT, k + 1), np.float32)
            u[:, i] = ns / LATTICE
            return run(tuples, u)["tau"] > i
        A[:, i] = lattice_boundary(pred, nT) / LATTICE

    # R[i, xi, a]: final-token distribution after a rejection at position i
    # with rejected draft xi (only where a rejection is possible: p_i(xi) < q_i(xi)).
    # Bonus[a]: final-token distribution when every draft is accepted.
    def final_token_dist(x_rows, u_fixed, pos):
        n = x_rows.shape[0]
        bounds = np.zeros((n, V + 1), np.int64)
        bounds[:, V] = LATTICE
        for a in range(1, V):
            def pred(ns, a=a):
                u = u_fixed.copy()
                u[:, k] = ns / LATTICE
                return run(x_rows, u)["tokens"][np.arange(n), pos] < a
            bounds[:, a] = lattice_boundary(pred, n)
        return np.diff(bounds, axis=1) / LATTICE

    R = np.zeros((k, V, V))
    for i in range(k):
        rej = np.nonzero(p[i] < q[i])[0]
        if rej.size == 0:
            continue
        x_rows = np.zeros((rej.size, k), np.int32)
        x_rows[:, i] = rej
        u_fixed = np.zeros((rej.size, k + 1), np.float32)
        u_fixed[:, i] = (LATTICE - 1) / LATTICE          # reject at i (p/q < 1 - 2^-24 there)
        assert np.all(run(x_rows, u_fixed)["tau"] == i)
        R[i, rej] = final_token_dist(x_rows, u_fixed, i)
    bonus = final_token_dist(np.zeros((1, k), np.int32), np.zeros((1, k + 1), np.float32), k)[0]

    wq = np.prod(q[np.arange(k), tuples], axis=1)       # weight of each tuple
    reach = np.ones(nT)
    for j in range(k):
        xj = tuples[:, j]
        emit = np.zeros((nT, V))
        emit[np.arange(nT), xj] += A[:, j]
        emit += (1.0 - A[:, j])[:, None] * R[j, xj]
        got = (wq[:, None] * reach[:, None] * emit).sum(0)
        want = p[j] * np.prod(1.0 - tv[:j])
        np.testing.assert_allclose(got, want, atol=4e-6, err_msg=f"position {j + 1}")
        # P(n = j+1) = prod_{i<j}(1 - TV_i) * TV_j
        p_stop = (wq * reach * (1.0 - A[:, j])).sum()
        assert abs(p_stop - np.prod(1.0 - tv[:j]) * tv[j]) < 4e-6
        reach = reach * A[:, j]
    got = (wq * reach).sum() * bonus
    np.testing.assert_allclose(got, p[k] * np.prod(1.0 - tv), atol=4e-6, err_msg="bonus position")


def pin_greedy_is_argmax_match(orc):
    rng = np.random.default_rng(21)
    B, k, V = 40, 5, 64
    t = rng.integers(-4, 5, (B, k + 1, V)).astype(np.float32)   # frequent ties
    d = rng.integers(-4, 5, (B, k, V)).astype(np.float32)
    am_t = np.argmax(t, -1)
    am_d = np.argmax(d, -1)
    # drafts: the draft argmax, except that some chains copy the target argmax
    x = am_d.copy()
    copy = rng.random((B, k)) < 0.7
    x[copy] = am_t[:, :k][copy]
    x = x.astype(np.int32)
    r = orc.verify(t, d, x, np.zeros(B, np.float32), rng.random((B, k + 1)).astype(np.float32), si.FP32)
    match = x == am_t[:, :k]
    tau = np.where(match.all(1), k, np.argmin(match, 1))
    assert np.array_equal(r["tau"], tau)
    for b in range(B):
        assert r["tokens"][b, :tau[b]].tolist() == x[b, :tau[b]].tolist()
        assert r["tokens"][b, tau[b]] == am_t[b, tau[b]]
        assert np.all(r["tokens"][b, tau[b] + 1:] == -1)
    assert np.array_equal(r["tv"], (am_t[:, :k] != am_d).astype(np.float64))


def pin_inverse_cdf_library(orc):
    """Final draw = first index whose inclusive cumulative weight exceeds u*S
    (numpy searchsorted, side='right'); zero-weight tokens are never drawn."""
    rng = np.random.default_rng(17)
    for _ in range(200):
        V = int(rng.integers(1, 40))
        w = rng.random(V) * (rng.random(V) < 0.6)
        if w.sum() == 0:
            w[rng.integers(V)] = 0.5
        u = float(rng.integers(0, LATTICE)) / LATTICE
        y, _, S = orc.sample(w, u)
        c = np.cumsum(w)
        assert abs(S - c[-1]) < 1e-12
        assert y == int(np.searchsorted(c, u * c[-1], side="right")), (w, u, y)
        assert w[y] > 0
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    assert orc.sample(w, 0.25)[0] == 3        # exactly on C_1: strict inequality moves past it
    assert orc.sample(w, 0.0)[0] == 1         # the first positive weight, not index 0


def pin_entropy_closed_forms(orc):
    """Entropy of rows whose distribution is known in closed form: a constant
    row is uniform (H = ln V); a row with n_a logits a and n_b logits b has two
    probability levels; -inf logits are masked out; T == 0 gives 0."""
    for V in (1, 2, 16, 1000, 151552):
        for T in (0.3, 1.0, 2.5):
            h = orc.entropy(np.full(V, 1.25, np.float32), T)
            # fp64 sum of V equal terms: rounding grows like V * eps
            assert abs(h - math.log(V)) <= 1e-15 * V * max(1.0, math.log(V)), (V, T, h)
    for n_a, n_b, a, b, T in ((1, 15, 3.0, 0.0, 1.0), (5, 995, 2.0, -1.0, 0.7), (100, 100, 0.0, -4.0, 2.0),
                              (1, 4095, 9.0, 0.0, 0.6)):
        z = np.concatenate([np.full(n_a, a), np.full(n_b, b)]).astype(np.float32)
        ea, eb = math.exp(a / T), math.exp(b / T)
        pa, pb = ea / (n_a * ea + n_b * eb), eb / (n_a * ea + n_b * eb)
        want = -(n_a * pa * math.log(pa) + n_b * pb * math.log(pb))
        assert abs(orc.entropy(z, T) - want) <= 1e-12, (n_a, n_b, a, b, T)
        masked = np.concatenate([z, np.full(37, -np.inf, np.float32)])
        assert abs(orc.entropy(masked, T) - want) <= 1e-12
    assert orc.entropy(np.array([0.0, 3.0, 3.0], np.float32), 0.0) == 0.0
    assert math.isnan(orc.entropy(np.array([0.0, np.nan], np.float32), 1.0))
    assert math.isnan(orc.entropy(np.array([0.0, 1.0], np.float32), -1.0))


def pin_entropy_library(orc):
    """H = scipy.stats.entropy of scipy's softmax(z / T), on random rows (fp32 and
    bf16 storage); 0 <= H <= ln V, and H grows with T."""
    import scipy.special
    import scipy.stats
    rng = np.random.default_rng(17)
    for V, T, s in ((16, 1.0, 2.0), (1000, 0.6, 3.0), (4096, 1.7, 0.5), (30000, 1.0, 4.0)):
        z = (rng.standard_normal(V) * s).astype(np.float32)
        want = scipy.stats.entropy(scipy.special.softmax(z.astype(np.float64) / T))
        got = orc.entropy(z, T)
        assert abs(got - want) <= 1e-11 * max(1.0, want), (V, T, got, want)
        assert 0.0 <= got <= math.log(V) + 1e-12
        assert orc.entropy(z, 0.5 * T) < got < orc.entropy(z, 2.0 * T)
        zb = z.view(np.uint32) >> 16 << 16        # a bf16 row: the oracle reads the high half
        bf = (zb >> 16).astype(np.uint16)
        want_b = scipy.stats.entropy(scipy.special.softmax(zb.view(np.float32).astype(np.float64) / T))
        assert abs(orc.entropy(bf, T, dtype=1) - want_b) <= 1e-11 * max(1.0, want_b)


def pin_overlap_loss_values(orc):
    """alpha = sum min(p, q) = 1 - TV with TV = 1/2 sum |p - q| from scipy's
    softmax; TV loss = 1 - alpha, overlap loss = -ln alpha; identical rows give
    alpha = 1, both losses 0 and a zero gradient; invalid rows give NaN."""
    import scipy.special
    rng = np.random.default_rng(31)
    for V, T in ((16, 1.0), (700, 0.6), (5000, 1.4)):
        zt = (rng.standard_normal(V) * 2).astype(np.float32)
        zd = (rng.standard_normal(V) * 2).astype(np.float32)
        p = scipy.special.softmax(zt.astype(np.float64) / T)
        q = scipy.special.softmax(zd.astype(np.float64) / T)
        tv = 0.5 * np.abs(p - q).sum()
        l0, a0, _, _ = orc.overlap_grad(zt, zd, T, 0)
        l1, a1, _, _ = orc.overlap_grad(zt, zd, T, 1)
        assert abs(a0 - (1.0 - tv)) <= 1e-12 and a0 == a1
        assert abs(l0 - tv) <= 1e-12 and abs(l1 + math.log(1.0 - tv)) <= 1e-12
        l, a, g, _ = orc.overlap_grad(zt, zt, T, 1)
        assert abs(a - 1.0) <= 1e-12 and abs(l) <= 1e-12 and not np.any(g)
    l, a, g, _ = orc.overlap_grad(np.array([0.0, np.nan], np.float32), np.zeros(2, np.float32), 1.0, 0)
    assert math.isnan(l) and not np.any(g)
    l, a, g, _ = orc.overlap_grad(np.zeros(3, np.float32), np.ones(3, np.float32), 0.0, 0)
    assert math.isnan(l) and not np.any(g)


def pin_overlap_gradient_finite_differences(orc):
    """The gradient against central differences of the loss in every draft
    logit (fp64 rows, away from p == q ties); it sums to zero over the row
    (softmax invariance to a constant shift); scaling the weight scales it."""
    rng = np.random.default_rng(37)
    for kind in (0, 1):
        for V, T in ((8, 1.0), (40, 0.7), (200, 1.6)):
            zt = rng.standard_normal(V) * 1.5
            zd = rng.standard_normal(V) * 1.5
            loss, alpha, g, tie = orc.overlap_grad(zt, zd, T, kind, 1.0, dtype=2)
            assert tie == 0.0
            h = 1e-6
            for m in range(V):
                zp, zm = zd.copy(), zd.copy()
                zp[m] += h
                zm[m] -= h
                fd = (orc.overlap_grad(zt, zp, T, kind, 1.0, dtype=2)[0] - orc.overlap_grad(zt, zm, T, kind, 1.0, dtype=2)[0]) / (2 * h)
                assert abs(fd - g[m]) <= 1e-6 * max(1.0, abs(g[m])), (kind, V, m, fd, g[m])
            assert abs(g.sum()) <= 1e-12 * max(1.0, np.abs(g).sum())
            _, _, g3, _ = orc.overlap_grad(zt, zd, T, kind, 3.0, dtype=2)
            assert np.allclose(g3, 3.0 * g, rtol=1e-14, atol=0)


def pin_tie_band(orc):
    """The tie flags mark exactly the decisions within 1e-6 of their threshold:
    an accept test with |u - p(x)/q(x)| < 1e-6, and a final draw with u*S within
    1e-6*S of the chosen CDF boundary or the one below it.  The thresholds are
    computed here from scipy's softmax and numpy's cumulative sum.  Greedy
    decisions are never flagged."""
    import scipy.special
    zt = np.array([0.3, -1.0, 0.8, 0.1, -0.4, 0.0], np.float32)   # target row 0
    zd = np.array([0.9, -0.2, 0.1, 0.4, -0.4, 0.0], np.float32)   # draft row 0
    zb = np.array([0.5, 0.2, -0.3, 1.1, 0.0, -2.0], np.float32)   # bonus row
    T = np.float32(1.0)
    p = scipy.special.softmax(zt.astype(np.float64))
    q = scipy.special.softmax(zd.astype(np.float64))
    ratio = p[0] / q[0]
    assert ratio < 0.9
    w = np.maximum(p - q, 0.0)
    C = np.cumsum(w)
    S = C[-1]

    def run(u0, u1, temp=T):
        target = np.stack([zt, zb])[None]
        out = orc.verify(target, zd[None, None], np.array([[0]], np.int32), np.array([temp], np.float32),
                         np.array([[u0, u1]], np.float32), 0)
        return out

    # accept tests: flagged inside the band, not outside; the decision itself follows u < ratio
    for d, flagged in ((-3e-7, True), (3e-7, True), (-5e-6, False), (5e-6, False)):
        out = run(np.float32(ratio + d), np.float32(0.5))
        assert bool(out["accept_tie"][0, 0]) == flagged, (d, out["accept_tie"])
        assert (out["tau"][0] == 1) == (np.float32(ratio + d) < ratio)
    # final draws after a rejection: u1 close to each inner boundary C_j / S
    for j in range(len(C) - 1):
        if w[j] == 0.0 or w[j + 1:].sum() == 0.0:
            continue
        for d, flagged in ((-3e-7, True), (3e-7, True), (-5e-6, False), (5e-6, False)):
            u1 = np.float32(C[j] / S + d)
            out = run(np.float32(0.999), u1)
            assert out["tau"][0] == 0
            assert bool(out["cdf_tie"][0]) == flagged, (j, d, out["cdf_tie"])
            want = int(np.searchsorted(C, float(u1) * S, side="right"))
            assert out["tokens"][0, 0] == want
    # greedy: exact decisions, never flagged
    out = run(np.float32(ratio), np.float32(C[0] / S), temp=np.float32(0.0))
    assert out["accept_tie"][0, 0] == 0 and out["cdf_tie"][0] == 0


def _padded_rows(rng, rows, pad, V, scale, dtype):
    """[rows, V] logits that are the head of a larger buffer with `pad` extra
    random rows behind them, so that a batch driver that mis-strides a row
    still reads inside the allocation (the pins then see wrong values, not a
    crash).  fp32 or bf16 storage (bf16: the high half of the fp32 bits)."""
    z = (rng.standard_normal((rows + pad, V)) * scale).astype(np.float32)
    if dtype == si.BF16:
        z = (z.view(np.uint32) >> 16).astype(np.uint16)
    return z, z[:rows]


def _row_values(z, dtype):
    """fp64 logit values of stored rows (bf16 bits widened exactly)."""
    if dtype == si.BF16:
        return (z.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return z.astype(np.float64)


def pin_batch_drivers(orc):
    """The batch drivers of the entropy and the overlap losses map chain b,
    position i to target row b*(k+1)+i, draft row b*k+i, the chain's
    temperature T[b] and the weight w[b, i].  Checked per row against scipy's
    softmax / entropy (independent of the oracle), against the single-row
    functions on explicitly indexed rows (bit-equal), and, for the weights,
    by the gradient's linearity in w[b, i] (page "Optimizing speculative
    decoding", sections "Kimi K3" and "Rejection sampling and a loss that
    optimizes acceptance directly")."""
    import scipy.special
    import scipy.stats
    rng = np.random.default_rng(41)
    B, k, V = 4, 3, 24
    T = np.array([0.7, 0.0, 1.3, 1.0], np.float32)        # chain 1 greedy
    w = rng.uniform(0.5, 2.0, (B, k)).astype(np.float32)   # distinct weights per (b, i)
    for dtype in (si.FP32, si.BF16):
        big_t, t2 = _padded_rows(rng, B * (k + 1), B * (k + 1), V, 2.0, dtype)
        big_d, d2 = _padded_rows(rng, B * k, B * (k + 1), V, 2.0, dtype)
        nan_bits = np.float32(np.nan).view(np.uint32) >> 16 if dtype == si.BF16 else np.float32(np.nan)
        t2[3 * (k + 1) + 1, 5] = nan_bits                  # chain 3: target row 1 is invalid
        target, draft = t2.reshape(B, k + 1, V), d2.reshape(B, k, V)
        tv, dv = _row_values(target, dtype), _row_values(draft, dtype)

        # ---- entropies
        ent_t, ent_d = orc.entropy_batch(target, draft, T, dtype)
        assert ent_t.shape == (B, k + 1) and ent_d.shape == (B, k)
        for b in range(B):
            for rows, vals, ent in ((target, tv, ent_t), (draft, dv, ent_d)):
                for i in range(rows.shape[1]):
                    one = orc.entropy(rows[b, i], float(T[b]), dtype=dtype)
                    got = ent[b, i]
                    assert (math.isnan(one) and math.isnan(got)) or one == got, (dtype, b, i, got, one)
                    if np.isnan(vals[b, i]).any():
                        assert math.isnan(got), (b, i)
                    elif T[b] == 0:
                        assert got == 0.0
                    else:
                        want = scipy.stats.entropy(scipy.special.softmax(vals[b, i] / float(T[b])))
                        assert abs(got - want) <= 1e-11 * max(1.0, want), (dtype, b, i, got, want)

        # ---- losses, overlaps and gradients
        for kind in (0, 1):
            r = orc.overlap_grad_batch(target, draft, T, kind, w, dtype)
            r1 = orc.overlap_grad_batch(target, draft, T, kind, None, dtype)
            for b in range(B):
                for i in range(k):
                    loss, alpha, g, tie = orc.overlap_grad(target[b, i], draft[b, i], float(T[b]), kind,
                                                           float(w[b, i]), dtype=dtype)
                    for name, one in (("loss", loss), ("alpha", alpha), ("tie", tie)):
                        got = r[name][b, i]
                        assert (math.isnan(one) and math.isnan(got)) or one == got, (name, dtype, kind, b, i)
                    assert np.array_equal(r["grad"][b, i], g), (dtype, kind, b, i)
                    invalid = T[b] <= 0 or np.isnan(tv[b, i]).any()
                    if invalid:
                        assert math.isnan(r["loss"][b, i]) and not np.any(r["grad"][b, i])
                        continue
                    p = scipy.special.softmax(tv[b, i] / float(T[b]))
                    q = scipy.special.softmax(dv[b, i] / float(T[b]))
                    a = float(np.minimum(p, q).sum())
                    assert abs(r["alpha"][b, i] - a) <= 1e-12, (dtype, kind, b, i)
                    want = 1.0 - a if kind == 0 else -math.log(a)
                    assert abs(r["loss"][b, i] - want) <= 1e-12 * max(1.0, abs(want))
                    # the weight enters the gradient linearly, and only its own position's
                    g1 = r1["grad"][b, i] * float(w[b, i])
                    assert np.allclose(r["grad"][b, i], g1, rtol=1e-14, atol=1e-300), (dtype, kind, b, i)
                    assert np.any(r["grad"][b, i])


ALL_PINS = [pin_worked_examples, pin_tie_band, pin_inverse_cdf_library, pin_softmax_library, pin_argmax_library, pin_tv_identities,
            pin_acceptance_is_overlap, pin_greedy_is_argmax_match, pin_target_preservation_exact,
            pin_entropy_closed_forms, pin_entropy_library, pin_overlap_loss_values,
            pin_overlap_gradient_finite_differences, pin_batch_drivers]
