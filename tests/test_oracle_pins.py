"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest
import scipy.stats

import spec_inputs as si
from tests import _pins


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle, pin):
    pin(oracle)


def test_target_preservation_exact_second_seed(oracle):
    _pins.pin_target_preservation_exact(oracle, seed=3)


def _replicated_tiny(n, seed, same_rows=False):
    """n chains that share the tiny workload's rows but draw their own drafts
    (Gumbel-max from q, distinct Philox rows) and their own uniforms."""
    b = si.generate(si.TINY)
    t = np.ascontiguousarray(np.broadcast_to(b.target[0], (n,) + b.target[0].shape))
    d = t[:, :si.TINY.k].copy() if same_rows else np.ascontiguousarray(np.broadcast_to(b.draft[0], (n,) + b.draft[0].shape))
    x = si.gumbel_argmax(seed, d, si.FP32, np.ones(n * si.TINY.k, np.float32)).astype(np.int32)
    u = si.uniforms(seed, si.STREAM_VERIFY, 0, n, si.TINY.k + 1)
    return t, d, x, u


def test_target_preservation_sampled(oracle):
    """200,000 chains: the token emitted at each position, given that the chain
    reached it, is distributed as the target row (chi-squared, p > 1e-4)."""
    n = 200_000
    t, d, x, u = _replicated_tiny(n, seed=101)
    r = oracle.verify(t, d, x, np.ones(n, np.float32), u, si.FP32, nthreads=8)
    k, V = si.TINY.k, si.TINY.vocab
    p = _pins.softmax_rows(t[0], 1.0)
    q = _pins.softmax_rows(d[0], 1.0)
    tv = 0.5 * np.abs(p[:k] - q).sum(-1)
    emitted = r["tau"] + 1
    for j in range(k + 1):
        sel = emitted >= j + 1
        counts = np.bincount(r["tokens"][sel, j], minlength=V)
        expected = p[j] * sel.sum()
        keep = expected > 5
        stat = scipy.stats.chisquare(counts[keep], expected[keep] * counts[keep].sum() / expected[keep].sum())
        assert stat.pvalue > 1e-4, (j, stat)
    # accepted-length distribution: P(tau = i) = prod_{m<i}(1 - TV_m) TV_i, P(tau = k) = prod(1 - TV)
    probs = [np.prod(1 - tv[:i]) * tv[i] for i in range(k)] + [np.prod(1 - tv)]
    counts = np.bincount(r["tau"], minlength=k + 1)
    assert scipy.stats.chisquare(counts, np.array(probs) * n).pvalue > 1e-4


def test_identical_rows_accept_everything(oracle):
    """p == q: every draft accepted (tau = k) and the bonus follows the last target row."""
    n = 100_000
    t, d, x, u = _replicated_tiny(n, seed=202, same_rows=True)
    r = oracle.verify(t, d, x, np.ones(n, np.float32), u, si.FP32, nthreads=8)
    k, V = si.TINY.k, si.TINY.vocab
    assert np.all(r["tau"] == k)
    assert np.array_equal(r["tokens"][:, :k], x)
    p = _pins.softmax_rows(t[0, k], 1.0)
    counts = np.bincount(r["tokens"][:, k], minlength=V)
    keep = p * n > 5
    assert scipy.stats.chisquare(counts[keep], p[keep] * counts[keep].sum() / p[keep].sum()).pvalue > 1e-4
    # also on a bf16 vocabulary-scale workload at two temperatures
    w = si.C3_T06.scaled(batch=4, vocab=20000)
    b = si.generate(w)
    for T in (0.6, 1.0):
        r = oracle.verify(b.target, b.target[:, :w.k].copy(), b.tokens, np.full(4, T, np.float32), b.uniforms,
                          si.BF16, nthreads=4)
        assert np.all(r["tau"] == w.k) and np.all(r["tv"] == 0.0)


def test_acceptance_frequency_monte_carlo(oracle):
    """Position-1 acceptance frequency over many chains equals mean(1 - TV_1) within 5 sigma."""
    w = si.C2.scaled(batch=20000, vocab=256)
    b = si.generate(w)
    r = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, si.FP32, nthreads=8)
    p = _pins.softmax_rows(b.target[:, 0], 1.0)
    q = _pins.softmax_rows(b.draft[:, 0], 1.0)
    beta = np.minimum(p, q).sum(-1)
    acc = (r["tau"] >= 1).astype(np.float64)
    sigma = np.sqrt((beta * (1 - beta)).sum()) / w.batch
    assert abs(acc.mean() - beta.mean()) < 5 * sigma


def test_tie_flags(oracle):
    lp, lq = np.log(0.3), np.log(0.6)           # threshold 0.5
    assert oracle.accept(lp, lq, 0.5 - 5e-7) == (True, True)
    assert oracle.accept(lp, lq, 0.5 + 5e-7) == (False, True)
    assert oracle.accept(lp, lq, 0.5 - 2e-6) == (True, False)
    assert oracle.accept(lp, lq, 0.5 + 2e-6) == (False, False)
    assert oracle.accept(lq, lq, 1.0 - 2 ** -24) == (True, True)   # p == q: threshold 1
    assert oracle.accept(lq, lq, 0.5) == (True, False)
    assert oracle.accept(-np.inf, lq, 0.0) == (False, False)       # p(x) = 0: exact
    assert oracle.accept(0.0, -np.inf, 0.9) == (True, False)       # q(x) = 0 < p(x)
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    assert oracle.sample(w, 0.2) == (1, False, 1.0)
    assert oracle.sample(w, 0.25 - 4e-7)[1] is True                # just below C_1 = 0.25
    y, tie, _ = oracle.sample(w, 0.25)
    assert y == 3 and tie                                           # exactly on a boundary: strict <
    assert oracle.sample(w, 0.9999)[0] == 4
    assert oracle.sample(np.zeros(4), 0.3)[0] == -1


def test_invalid_chains(oracle):
    w = si.TINY
    b = si.generate(w)
    base = dict(target=b.target, draft=b.draft, tokens=b.tokens, temperature=b.temperature, uniforms=b.uniforms)

    def run(**kw):
        a = dict(base, **kw)
        return oracle.verify(a["target"], a["draft"], a["tokens"], a["temperature"], a["uniforms"], si.FP32)

    good = run()
    assert good["tau"][0] >= 0
    for bad in (dict(tokens=np.array([[0, -1, 2]], np.int32)), dict(tokens=np.array([[0, 16, 2]], np.int32)),
                dict(temperature=np.array([-1.0], np.float32)), dict(temperature=np.array([np.nan], np.float32)),
                dict(temperature=np.array([np.inf], np.float32))):
        r = run(**bad)
        assert r["tau"][0] == -1 and np.all(r["tokens"][0] == -1), bad
    for val in (np.nan, np.inf):
        t = b.target.copy()
        t[0, 3, 5] = val                                   # the bonus row
        r = run(target=t)
        assert r["tau"][0] == -1
    d = b.draft.copy()
    d[0, 1, :] = -np.inf                                   # a row with no finite logit
    assert run(draft=d)["tau"][0] == -1
    d = b.draft.copy()
    d[0, 1, 3] = -np.inf                                   # -inf entries are masked tokens: valid
    assert run(draft=d)["tau"][0] >= 0
