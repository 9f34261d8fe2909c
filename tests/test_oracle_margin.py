"""Pins of the oracle's margin confidence, scaled logits and greedy argmax
beside a sample (orc_token_stats_ex).

Worked examples (tests/golden), brute force through the probability vector
on tiny rows (the runner-up found as the largest probability at another id,
not as a logit), invariants, and the categorical sampler of the uniform-noise
loop checked statistically against softmax of the scaled logits.  CPU only.
"""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle


def test_margin_worked_examples(golden):
    for ex in golden["token_stats_margin"]:
        z = np.asarray([ex["logits"]], dtype=np.float32)
        x0, p, h, mar, am = oracle.token_stats_ex(z, logit_scale=ex["logit_scale"], suppress_ids=ex["suppress_ids"])
        assert x0[0] == ex["x0"] and am[0] == ex["argmax"], ex["cite"]
        # the fp32 rounding of the logits moves the values by ~1e-8
        assert p[0] == pytest.approx(ex["prob"], rel=1e-7, abs=1e-12), ex["cite"]
        assert mar[0] == pytest.approx(ex["margin"], rel=1e-7, abs=1e-12), ex["cite"]
        assert h[0] == pytest.approx(ex["entropy"], rel=1e-7, abs=1e-12), ex["cite"]


def _sanitised(z):
    """The reading of a logit: NaN carries no mass (-inf); every other value is itself."""
    z = np.asarray(z, dtype=np.float32).copy()
    z[np.isnan(z)] = -np.inf
    return z


def _brute(z, s, sup):
    """x0, prob, margin, argmax of one row from its probability vector."""
    V = z.size
    A = [v for v in range(V) if v not in sup]
    with np.errstate(over="ignore", invalid="ignore"):
        zs = _sanitised(z) * np.float32(s)          # one fp32 multiplication per logit (may overflow to inf)
    zs[np.isinf(zs) & (zs < 0)] = -np.inf
    za = zs[A].astype(np.float64)
    if np.all(za == -np.inf):
        p = np.full(len(A), 1.0 / len(A))
    elif za.max() == np.inf:
        p = (za == np.inf) / np.count_nonzero(za == np.inf)   # the +inf entries share the mass
    else:
        p = np.exp(za - za.max())
        p /= p.sum()
    best = max(za)
    i0 = next(i for i, v in enumerate(za) if v == best)
    others = [p[i] for i in range(len(A)) if i != i0]
    margin = p[i0] - (max(others) if others else 0.0)
    return A[i0], p[i0], margin


def test_margin_bruteforce_tiny_rows():
    rng = np.random.default_rng(2024)
    specials = [np.nan, np.inf, -np.inf, np.float32(2.0**101), np.float32(-2.0**105), np.float32(3e38),
                np.float32(-1e31)]
    for trial in range(400):
        V = int(rng.integers(1, 9))
        if trial % 3 == 0:
            z = rng.integers(-2, 3, size=V).astype(np.float32)   # many exact ties
        else:
            z = (rng.standard_normal(V) * 3).astype(np.float32)
        if trial % 5 == 0:
            z[rng.integers(0, V)] = specials[trial % len(specials)]
        sup = set(int(v) for v in rng.choice(V, size=int(rng.integers(0, V)), replace=False))
        s = float(rng.choice([1.0, 0.5, 1.25, 2.5, 3.0, 1 / 0.7]))
        x0e, pe, me = _brute(z, s, sup)
        x0, p, h, mar, am = oracle.token_stats_ex(z[None], logit_scale=s, suppress_ids=sorted(sup))
        assert x0[0] == x0e and am[0] == x0e, (z, s, sup)
        assert p[0] == pytest.approx(pe, rel=1e-12, abs=1e-15), (z, s, sup)
        assert mar[0] == pytest.approx(me, rel=1e-12, abs=1e-15), (z, s, sup)


def test_margin_invariants_and_unit_scale():
    rng = np.random.default_rng(7)
    z = (rng.standard_normal((64, 300)) * 2.5).astype(np.float32)
    x0, p, h, mar, am = oracle.token_stats_ex(z)
    y0, q, g = oracle.token_stats(z)
    assert np.array_equal(x0, y0) and np.array_equal(am, y0)
    assert np.array_equal(p, q) and np.array_equal(h, g)          # scale 1 is the plain pass
    assert np.all(mar >= 0) and np.all(mar <= p)                  # greedy: x0 has the largest probability
    # sampling: argmax stays the greedy proposal; the margin may be negative
    # but is then exactly prob(x0) - prob(greedy argmax)
    s0, sp, sh, smar, sam = oracle.token_stats_ex(z, temperature=0.8, key=99)
    assert np.array_equal(sam, y0)
    assert np.array_equal(sh, g)
    moved = s0 != y0
    assert moved.any()
    assert np.allclose(smar[moved], sp[moved] - q[moved], rtol=0, atol=1e-12)


def test_scaled_categorical_matches_softmax_of_scaled_logits():
    """Gumbel-max at t = 1 on z' = fp32(z / T) draws from softmax(z'), as
    the uniform-noise loop's categorical sample must; the entropy is that
    of softmax(z')."""
    z = np.array([1.0, 0.0, -0.5, 2.0, 0.25, -1.0, 1.5, 0.0], dtype=np.float32)
    T = 0.6
    s = np.float32(1.0 / T)
    n = 100_000
    rows = np.broadcast_to(z, (n, z.size))
    x0, p, h, mar, am = oracle.token_stats_ex(rows, temperature=1.0, key=4242, logit_scale=s)
    counts = np.bincount(x0, minlength=z.size)
    zs = (z * s).astype(np.float64)
    q = scipy.special.softmax(zs)
    chi2, pval = scipy.stats.chisquare(counts, q * n)
    assert pval > 1e-4, (counts, q * n, pval)
    assert np.allclose(h, scipy.stats.entropy(q), rtol=1e-12)
    assert np.all(am == 3)
    assert np.allclose(p, q[x0], rtol=1e-12)


def test_scale_validation():
    z = np.zeros((1, 4), dtype=np.float32)
    for bad in (0.0, -1.0, float("nan"), 1e6):
        with pytest.raises(ValueError):
            oracle.token_stats_ex(z, logit_scale=bad)
