"""Pins of the oracle's Gumbel chain: Philox4x32-10, ln_p and Gumbel-max.

* Philox against PyTorch's independent header-only engine
  (ATen/core/PhiloxRNGEngine.h), compiled here with g++.
* ln_p against the true logarithm, exhaustively over every uniform the
  transform can draw, within 2.5 ulp of the result.
* Gumbel-max: chi-square of the sampled x0 against softmax(z / t).
CPU only.
"""
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _torch_philox_binary(tmpdir):
    torch = pytest.importorskip("torch")
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    if not shutil.which("g++") or not os.path.exists(os.path.join(inc, "ATen", "core", "PhiloxRNGEngine.h")):
        pytest.skip("g++ or PyTorch headers unavailable")
    exe = os.path.join(tmpdir, "philox_torch")
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", inc, "-o", exe,
                    os.path.join(HERE, "pins", "philox_torch.cpp")], check=True)
    return exe


def test_philox_matches_pytorch_engine():
    rng = np.random.default_rng(31)
    cases = [np.zeros(6, np.uint32), np.full(6, 0xFFFFFFFF, np.uint32)]
    cases += [rng.integers(0, 2**32, size=6, dtype=np.uint64).astype(np.uint32) for _ in range(500)]
    # the counter layout the Gumbel transform uses: (v >> 2, row_lo, row_hi, 0)
    cases += [np.array([v, r, 0, 0, 0x9E37, 0x1234], np.uint32) for v in range(8) for r in range(3)]
    with tempfile.TemporaryDirectory() as d:
        exe = _torch_philox_binary(d)
        text = "\n".join(" ".join(str(int(x)) for x in c) for c in cases) + "\n"
        out = subprocess.run([exe], input=text, capture_output=True, text=True, check=True).stdout.split("\n")
    for c, line in zip(cases, out):
        want = [int(x) for x in line.split()]
        got = oracle.philox4x32_10(c[:4], c[4:]).tolist()
        assert got == want, (c, got, want)


def test_ln_p_within_bound_of_true_log():
    k = np.arange(2**23, dtype=np.uint64)
    u = ((2 * k + 1).astype(np.float64) * 2.0**-24).astype(np.float32)     # every uniform drawn
    rng = np.random.default_rng(32)
    E = np.concatenate([(-np.log(u.astype(np.float64))).astype(np.float32),
                        rng.uniform(5e-8, 17, 1_000_000).astype(np.float32),
                        np.float32(2.0) ** rng.uniform(-24, 4.1, 1_000_000).astype(np.float32)])
    for x in (u, E):
        got = oracle.ln_p_many(x).astype(np.float64)
        true = np.log(x.astype(np.float64))
        ulp = np.spacing(np.maximum(np.abs(got), 1e-30).astype(np.float32)).astype(np.float64)
        err = np.abs(got - true) / ulp
        assert err.max() <= 2.5, float(err.max())
    assert oracle.ln_p(1.0) == 0.0


def test_gumbel_scores_reproduce_x0():
    rng = np.random.default_rng(33)
    V = 50
    z = (rng.standard_normal((4, V)) * 2).astype(np.float32)
    key = 0xDEADBEEF12345
    x0, _, _ = oracle.token_stats(z, temperature=0.7, key=key, row_ids=[5, 6, 7, 8])
    for r in range(4):
        s = np.array([oracle.gumbel_score(z[r, v], 0.7, key, 5 + r, v) for v in range(V)], dtype=np.float32)
        assert x0[r] == int(np.argmax(s))
        g = (s - z[r]) / np.float32(0.7)
        assert np.all(np.isfinite(g)) and g.max() < 17.5 and g.min() > -3.5


def test_gumbel_max_samples_softmax_of_scaled_logits():
    z = np.array([1.0, 0.0, -0.5, 2.0, 0.25, -1.0, 1.5, 0.0], dtype=np.float32)
    t = 0.7
    n = 100_000
    rows = np.broadcast_to(z, (n, z.size))
    x0, p, h = oracle.token_stats(rows, temperature=t, key=987654321)
    counts = np.bincount(x0, minlength=z.size)
    expect = scipy.special.softmax(z.astype(np.float64) / t) * n
    chi2, pval = scipy.stats.chisquare(counts, expect)
    assert pval > 1e-4, (counts, expect, pval)
    # prob and entropy stay those of the untempered softmax
    q = scipy.special.softmax(z.astype(np.float64))
    assert np.allclose(p, q[x0], rtol=1e-12)
    assert np.allclose(h, scipy.stats.entropy(q), rtol=1e-12)
    # a different key gives a different sample stream
    y0, _, _ = oracle.token_stats(rows[:2000], temperature=t, key=987654322)
    assert not np.array_equal(y0, x0[:2000])


def test_gumbel_extreme_uniforms():
    # u = 2^-24 and u = 1 - 2^-24 stay finite through both logarithms
    lo, hi = np.float32(2.0**-24), np.float32(1 - 2.0**-24)
    for u in (lo, hi):
        E = -oracle.ln_p(u)
        g = -oracle.ln_p(E)
        assert np.isfinite(g)
        assert g == pytest.approx(-math.log(-math.log(float(u))), rel=1e-5)
