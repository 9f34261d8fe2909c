"""Brute-force pins of the oracle's commit rules on tiny rows.

Each rule's output is characterised over ALL subsets of the candidates,
without sorting: a committed set must be a "prefix set" of the ranking (every
member outranks every non-member; ranking = higher confidence first, then lower
position) and be the largest such set whose members all satisfy the rule's
predicate.  Values are dyadic rationals so every sum and product is exact and
the summation order cannot matter.  CPU only.
"""
import itertools

import numpy as np

import oracle

DYADIC_CONF = np.arange(0, 17, dtype=np.float32) / 16       # 0, 1/16, ..., 1
DYADIC_ENT = np.arange(0, 12, dtype=np.float32) / 32        # 0 .. 11/32


def outranks(c, i, j):
    return c[i] > c[j] or (c[i] == c[j] and i < j)


def prefix_sets(c, cands):
    for r in range(len(cands) + 1):
        for S in itertools.combinations(cands, r):
            rest = [j for j in cands if j not in S]
            if all(outranks(c, i, j) for i in S for j in rest):
                yield set(S)


def rank_in(c, S, i):
    return sum(1 for j in S if j != i and outranks(c, j, i))


def random_row(rng, L, values):
    c = rng.choice(values, size=L).astype(np.float32)
    cand = (rng.random(L) < 0.7).astype(np.uint8)
    return c, cand


def test_topk_bruteforce():
    rng = np.random.default_rng(21)
    for _ in range(300):
        L = int(rng.integers(1, 9))
        c, cand = random_row(rng, L, DYADIC_CONF)
        k = int(rng.integers(-1, L + 2))
        cands = [i for i in range(L) if cand[i]]
        want = [S for S in prefix_sets(c, cands) if len(S) == min(max(k, 0), len(cands))]
        assert len(want) == 1
        got = oracle.topk_transfer(c, cand, k)[0]
        assert set(np.flatnonzero(got).tolist()) == want[0]


def test_threshold_bruteforce():
    rng = np.random.default_rng(22)
    for _ in range(300):
        L = int(rng.integers(1, 9))
        c, cand = random_row(rng, L, DYADIC_CONF)
        tau = float(rng.choice(DYADIC_CONF))
        strict = bool(rng.integers(0, 2))
        cands = [i for i in range(L) if cand[i]]
        passing = {i for i in cands if (c[i] > tau if strict else c[i] >= tau)}
        if cands and not passing:
            # exactly one: the member of the size-1 prefix set
            (want,) = [S for S in prefix_sets(c, cands) if len(S) == 1]
        else:
            want = passing
        got = oracle.threshold_transfer(c, cand, tau, strict)[0]
        assert set(np.flatnonzero(got).tolist()) == want


def test_factor_bruteforce():
    rng = np.random.default_rng(23)
    for _ in range(300):
        L = int(rng.integers(1, 9))
        c, cand = random_row(rng, L, DYADIC_CONF)
        f = float(rng.choice(np.arange(0, 33) / 16))
        cands = [i for i in range(L) if cand[i]]
        ok = [S for S in prefix_sets(c, cands)
              if all((rank_in(c, S, i) + 1) * (1 - float(c[i])) <= f for i in S)]
        want = max(ok, key=len)
        if cands and not want:
            (want,) = [S for S in prefix_sets(c, cands) if len(S) == 1]
        got = oracle.factor_transfer(c, cand, f)[0]
        assert set(np.flatnonzero(got).tolist()) == want


def test_entropy_bound_bruteforce():
    rng = np.random.default_rng(24)
    for _ in range(300):
        L = int(rng.integers(1, 9))
        h, cand = random_row(rng, L, DYADIC_ENT)
        gamma = float(rng.choice(np.arange(-2, 40) / 32))
        neg = -h  # low entropy ranks first: rank by -H, then position
        cands = [i for i in range(L) if cand[i]]
        ok = [S for S in prefix_sets(neg, cands)
              if all(sum(float(h[j]) for j in S if outranks(neg, j, i)) <= gamma for i in S)]
        want = max(ok, key=len)
        if cands and not want:
            (want,) = [S for S in prefix_sets(neg, cands) if len(S) == 1]
        got = oracle.entropy_bound_transfer(h, cand, gamma)[0]
        assert set(np.flatnonzero(got).tolist()) == want


def test_rules_invariants_random_floats():
    rng = np.random.default_rng(25)
    for _ in range(50):
        B, L = int(rng.integers(1, 5)), int(rng.integers(1, 300))
        c = rng.random((B, L)).astype(np.float32)
        c[rng.random((B, L)) < 0.05] = np.nan
        cand = (rng.random((B, L)) < 0.5).astype(np.uint8)
        n_c = cand.sum(1)
        k = rng.integers(0, L + 1, size=B).astype(np.int32)
        for out in (oracle.threshold_transfer(c, cand, 0.9, True), oracle.factor_transfer(c, cand, 1.0),
                    oracle.entropy_bound_transfer(c, cand, 0.1)):
            assert np.all(out <= cand)
            assert np.all((out.sum(1) >= 1) == (n_c >= 1))
        t = oracle.topk_transfer(c, cand, k)
        assert np.all(t <= cand) and np.array_equal(t.sum(1), np.minimum(k, n_c))


def test_nan_confidence_ranks_last():
    c = np.array([np.nan, 0.2, np.nan, 0.1], dtype=np.float32)
    cand = np.ones(4, np.uint8)
    assert oracle.topk_transfer(c, cand, 3)[0].tolist() == [1, 1, 0, 1]
    assert oracle.threshold_transfer([np.nan, np.nan], [1, 1], 0.5)[0].tolist() == [1, 0]
    h = np.array([np.nan, 0.01, 0.02], dtype=np.float32)
    assert oracle.entropy_bound_transfer(h, [1, 1, 1], 10.0)[0].tolist() == [1, 1, 1]
    assert oracle.entropy_bound_transfer(h, [1, 0, 0], 10.0)[0].tolist() == [1, 0, 0]
