"""Pins of the CPU oracle to what the pages and the mathematics fix.

Worked examples (tests/golden), closed forms, textbook routines (scipy),
and the NaN / infinity / suppression conventions.  CPU only.
"""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
from dllm_workloads import f32_to_bf16_bits


def test_token_stats_worked_examples(golden):
    for ex in golden["token_stats"]:
        z = np.asarray([ex["logits"]], dtype=np.float32)
        x0, p, h = oracle.token_stats(z, suppress_ids=ex["suppress_ids"])
        assert x0[0] == ex["x0"], ex["cite"]
        # the fp32 rounding of ln 3 moves p by ~1e-8
        assert p[0] == pytest.approx(ex["prob"], rel=1e-7), ex["cite"]
        assert h[0] == pytest.approx(ex["entropy"], rel=1e-7), ex["cite"]


def test_closed_form_uniform_row():
    for V in (1, 7, 4096, 126464):
        z = np.full((1, V), 1.25, dtype=np.float32)
        x0, p, h = oracle.token_stats(z)
        assert x0[0] == 0
        assert p[0] == pytest.approx(1.0 / V, rel=1e-12)
        assert h[0] == pytest.approx(math.log(V), rel=1e-12, abs=1e-15)


def test_closed_form_two_level_row():
    # one logit a above V-1 equal ones: p = e^a / (e^a + V - 1),
    # H = ln(e^a + V - 1) - a e^a / (e^a + V - 1)
    for a, V, pos in ((8.0, 4096, 17), (3.0, 1000, 999), (0.5, 2, 0)):
        z = np.zeros((1, V), dtype=np.float32)
        z[0, pos] = a
        x0, p, h = oracle.token_stats(z)
        ea = math.exp(a)
        assert x0[0] == pos
        assert p[0] == pytest.approx(ea / (ea + V - 1), rel=1e-12)
        assert h[0] == pytest.approx(math.log(ea + V - 1) - a * ea / (ea + V - 1), rel=1e-11)
    # the values quoted for a=8, V=4096
    z = np.zeros((1, 4096), dtype=np.float32)
    z[0, 0] = 8.0
    _, p, h = oracle.token_stats(z)
    assert p[0] == pytest.approx(0.4212798, abs=1e-7)
    assert h[0] == pytest.approx(5.494220, abs=1e-6)


def test_textbook_softmax_entropy_scipy():
    rng = np.random.default_rng(11)
    for V, scale in ((3, 1.0), (50, 4.0), (4096, 3.0), (20000, 0.3)):
        z = (rng.standard_normal((6, V)) * scale).astype(np.float32)
        x0, p, h = oracle.token_stats(z)
        for r in range(z.shape[0]):
            q = scipy.special.softmax(z[r].astype(np.float64))
            assert x0[r] == int(np.argmax(z[r]))
            assert p[r] == pytest.approx(q[x0[r]], rel=1e-12)
            assert h[r] == pytest.approx(scipy.stats.entropy(q), rel=1e-10, abs=1e-13)


def test_suppression_equals_deleting_columns():
    rng = np.random.default_rng(12)
    V = 300
    z = (rng.standard_normal((5, V)) * 2).astype(np.float32)
    sup = [0, 3, 17, 299, 150]
    x0, p, h = oracle.token_stats(z, suppress_ids=sup)
    keep = np.array([v for v in range(V) if v not in sup])
    for r in range(5):
        q = scipy.special.softmax(z[r, keep].astype(np.float64))
        j = int(np.argmax(z[r, keep]))
        assert x0[r] == keep[j]
        assert p[r] == pytest.approx(q[j], rel=1e-12)
        assert h[r] == pytest.approx(scipy.stats.entropy(q), rel=1e-10)
    # suppressing the argmax moves x0 to the runner-up
    z2 = np.array([[0.0, 5.0, 4.0, 1.0]], dtype=np.float32)
    assert oracle.token_stats(z2, suppress_ids=[1])[0][0] == 2


def test_nan_and_neg_inf_carry_no_mass():
    z = np.array([[np.nan, 1.0, -np.inf, 2.0, np.nan, -3e30]], dtype=np.float32)
    x0, p, h = oracle.token_stats(z)
    q = scipy.special.softmax(np.array([1.0, 2.0]))
    assert x0[0] == 3
    assert p[0] == pytest.approx(q[1], rel=1e-12)
    assert h[0] == pytest.approx(scipy.stats.entropy(q), rel=1e-12)


def test_all_masked_row_is_uniform_limit():
    V = 9
    for fill in (np.nan, -np.inf, -2.0**100):
        z = np.full((1, V), fill, dtype=np.float32)
        x0, p, h = oracle.token_stats(z, suppress_ids=[0, 4])
        assert x0[0] == 1
        assert p[0] == pytest.approx(1.0 / 7)
        assert h[0] == pytest.approx(math.log(7))


def test_positive_infinity_shares_mass():
    # +inf entries share the mass equally; finite logits, however large, get none
    z = np.array([[0.0, np.inf, 5.0, 2.0**101, np.inf, 1.0]], dtype=np.float32)
    x0, p, h = oracle.token_stats(z)
    assert x0[0] == 1 and p[0] == pytest.approx(1 / 2) and h[0] == pytest.approx(math.log(2))
    x0, p, h = oracle.token_stats(z, temperature=0.5, key=3)
    assert x0[0] in (1, 4) and p[0] == pytest.approx(1 / 2)


def test_huge_finite_logits_take_the_plain_softmax():
    """Finite logits beyond any clamp are ordinary logits ("dLLM block
    decoding", What mlx-arsenal ships: token_stats is NaN-safe; nothing else
    is special).  exp(1e37 - 1e38) is 0 in double, so the larger takes all."""
    z = np.array([[1e38, 1e37]], dtype=np.float32)
    x0, p, h = oracle.token_stats(z)
    assert x0[0] == 0 and p[0] == 1.0 and h[0] == 0.0
    # a single finite logit among NaNs is certain, however negative it is
    z = np.array([[-1e31, np.nan, np.nan]], dtype=np.float32)
    x0, p, h = oracle.token_stats(z)
    assert x0[0] == 0 and p[0] == 1.0 and h[0] == 0.0
    # three equal maxima at the top of the fp32 range share the mass
    top = np.float32(3.4e38)
    z = np.array([[5.0, top, -top, top, 1e30, top]], dtype=np.float32)
    x0, p, h = oracle.token_stats(z)
    assert x0[0] == 1 and p[0] == pytest.approx(1 / 3, rel=1e-15) and h[0] == pytest.approx(math.log(3), rel=1e-15)
    # the same row sampled: one of the maxima, with its share
    x0, p, h = oracle.token_stats(z, temperature=0.8, key=11)
    assert x0[0] in (1, 3, 5) and p[0] == pytest.approx(1 / 3, rel=1e-15)


@pytest.mark.parametrize("level", [0.0, 1e3, -1e3, 2.0**20, -(2.0**20), 1e9, -1e9])
def test_two_level_rows_at_any_offset(level):
    """Closed form of a row with a entries at x and b entries at x - d:
    p = 1 / (a + b e^-d) for an entry at x, H = ln(a + b e^-d) + b d e^-d / (a + b e^-d).
    Softmax is shift invariant, so the answer does not depend on x: the
    oracle must give it at every offset, up to the fp32 spacing of x."""
    x = np.float32(level)
    ulp = float(np.spacing(np.abs(x))) if x != 0 else 2.0**-149
    d = float(np.float32(max(1.5, ulp)))          # an exact fp32 gap at this offset
    lo = np.float32(x - np.float32(d))
    d = float(x) - float(lo)
    a, b = 3, 5
    z = np.array([[lo] * b + [x] * a], dtype=np.float32)
    x0, p, h = oracle.token_stats(z)
    Z = a + b * math.exp(-d)
    assert x0[0] == b
    assert p[0] == pytest.approx(1 / Z, rel=1e-12)
    assert h[0] == pytest.approx(math.log(Z) + b * d * math.exp(-d) / Z, rel=1e-10, abs=1e-15)


def test_bf16_widening_matches_torch():
    rng = np.random.default_rng(13)
    z = (rng.standard_normal((3, 777)) * 5).astype(np.float32)
    bits = f32_to_bf16_bits(z)
    widened = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    xa, pa, ha = oracle.token_stats(bits, dtype="bf16")
    xb, pb, hb = oracle.token_stats(widened)
    assert np.array_equal(xa, xb) and np.array_equal(pa, pb) and np.array_equal(ha, hb)
    # the generator's rounding agrees with torch's float -> bf16 conversion
    tb = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(tb, bits)


def test_stats_invariants_random():
    rng = np.random.default_rng(14)
    for trial in range(20):
        V = int(rng.integers(2, 3000))
        z = (rng.standard_normal((4, V)) * rng.uniform(0.1, 30)).astype(np.float32)
        nsup = int(rng.integers(0, min(V - 1, 5) + 1))
        sup = rng.choice(V, size=nsup, replace=False).tolist()
        t = float(rng.choice([0.0, 0.7, 1.3]))
        x0, p, h = oracle.token_stats(z, temperature=t, key=int(rng.integers(1, 2**62)), suppress_ids=sup)
        veff = V - nsup
        assert np.all(p > 0) and np.all(p <= 1)
        assert np.all(h >= 0) and np.all(h <= math.log(veff) + 1e-12)
        assert not set(x0.tolist()) & set(sup)


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(15)
    z = (rng.standard_normal((37, 1000)) * 3).astype(np.float32)
    a = oracle.token_stats(z, temperature=0.9, key=77, n_threads=1)
    b = oracle.token_stats(z, temperature=0.9, key=77, n_threads=5)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


@pytest.mark.parametrize("rule", ["threshold_transfer", "topk_transfer", "factor_transfer",
                                  "entropy_bound_transfer"])
def test_rule_worked_examples(golden, rule):
    for ex in golden[rule]:
        if rule == "threshold_transfer":
            got = oracle.threshold_transfer(ex["conf"], ex["cand"], ex["tau"], ex["strict"])
        elif rule == "topk_transfer":
            got = oracle.topk_transfer(ex["conf"], ex["cand"], ex["k"])
        elif rule == "factor_transfer":
            got = oracle.factor_transfer(ex["conf"], ex["cand"], ex["factor"])
        else:
            got = oracle.entropy_bound_transfer(ex["entropy"], ex["cand"], ex["gamma"])
        assert got[0].tolist() == ex["commit"], ex["cite"]


def test_edit_worked_examples(golden):
    for ex in golden["edit_transfer"]:
        got = oracle.edit_transfer(ex["x0"], ex["prob"], ex["tokens"], ex["editable"], ex["tau_edit"])
        assert got.tolist() == ex["edit"], ex["cite"]


def test_schedule_worked_examples(golden):
    for ex in golden["transfer_schedule"]:
        assert oracle.transfer_schedule(ex["counts"], ex["steps"]).tolist() == ex["quotas"], ex["cite"]
    for ex in golden["block_ranges"]:
        got = oracle.block_ranges(ex["P"], ex["gen_len"], ex["block_len"], ex["align"])
        assert [list(r) for r in got] == ex["ranges"], ex["cite"]


def test_schedule_invariants_determine_it():
    # A non-increasing sequence of `steps` integers summing to n whose entries
    # differ by at most one is unique, so these checks pin the schedule fully.
    rng = np.random.default_rng(16)
    for _ in range(200):
        steps = int(rng.integers(1, 70))
        counts = rng.integers(0, 600, size=3)
        q = oracle.transfer_schedule(counts, steps)
        for b in range(3):
            assert q[b].sum() == counts[b]
            assert np.all(np.diff(q[b]) <= 0)
            assert q[b].max() - q[b].min() <= 1
    assert oracle.transfer_schedule([-4], 3).tolist() == [[0, 0, 0]]
    assert oracle.transfer_schedule([256], 32)[0, 0] == 8


def test_block_ranges_tile_the_generation_region():
    rng = np.random.default_rng(17)
    for _ in range(300):
        P, gen, bl = int(rng.integers(0, 300)), int(rng.integers(0, 500)), int(rng.integers(1, 70))
        for align in (False, True):
            r = oracle.block_ranges(P, gen, bl, align)
            if gen == 0:
                assert r == []
                continue
            covered = []
            for (s, e) in r:
                assert 0 < e - s <= bl
                covered.extend(range(max(s, P), e))
                if align:
                    assert s % bl == 0
            assert covered == list(range(P, P + gen))
            assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
            if not align:
                assert r[0][0] == P
    assert len(oracle.block_ranges(128, 1024, 32)) == 32
    assert oracle.block_ranges(128, 1024, 32, True) == oracle.block_ranges(128, 1024, 32, False)


def test_entropy_bound_sums_exactly():
    """The prefix sums of the entropy-bound rule are exact (fixed point, 40
    fractional bits) and compared exactly with gamma: sums that reach gamma
    exactly are within it; a tiny excess is not; a NaN entropy ranks last."""
    e = np.array([[0.25, 0.25, 0.5]], np.float32)          # exclusive sums 0, 0.25, 0.5
    assert oracle.entropy_bound_transfer(e, np.ones_like(e, np.uint8), 0.5).tolist() == [[1, 1, 1]]
    assert oracle.entropy_bound_transfer(e, np.ones_like(e, np.uint8), np.nextafter(np.float32(0.5), np.float32(0))
                                         ).tolist() == [[1, 1, 0]]
    # 1000 entropies of 2^-30 sum to 1000 * 2^-30 exactly: within gamma = 1000 * 2^-30, one ulp below is not
    tiny = np.full((1, 1001), 2.0**-30, np.float32)
    g = np.float32(1000 * 2.0**-30)
    assert oracle.entropy_bound_transfer(tiny, np.ones_like(tiny, np.uint8), g).sum() == 1001
    assert oracle.entropy_bound_transfer(tiny, np.ones_like(tiny, np.uint8),
                                         np.nextafter(g, np.float32(0))).sum() == 1000
    # NaN ranks last; its exclusive prefix is the other two: 0.01 > 0.005
    n = np.array([[np.nan, 0.0, 0.01]], np.float32)
    assert oracle.entropy_bound_transfer(n, np.ones_like(n, np.uint8), 100.0).tolist() == [[1, 1, 1]]
    assert oracle.entropy_bound_transfer(n, np.ones_like(n, np.uint8), 0.005).tolist() == [[0, 1, 1]]
