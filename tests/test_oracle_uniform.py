"""Pins of the oracle's uniform-noise decoding helpers and loop ("dLLM block
decoding", function table and "Uniform-noise decoding (DiffusionGemma)").

linear_temperature against its endpoints and closed form; uniform_canvas
against Philox4x32-10 (itself pinned to PyTorch's engine) for power-of-two
vocabularies, where floor(r V / 2^32) is the top bits of r, and statistically
for other sizes; renoise on a worked example; the stopping criterion on
hand-built call sequences; the loop on a model that is confident from the
start (closed-form step count) and on the synthetic generator (invariants).
CPU only.
"""
import numpy as np
import pytest
import scipy.stats

import dllm_workloads as W
import oracle
from oracle.loop import decode_uniform, uniform_keys


def test_linear_temperature_endpoints_and_midpoint():
    assert oracle.linear_temperature(48, 48, 0.4, 0.8) == np.float32(0.8)
    assert oracle.linear_temperature(0, 48, 0.4, 0.8) == np.float32(0.4)
    assert oracle.linear_temperature(24, 48, 0.4, 0.8) == np.float32(0.6)
    assert oracle.linear_temperature(1, 4, 1.0, 2.0) == np.float32(1.25)
    ts = [float(oracle.linear_temperature(r, 48)) for r in range(48, 0, -1)]
    assert all(a > b for a, b in zip(ts, ts[1:]))                  # decays with every step
    for bad in ((5, 4, 0.4, 0.8), (-1, 4, 0.4, 0.8), (1, 0, 0.4, 0.8), (1, 4, 0.0, 0.8), (1, 4, 0.9, 0.8)):
        with pytest.raises(ValueError):
            oracle.linear_temperature(*bad)


def test_uniform_canvas_power_of_two_is_the_top_bits_of_philox():
    key = 0x0123456789ABCDEF
    for k in (1, 12, 18):
        V = 1 << k
        c = oracle.uniform_canvas(3, 9, V, key)
        for b in range(3):
            for j in range(9):
                r = oracle.philox4x32_10([j >> 2, b, 0, 1], [key & 0xFFFFFFFF, key >> 32])[j & 3]
                assert c[b, j] == int(r) >> (32 - k)


def test_uniform_canvas_is_uniform_and_keyed():
    V = 7
    c = oracle.uniform_canvas(50, 2000, V, 99)
    counts = np.bincount(c.reshape(-1), minlength=V)
    _, pval = scipy.stats.chisquare(counts)
    assert pval > 1e-4 and c.min() >= 0 and c.max() < V
    big = oracle.uniform_canvas(2, 4096, 262144, 5)
    assert big.min() >= 0 and big.max() < 262144 and len(np.unique(big)) > 7000
    assert not np.array_equal(big, oracle.uniform_canvas(2, 4096, 262144, 6))
    assert np.array_equal(big, oracle.uniform_canvas(2, 4096, 262144, 5))


def test_renoise_worked_example():
    out = oracle.renoise([[5, 6, 7, 8]], [[1, 0, 1, 0]], [[1, 2, 3, 4]])
    assert out.tolist() == [[5, 2, 7, 4]]


def test_stopping_criterion_sequences():
    e_low = np.full((1, 4), 0.001, np.float32)
    e_high = np.full((1, 4), 0.01, np.float32)
    a = np.array([[1, 2, 3, 4]], np.int32)
    b = np.array([[1, 2, 3, 5]], np.int32)
    st = oracle.StableConfidentStopping(1, 4, stability_threshold=1, confidence_threshold=0.005)
    assert st(a, e_low)[0] == 0          # the first canvas has nothing to be stable against
    assert st(a, e_low)[0] == 1          # stable once and confident
    assert st(b, e_low)[0] == 0          # a change resets the count
    assert st(b, e_high)[0] == 0         # stable but not confident
    assert st(b, e_low)[0] == 1
    st2 = oracle.StableConfidentStopping(1, 4, stability_threshold=2, confidence_threshold=0.005)
    assert [int(st2(a, e_low)[0]) for _ in range(4)] == [0, 0, 1, 1]
    # confident means a mean strictly below the threshold, decided exactly:
    # (0.25 + 0.75) / 2 equals 0.5, and one ulp less is below it
    st3 = oracle.StableConfidentStopping(1, 2, 1, 0.5)
    half = np.array([[0.25, 0.75]], np.float32)
    st3(np.array([[0, 0]], np.int32), half)
    assert st3(np.array([[0, 0]], np.int32), half)[0] == 0
    below = np.array([[0.25, np.nextafter(np.float32(0.75), np.float32(0))]], np.float32)
    assert st3(np.array([[0, 0]], np.int32), below)[0] == 1
    # NaN and huge entropies count as 64; the threshold must lie in [0, 64]
    st5 = oracle.StableConfidentStopping(1, 2, 0, 40.0)
    assert st5(np.array([[0, 0]], np.int32), np.array([[np.nan, 0.0]], np.float32))[0] == 1   # mean 32
    assert st5(np.array([[0, 0]], np.int32), np.array([[np.nan, 17.0]], np.float32))[0] == 0  # mean 40.5
    with pytest.raises(ValueError):
        oracle.StableConfidentStopping(1, 2, 1, 65.0)(np.zeros((1, 2), np.int32), np.zeros((1, 2), np.float32))
    # rows are independent
    st4 = oracle.StableConfidentStopping(2, 4, 1, 0.005)
    st4(np.vstack([a, a]), np.vstack([e_low, e_low]))
    assert st4(np.vstack([a, b]), np.vstack([e_low, e_low])).tolist() == [1, 0]


def test_loop_confident_from_the_start_stops_at_step_two():
    """Peaks from step 0: step 1 has no previous canvas, step 2 is stable and
    confident, so every row stops after exactly two steps with the targets."""
    spec = W.uniform_spec(B=2, N=16, V=1024, dtype="f32", max_onset=0)
    gen = W.UniformGenerator(spec)
    tr = []
    am, steps = decode_uniform(lambda st, c: gen.host_logits(st), batch=2, canvas_len=16, vocab_size=1024,
                               key=spec.key, dtype="f32", trace=tr)
    assert steps == 2 and np.array_equal(am, gen.targets)
    assert [t[2] for t in tr] == [0, 2]


def test_loop_invariants_on_the_generator():
    spec = W.uniform_spec(B=3, N=24, V=2048, dtype="bf16", max_onset=6)
    gen = W.UniformGenerator(spec)
    tr = []
    am, steps = decode_uniform(lambda st, c: gen.host_logits(st), batch=3, canvas_len=24, vocab_size=2048,
                               key=spec.key, dtype="bf16", trace=tr)
    # every position is confident from step index 6 on: stable at step 8 at the latest
    assert steps <= 8 and np.array_equal(am, gen.targets)
    assert all(t[1] >= 3 for t in tr)                 # at least one accepted position per row
    assert uniform_keys(spec.key, 1) == (spec.key + 1, spec.key + 2)
    # the step budget bounds the loop
    am2, steps2 = decode_uniform(lambda st, c: gen.host_logits(st), batch=3, canvas_len=24, vocab_size=2048,
                                 key=spec.key, dtype="bf16", num_steps=4)
    assert steps2 == 4
