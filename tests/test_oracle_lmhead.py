"""Pins of the oracle's fused LM head + statistics: the logits against exact
rational arithmetic (Python fractions) on small shapes, an identity weight
(the logits are the hidden values themselves), and the statistics equal to
token_stats of those logits.  CPU only."""
from fractions import Fraction

import numpy as np

import oracle
from dllm_workloads import f32_to_bf16_bits


def bf16_value(bits) -> Fraction:
    return Fraction(float((np.uint32(bits) << np.uint32(16)).view(np.float32)))


def test_logits_equal_the_exact_sum_rounded_once():
    rng = np.random.default_rng(1)
    h = f32_to_bf16_bits(rng.standard_normal((4, 96)).astype(np.float32) * 3)
    w = f32_to_bf16_bits(rng.standard_normal((7, 96)).astype(np.float32))
    got = oracle.lm_head_logits(h, w)
    for t in range(4):
        for v in range(7):
            exact = sum(bf16_value(h[t, k]) * bf16_value(w[v, k]) for k in range(96))
            assert got[t, v] == np.float32(float(exact))


def test_identity_weight_gives_the_hidden_values():
    rng = np.random.default_rng(2)
    d = 64
    h = f32_to_bf16_bits(rng.standard_normal((5, d)).astype(np.float32) * 2)
    eye = f32_to_bf16_bits(np.eye(d, dtype=np.float32))
    logits = oracle.lm_head_logits(h, eye)
    assert np.array_equal(logits, (h.astype(np.uint32) << 16).view(np.float32))
    x0, p, e = oracle.lm_head_stats(h, eye, suppress_ids=[3])
    y0, q, f = oracle.token_stats(h, dtype="bf16", suppress_ids=[3])
    assert np.array_equal(x0, y0) and np.array_equal(p, q) and np.array_equal(e, f)
