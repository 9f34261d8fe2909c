"""The seeded input generator: determinism, sampled rows, shapes, and the
spread of the LLaDA-shaped rows' top-1 probabilities (measured by the oracle).
CPU only."""
import numpy as np

import dllm_workloads as W
import oracle


def test_tiny_shape_and_peaks():
    w = W.tiny()
    assert w.logits.shape == (64, 4096) and w.logits.dtype == np.float32
    assert w.candidates.sum() == 64 and w.suppress_ids == [4095]
    x0, p, _ = oracle.token_stats(w.logits, suppress_ids=w.suppress_ids)
    assert (x0 != 4095).all() and 0 < p.min() and p.max() < 1


def test_sampled_rows_equal_full_rows():
    full = W.tiny()
    part = W.tiny(rows=[3, 40, 63])
    assert np.array_equal(part.logits, full.logits[[3, 40, 63]])
    a = W.llada(rows=[0, 31])
    b = W.llada(rows=[31])
    assert np.array_equal(a.logits[1], b.logits[0])


def test_llada_candidates_and_spread():
    w = W.llada()
    assert w.logits.shape == (32, W.LLADA_VOCAB) and w.logits.dtype == np.uint16
    assert w.candidates.sum() == 19
    _, p, _ = oracle.token_stats(w.logits, dtype="bf16", suppress_ids=w.suppress_ids)
    assert p.min() < 0.1 and p.max() > 0.99


def test_dream_and_large_rows():
    d = W.dream(rows=np.arange(0, 2048, 97))
    assert d.logits.shape == (22, W.DREAM_VOCAB) and d.temperature == 0.7 and d.key % 2 == 1
    g = W.large(rows=[0, 16383])
    assert g.logits.shape == (2, W.LLADA_VOCAB) and g.candidates.sum() == 32 * 256


def test_loop_generator_host_rows():
    spec = W.LoopSpec(V=4096, mask_id=4000, bank_rows=8)
    gen = W.LoopGenerator(spec)
    a = gen.host_logits(0, 0, 128, 32)
    b = gen.host_logits(0, 0, 128, 32)
    assert np.array_equal(a, b) and a.shape == (spec.B * 32, 4096)
    c = gen.host_logits(0, 1, 128, 32)
    assert not np.array_equal(a, c)
    assert not (gen.targets == spec.mask_id).any()
