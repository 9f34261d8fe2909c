"""Pins of the oracle's block_causal_mask: worked examples (tests/golden),
and the special cases that reduce to textbook masks -- blocks of one token
give the causal mask (numpy triu), blocks at least as long as the window give
the full bidirectional mask.  CPU only."""
import numpy as np

import oracle


def test_mask_worked_examples(golden):
    for ex in golden["block_causal_mask"]:
        got = oracle.block_causal_mask(ex["Lq"], ex["block_len"], Lk=ex["Lk"], q_offset=ex["q_offset"],
                                       k_offset=ex["k_offset"])
        want = np.array([[-np.inf if v is None else v for v in row] for row in ex["mask"]])
        assert np.array_equal(got, want), ex["cite"]


def test_unit_blocks_are_the_causal_mask():
    for L in (1, 5, 64):
        causal = np.triu(np.full((L, L), -np.inf), k=1)
        assert np.array_equal(oracle.block_causal_mask(L, 1), causal)


def test_one_block_is_bidirectional():
    for L, bl in ((7, 7), (7, 100), (32, 32)):
        assert np.array_equal(oracle.block_causal_mask(L, bl), np.zeros((L, L)))


def test_mask_is_blockwise_lower_triangular():
    L, bl = 96, 32
    m = oracle.block_causal_mask(L, bl)
    blocks = np.arange(L) // bl
    allowed = blocks[:, None] >= blocks[None, :]
    assert np.array_equal(m == 0, allowed) and np.all(np.isneginf(m[~allowed]))
