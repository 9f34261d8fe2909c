"""Pins of the oracle's block-decoding loop with editing on toy models whose
trajectory is known in closed form.  CPU only."""
import numpy as np

from oracle.loop import decode_with_editing

V, MASK = 16, 15


def peaked_rows(ids, height=30.0):
    ids = np.asarray(ids).reshape(-1)
    z = np.zeros((ids.size, V), dtype=np.float32)
    z[np.arange(ids.size), ids] = height
    return z


def test_confident_model_takes_two_passes_per_block():
    B, P, gen, bl = 2, 3, 10, 4
    target = (np.arange(B * (P + 16)).reshape(B, -1) % 7).astype(np.int32)

    def model(bi, step, col0, n):
        return peaked_rows(target[:, col0:col0 + n])

    out, fw = decode_with_editing(model, np.zeros((B, P), np.int32), gen_len=gen, block_len=bl,
                                  mask_id=MASK, dtype="f32", suppress_ids=[MASK])
    # aligned blocks [0,4) [4,8) [8,12) [12,16): each needs a commit pass and a
    # post pass that sees no mask and makes no edit
    assert fw == 2 * 4
    assert np.array_equal(out, target[:, P:P + gen])


def test_draft_then_revision_takes_three_passes():
    B, P, gen, bl = 1, 4, 8, 4
    draft = np.full((B, 12), 3, np.int32)
    final = np.full((B, 12), 9, np.int32)

    def model(bi, step, col0, n):
        src = draft if step == 0 else final
        return peaked_rows(src[:, col0:col0 + n])

    trace = []
    out, fw = decode_with_editing(model, np.zeros((B, P), np.int32), gen_len=gen, block_len=bl,
                                  mask_id=MASK, dtype="f32", trace=trace)
    # per block: commit the draft, edit to the final tokens, a pass with no edit
    assert fw == 3 * 2
    assert [t[2:] for t in trace] == [(4, 0), (0, 4), (0, 0)] * 2
    assert np.array_equal(out, final[:, P:P + gen])


def test_unconfident_model_forces_one_per_step_and_stops_after_post_steps():
    B, P, gen, bl = 1, 0, 4, 4

    def model(bi, step, col0, n):
        z = np.zeros((n, V), dtype=np.float32)       # uniform: p = 1/15 < 0.95
        z[:, 5] = 0.5 + 0.01 * np.arange(n)          # argmax 5, the last row most confident
        return z

    trace = []
    out, fw = decode_with_editing(model, np.zeros((B, P), np.int32), gen_len=gen, block_len=bl,
                                  mask_id=MASK, dtype="f32", suppress_ids=[MASK], max_post_steps=2,
                                  trace=trace)
    # one forced commit per step, most confident (last) masked row first
    assert [t[2] for t in trace[:4]] == [1, 1, 1, 1]
    assert np.array_equal(out, np.full((1, 4), 5))
    # the first post pass makes no edit (x0 equals the tokens) and ends the block
    assert fw == 5
