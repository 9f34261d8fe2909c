"""Block decoding with token editing, composed from the oracle's primitives.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows the LLaDA2.1-style loop of the mlx-arsenal "dLLM block decoding"
notes, section "Token editing (LLaDA2.1)": whole blocks aligned on absolute
positions; per step, the masked positions of the block are the candidates of
a strict threshold commit and the block's other generated positions may be
edited; a block ends after a step that had no mask and made no edit, or once
more than ``max_post_steps`` extra passes ran on a full block.  Batch rows
share the loop's termination, as the notes state for B > 1.

The caller's ``model(block_index, step_in_block, col0, n_cols)`` returns the
logits of canvas columns [col0, col0 + n_cols) for every batch row, as a
(B * n_cols, V) array; only in-block rows can commit or edit, so the rows of
the rest of the window are never needed.
"""
from __future__ import annotations

import numpy as np

from . import block_ranges, edit_transfer, threshold_transfer, token_stats


def decode_with_editing(model, prompt: np.ndarray, *, gen_len: int, block_len: int, mask_id: int,
                        dtype: str = "bf16", threshold: float = 0.95, editing_threshold: float = 0.9,
                        max_post_steps: int = 16, suppress_ids=(), n_threads: int = 0, trace=None):
    B, P = prompt.shape
    total = -(-(P + gen_len) // block_len) * block_len          # whole blocks
    x = np.concatenate([prompt.astype(np.int32), np.full((B, total - P), mask_id, np.int32)], axis=1)
    forwards = 0
    for bi, (start, end) in enumerate(block_ranges(P, total - P, block_len, align=True)):
        lo = max(start, P)                                     # in-block and outside the prompt
        n = end - lo
        post_steps = 0
        step = 0
        while True:
            window = x[:, lo:end]
            masked = window == mask_id
            has_mask = bool(masked.any())
            if not has_mask:
                post_steps += 1
                if post_steps > max_post_steps:
                    break
            logits = model(bi, step, lo, n)
            x0, prob, _ = token_stats(logits, dtype=dtype, suppress_ids=suppress_ids, n_threads=n_threads)
            forwards += 1
            x0 = x0.reshape(B, n)
            conf = prob.astype(np.float32).reshape(B, n)        # confidences are float32 values
            commit = threshold_transfer(conf, masked, threshold, strict=True).astype(bool)
            edit = edit_transfer(x0, conf, window, ~masked, editing_threshold).astype(bool)
            x[:, lo:end] = np.where(commit | edit, x0, window)
            if trace is not None:
                trace.append((bi, step, int(commit.sum()), int(edit.sum())))
            step += 1
            if not has_mask and not edit.any():
                break
    return x[:, P:P + gen_len], forwards
