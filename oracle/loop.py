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

from . import (StableConfidentStopping, block_ranges, edit_transfer, entropy_bound_transfer, linear_temperature,
               renoise, threshold_transfer, token_stats, token_stats_ex, uniform_canvas)


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


def uniform_keys(key: int, step: int):
    """The Philox keys of one step of the uniform-noise loop: the initial
    canvas uses `key` (step 0); step i >= 1 samples with key + 2i - 1 and
    re-noises with key + 2i (mod 2^64)."""
    m = 2**64
    return (key + 2 * step - 1) % m, (key + 2 * step) % m


def decode_uniform(model, *, batch: int, canvas_len: int, vocab_size: int, key: int, num_steps: int = 48,
                   entropy_bound: float = 0.1, t_min: float = 0.4, t_max: float = 0.8, stability_threshold: int = 1,
                   confidence_threshold: float = 0.005, dtype: str = "bf16", suppress_ids=(), n_threads: int = 0,
                   trace=None):
    """Uniform-noise decoding, composed from the oracle's primitives.

    Follows the loop of the mlx-arsenal "dLLM block decoding" notes, section
    "Uniform-noise decoding (DiffusionGemma)": the canvas starts uniformly
    random; at every step the logits are divided by the linearly decaying
    temperature, the entropy and argmax of the scaled softmax are taken and a
    categorical sample drawn from it; the lowest-entropy positions are
    accepted under the entropy budget (over all positions), every other
    position is re-noised; rows that met the stopping criterion are frozen;
    the loop ends when every row stopped or the steps ran out.  The scaled
    logits are z' = fp32(z * fp32(1 / T)); the categorical sample is the
    Gumbel-max sample at temperature 1 of z'.  ``model(step_index, canvas)``
    returns the (B * N, V) logits.  Returns (argmax canvas (B, N), steps).
    """
    B, N, V = batch, canvas_len, vocab_size
    canvas = uniform_canvas(B, N, V, key)
    stop = StableConfidentStopping(B, N, stability_threshold, confidence_threshold)
    everywhere = np.ones((B, N), dtype=np.uint8)
    done = np.zeros(B, dtype=bool)
    argmax = canvas.copy()
    steps = 0
    for remaining in range(num_steps, 0, -1):
        steps += 1
        T = linear_temperature(remaining, num_steps, t_min, t_max)
        s = np.float32(1.0 / float(T))
        k_sample, k_noise = uniform_keys(key, steps)
        logits = model(steps - 1, canvas)
        sample, _, ent, _, am = token_stats_ex(logits, dtype=dtype, temperature=1.0, key=k_sample, logit_scale=s,
                                               suppress_ids=suppress_ids, n_threads=n_threads)
        ent32 = ent.astype(np.float32).reshape(B, N)        # entropies are float32 values
        accepted = entropy_bound_transfer(ent32, everywhere, entropy_bound)
        new_canvas = renoise(sample.reshape(B, N), accepted, uniform_canvas(B, N, V, k_noise))
        argmax = np.where(done[:, None], argmax, am.reshape(B, N))
        canvas = np.where(done[:, None], canvas, new_canvas)
        done = done | (stop(argmax, ent32) != 0)
        if trace is not None:
            trace.append((steps, int(accepted.sum()), int(done.sum())))
        if done.all():
            break
    return argmax, steps
