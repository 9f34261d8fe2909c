"""Decoding loops on the GPU, built on the fused commit step.

``decode_with_editing`` follows the loop of the mlx-arsenal "dLLM block
decoding" notes, section "Token editing (LLaDA2.1)": whole blocks aligned on
absolute positions; at each step the block's masked positions are the
candidates of a strict threshold commit and its other generated positions may
be edited; a block ends after a step with no mask and no edit, or once more
than ``max_post_steps`` extra passes ran on a full block; batch rows share the
termination.  Each step is one fused launch (statistics, threshold, edit and
canvas update) plus one read of three counters per batch row.  The caller's
``model(block_index, step_in_block, col0, n_cols)`` returns the
(B * n_cols, V) logits of canvas columns [col0, col0 + n_cols) on the device.

``decode_uniform`` follows the same notes' "Uniform-noise decoding
(DiffusionGemma)" loop (see its docstring).
"""
from __future__ import annotations

import numpy as np
import torch

from . import (RULE_ENTROPY_BOUND, RULE_THRESHOLD, StableConfidentStopping, block_ranges, commit_step,
               linear_temperature, uniform_canvas, uniform_update)

_GATE_CYCLES = 1_000_000   # about 0.5 ms of SM clock: well beyond what the host needs to enqueue a step


def decode_with_editing(model, prompt: torch.Tensor, *, gen_len: int, block_len: int, mask_id: int,
                        threshold: float = 0.95, editing_threshold: float = 0.9, max_post_steps: int = 16,
                        suppress_ids=(), step_times=None, trace=None):
    """Returns (generated tokens (B, gen_len), number of forwards).

    ``step_times``: optional list receiving the GPU time (ms) of each fused
    commit step, measured with CUDA events on the current stream.
    """
    dev = prompt.device
    B, P = prompt.shape
    total = -(-(P + gen_len) // block_len) * block_len
    x = torch.full((B, total), mask_id, dtype=torch.int32, device=dev)
    x[:, :P] = prompt.to(torch.int32)
    counts = torch.zeros((B, 3), dtype=torch.int32, device=dev)
    counts_host = torch.zeros((B, 3), dtype=torch.int32).pin_memory()
    forwards = 0
    for bi, (start, end) in enumerate(block_ranges(P, total - P, block_len, align=True)):
        lo = max(start, P)
        n = end - lo
        if n <= 0:
            continue
        has_mask = bool((x[:, lo:end] == mask_id).any().item())
        post_steps = 0
        step = 0
        while True:
            if not has_mask:
                post_steps += 1
                if post_steps > max_post_steps:
                    break
            logits = model(bi, step, lo, n).view(B, n, -1)
            if step_times is not None:
                # Hold the GPU busy while the host enqueues the step, so that
                # the events time the commit step rather than the host's launch
                # (in a real loop the model's forward plays this part).
                torch.cuda._sleep(_GATE_CYCLES)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
            commit_step(logits, rule=RULE_THRESHOLD, tau=threshold, strict=True, suppress_ids=suppress_ids,
                        mask_id=mask_id, edit=True, tau_edit=editing_threshold, canvas=x, canvas_offset=lo,
                        counts=counts)
            if step_times is not None:
                e1.record()
            forwards += 1
            counts_host.copy_(counts)          # the one host read of the step
            c = counts_host.numpy()
            if step_times is not None:
                step_times.append(e0.elapsed_time(e1))
            n_commit, n_edit = int(c[:, 1].sum()), int(c[:, 2].sum())
            if trace is not None:
                trace.append((bi, step, n_commit, n_edit))
            masked_after = int((c[:, 0] - c[:, 1]).sum())
            step += 1
            if not has_mask and n_edit == 0:
                break
            has_mask = masked_after > 0
    return x[:, P:P + gen_len], forwards


def uniform_keys(key: int, step: int):
    """Philox keys of step `step` (>= 1) of the uniform-noise loop: the sample
    uses key + 2 step - 1 and the re-noising key + 2 step (mod 2^64); the
    initial canvas uses key itself."""
    m = 2**64
    return (key + 2 * step - 1) % m, (key + 2 * step) % m


def decode_uniform(model, *, batch: int, canvas_len: int, vocab_size: int, key: int, num_steps: int = 48,
                   entropy_bound: float = 0.1, t_min: float = 0.4, t_max: float = 0.8, stability_threshold: int = 1,
                   confidence_threshold: float = 0.005, suppress_ids=(), device=None, step_times=None, trace=None):
    """Uniform-noise (DiffusionGemma-style) decoding on the GPU.

    Follows the loop of the mlx-arsenal "dLLM block decoding" notes, section
    "Uniform-noise decoding (DiffusionGemma)": a uniformly random canvas; per
    step, one fused launch takes the statistics of the logits scaled by
    1 / linear_temperature (argmax, entropy, and a categorical sample as the
    Gumbel-max sample at temperature 1) and accepts the lowest-entropy
    positions under the entropy bound over every position; then the rest is
    re-noised, the rows that already stopped stay frozen, and the stopping
    criterion updates the rows' done flags -- all of that a second launch
    (one 1-byte-per-row host read per step decides the loop's end).  ``model(step_index, canvas)`` returns the
    (B * N, V) logits on the device.  Returns (argmax canvas (B, N), steps).
    """
    B, N, V = batch, canvas_len, vocab_size
    dev = torch.device(device or "cuda")
    canvas = uniform_canvas(B, N, V, key, device=dev)
    argmax = canvas.clone()
    am_new = torch.empty_like(canvas)
    sample = torch.empty_like(canvas)
    prob = torch.empty((B, N), dtype=torch.float32, device=dev)
    ent = torch.empty_like(prob)
    accepted = torch.empty((B, N), dtype=torch.uint8, device=dev)
    everywhere = torch.ones((B, N), dtype=torch.uint8, device=dev)
    done = torch.zeros((B,), dtype=torch.uint8, device=dev)
    done_host = torch.zeros((B,), dtype=torch.uint8).pin_memory()
    stop = StableConfidentStopping(B, N, stability_threshold, confidence_threshold, device=dev)
    steps = 0
    for remaining in range(num_steps, 0, -1):
        steps += 1
        T = linear_temperature(remaining, num_steps, t_min, t_max)
        scale = float(np.float32(1.0 / T))
        k_sample, k_noise = uniform_keys(key, steps)
        logits = model(steps - 1, canvas).view(B, N, V)
        if step_times is not None:
            torch.cuda._sleep(_GATE_CYCLES)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
        commit_step(logits, rule=RULE_ENTROPY_BOUND, gamma=entropy_bound, temperature=1.0, key=k_sample,
                    suppress_ids=suppress_ids, cand=everywhere, logit_scale=scale, argmax=am_new,
                    out=(sample, prob, ent, accepted, None))
        # noise, re-noising, the frozen rows' argmax and the stopping update, one launch
        uniform_update(sample, accepted, am_new, ent, V, k_noise, stop, canvas, argmax, done)
        if step_times is not None:
            e1.record()
        done_host.copy_(done)                  # the one host read of the step
        if step_times is not None:
            step_times.append(e0.elapsed_time(e1))
        n_done = int(done_host.sum())
        if trace is not None:
            trace.append((steps, n_done))
        if n_done == B:
            break
    return argmax, steps
