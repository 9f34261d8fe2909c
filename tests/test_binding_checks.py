"""The Python binding rejects, before any call into the library, the device
tensors a kernel would index out of bounds: a wrong element count, dtype,
layout or device, and a canvas too small for the columns a step updates.
Host logic only (CPU tensors stand in for device tensors here)."""
import importlib.util
import os

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _built_package():
    spec = importlib.util.spec_from_file_location("_b", os.path.join(ROOT, "commit_step_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()      # the package refuses to import without its library
    import commit_step_gb300

    return commit_step_gb300


cs = _built_package()

CPU = torch.device("cpu")


def test_arg_accepts_the_right_tensor_and_none():
    cs._arg(torch.zeros(6, dtype=torch.int32), "x0", 6, cs._I32, CPU)
    cs._arg(torch.zeros((2, 3), dtype=torch.bool), "commit", 6, cs._MASK, CPU)
    cs._arg(None, "counts", 6, cs._I32, CPU)


@pytest.mark.parametrize("bad", [
    torch.zeros(5, dtype=torch.int32),                 # too few elements
    torch.zeros(7, dtype=torch.int32),                 # too many
    torch.zeros(6, dtype=torch.int64),                 # wrong dtype
    torch.zeros(12, dtype=torch.int32)[::2],           # not contiguous
    [0] * 6,                                           # not a tensor
])
def test_arg_rejects(bad):
    with pytest.raises((ValueError, TypeError)):
        cs._arg(bad, "x0", 6, cs._I32, CPU)


def test_arg_rejects_another_device():
    with pytest.raises(ValueError):
        cs._arg(torch.zeros(6, dtype=torch.int32), "x0", 6, cs._I32, torch.device("cuda", 0))


def test_canvas_must_hold_the_updated_columns():
    cs._canvas_check(torch.zeros((2, 72), dtype=torch.int32), 2, 32, 40, CPU)
    for canvas, off in ((torch.zeros((2, 71), dtype=torch.int32), 40),    # one column short
                        (torch.zeros((1, 96), dtype=torch.int32), 0),     # one row short
                        (torch.zeros((2, 96), dtype=torch.int64), 0),     # wrong dtype
                        (torch.zeros((96, 2), dtype=torch.int32).t(), 0),  # columns not unit-stride
                        (torch.zeros((2, 96), dtype=torch.int32), -1)):   # negative offset
        with pytest.raises(ValueError):
            cs._canvas_check(canvas, 2, 32, off, CPU)


def test_fused_step_arguments():
    B, L = 2, 8
    ok = dict(k=torch.zeros(B, dtype=torch.int32), cand=torch.zeros((B, L), dtype=torch.uint8),
              canvas=torch.zeros((B, 16), dtype=torch.int32), canvas_offset=8,
              counts=torch.zeros((B, 3), dtype=torch.int32))
    cs._fused_args(B, L, CPU, cs.RULE_TOPK, False, **ok, commit=torch.zeros((B, L), dtype=torch.uint8),
                   check_commit=True)
    with pytest.raises(ValueError):   # counts holds 3 ints per batch row
        cs._fused_args(B, L, CPU, cs.RULE_TOPK, False, **{**ok, "counts": torch.zeros(B, dtype=torch.int32)})
    with pytest.raises(ValueError):   # a rule writes a commit mask
        cs._fused_args(B, L, CPU, cs.RULE_THRESHOLD, False, **ok, commit=None, check_commit=True)
    with pytest.raises(ValueError):   # the edit rule writes an edit mask
        cs._fused_args(B, L, CPU, cs.RULE_NONE, True, **ok, edit_mask=None)
    with pytest.raises(ValueError):   # k holds one count per batch row
        cs._fused_args(B, L, CPU, cs.RULE_TOPK, False, **{**ok, "k": torch.zeros(B + 1, dtype=torch.int32)})


def test_stats_outputs():
    T = 12
    good = (torch.zeros(T, dtype=torch.int32), torch.zeros((3, 4), dtype=torch.float32), torch.zeros(T))
    cs._stats_out(good, T, CPU)
    with pytest.raises(ValueError):   # prob as float64
        cs._stats_out((good[0], torch.zeros(T, dtype=torch.float64), good[2]), T, CPU)
    with pytest.raises(ValueError):   # x0 one short
        cs._stats_out((torch.zeros(T - 1, dtype=torch.int32), good[1], good[2]), T, CPU)


def test_noalloc_tensors_must_be_on_the_current_device():
    """dllm_token_stats_noalloc takes its scratch address and launch limits
    from the current device: the binding refuses tensors or a stream elsewhere."""
    cs._on_current_device(torch.device("cuda", 1), 1)
    cs._on_current_device(torch.device("cuda", 0), 0, stream_device=0)
    with pytest.raises(ValueError):
        cs._on_current_device(torch.device("cuda", 1), 0)
    with pytest.raises(ValueError):
        cs._on_current_device(torch.device("cpu"), 0)
    with pytest.raises(ValueError):
        cs._on_current_device(torch.device("cuda", 0), 0, stream_device=1)
