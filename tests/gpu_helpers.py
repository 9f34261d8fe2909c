"""Helpers of the GPU parity tests: moving workloads to the device and the
tolerances of the statistics.

Tolerances (prob and entropy against the fp64 oracle): fp32 logits 1e-5
relative + 1e-6 absolute; bf16 logits 2e-3 relative (the bf16 inputs are exact
in fp32, so only the fp32 accumulation differs; 2e-3 is the stated bound).
x0, masks, schedules and ranges are compared bit for bit.
"""
import numpy as np
import torch

TOL = {"f32": (1e-5, 1e-6), "bf16": (2e-3, 1e-6)}


def to_device(logits: np.ndarray, dtype: str, device="cuda", stride=None):
    """(rows, V) host array -> device tensor; bf16 inputs are uint16 bit arrays.

    With ``stride`` > V the rows live in a wider buffer (padding filled with
    NaN bits so a kernel that reads past V would be caught)."""
    rows, V = logits.shape
    if dtype == "bf16":
        src = torch.from_numpy(np.ascontiguousarray(logits).view(np.int16))
    else:
        src = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32))
    if stride is None or stride == V:
        t = src.to(device)
    else:
        wide = torch.full((rows, stride), -1, dtype=src.dtype)    # int16 -1 = bf16 NaN bits
        if dtype == "f32":
            wide.fill_(float("nan"))
        wide[:, :V] = src
        t = wide.to(device)[:, :V]
    return t.view(torch.bfloat16) if dtype == "bf16" else t


def assert_stats_close(dtype, got_prob, got_ent, want_prob, want_ent, what=""):
    rtol, atol = TOL[dtype]
    gp = np.asarray(got_prob, dtype=np.float64).reshape(-1)
    ge = np.asarray(got_ent, dtype=np.float64).reshape(-1)
    wp = np.asarray(want_prob).reshape(-1)
    we = np.asarray(want_ent).reshape(-1)
    bad_p = ~np.isclose(gp, wp, rtol=rtol, atol=atol)
    bad_e = ~np.isclose(ge, we, rtol=rtol, atol=atol)
    if bad_p.any() or bad_e.any():
        i = int(np.flatnonzero(bad_p | bad_e)[0])
        raise AssertionError(f"{what}: {int(bad_p.sum())} prob / {int(bad_e.sum())} entropy outside "
                             f"tolerance; first row {i}: prob {gp[i]!r} vs {wp[i]!r}, entropy {ge[i]!r} vs {we[i]!r}")
