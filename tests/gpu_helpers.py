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


def mask_mismatch_rows(rule, got, cand, scores, params, dtype):
    """Batch rows where the GPU's commit mask differs from the oracle rule
    evaluated on the oracle's own statistics (rounded to fp32), split into
    rows whose deciding comparison lies within the statistics tolerance (a
    near-tie or a score within tolerance of the bound: either answer is
    correct) and rows with no such excuse.  Returns (unexplained, ambiguous).
    """
    import oracle

    rtol, atol = TOL[dtype]
    s32 = np.asarray(scores, dtype=np.float32)
    if rule == "threshold":
        want = oracle.threshold_transfer(s32, cand, params["tau"], params["strict"])
    elif rule == "topk":
        want = oracle.topk_transfer(s32, cand, params["k"])
    elif rule == "factor":
        want = oracle.factor_transfer(s32, cand, params["factor"])
    else:
        want = oracle.entropy_bound_transfer(s32, cand, params["gamma"])
    unexplained, ambiguous = [], []
    for b in np.flatnonzero((want != got).any(axis=1)):
        c = np.flatnonzero(cand[b])
        v = np.asarray(scores[b], dtype=np.float64)[c]
        band = rtol * np.abs(v) + atol
        amb = False
        if rule == "threshold":
            tau = params["tau"]
            amb = bool(np.any(np.abs(v - tau) <= band))
            top = np.sort(v)[::-1]
            if len(top) > 1 and top[0] - top[1] <= 2 * band.max():
                amb = True
        else:
            order = np.argsort(-v if rule != "entropy_bound" else v, kind="stable")
            sv = v[order]
            sb = band[order]
            gaps = np.abs(np.diff(sv)) <= sb[:-1] + sb[1:]
            if rule == "topk":
                k = int(params["k"][b]) if np.ndim(params["k"]) else int(params["k"])
                amb = 0 < k < len(sv) and bool(gaps[k - 1])
            elif rule == "factor":
                lhs = (np.arange(len(sv)) + 1) * (1 - sv)
                amb = bool(np.any(np.abs(lhs - params["factor"]) <= (np.arange(len(sv)) + 1) * sb)) or bool(gaps.any())
            else:
                pref = np.concatenate([[0.0], np.cumsum(sv)[:-1]])
                amb = bool(np.any(np.abs(pref - params["gamma"]) <= np.cumsum(sb))) or bool(gaps.any())
        (ambiguous if amb else unexplained).append(int(b))
    return unexplained, ambiguous
