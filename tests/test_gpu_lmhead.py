"""GPU parity of the LM head fused with the statistics pass
(dllm_lm_head_stats, tcgen05 tensor cores) against the oracle: the optional
logits output within the fp32-accumulation bound, and x0 / prob / entropy of
the logits -- x0 exact except where the oracle's two best logits are closer
than that bound (then either is right), prob / entropy within the fp32
statistics tolerance widened by the logits' own accumulation error -- over
ragged token and vocabulary tiles, suppressed ids, Gumbel-max sampling, and
the LLaDA-8B LM head shape (d = 4096, V = 126464)."""
import numpy as np
import pytest
import torch

import dllm_workloads as W
import oracle
from gpu_helpers import TOL

pytestmark = pytest.mark.gpu


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def oracle_logits(h, w, chunk=8192):
    return np.concatenate([oracle.lm_head_logits(h, w[c:c + chunk]) for c in range(0, w.shape[0], chunk)], axis=1)


def accumulation_bound(h, w, chunk=8192):
    """|fp32 sum - exact| <= d 2^-23 sum_k |h_k w_k| (any summation order)."""
    ha = np.abs((h.astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
    out = []
    for c in range(0, w.shape[0], chunk):
        wa = np.abs((w[c:c + chunk].astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
        out.append(ha @ wa.T)
    return np.concatenate(out, axis=1) * h.shape[1] * 2.0**-23


def check(cs, h, w, temperature=0.0, key=0, suppress=(), want_logits=True):
    T, V = h.shape[0], w.shape[0]
    logits = torch.empty((T, V), device="cuda") if want_logits else None
    x0, prob, ent = cs.lm_head_stats(dev_bf16(h), dev_bf16(w), temperature=temperature, key=key,
                                     suppress_ids=suppress, logits=logits)
    torch.cuda.synchronize()
    z = oracle_logits(h, w)
    bound = accumulation_bound(h, w)
    if want_logits:
        err = np.abs(logits.cpu().numpy().astype(np.float64) - z)
        assert np.all(err <= bound + 1e-30), float((err - bound).max())
    ox0, op, oe = oracle.token_stats(z, dtype="f32", temperature=temperature, key=key, suppress_ids=suppress)
    gx0 = x0.cpu().numpy()
    for t in np.flatnonzero(gx0 != ox0):
        # a near-tie: the two candidates' scores differ by less than the logits' error
        zt = z[t].astype(np.float64)
        if temperature == 0.0:
            assert abs(zt[gx0[t]] - zt[ox0[t]]) <= bound[t, gx0[t]] + bound[t, ox0[t]], (t, gx0[t], ox0[t])
        else:
            s_g = oracle.gumbel_score(z[t, gx0[t]], temperature, key, t, gx0[t])
            s_o = oracle.gumbel_score(z[t, ox0[t]], temperature, key, t, ox0[t])
            assert abs(float(s_g) - float(s_o)) <= 2 * (bound[t, gx0[t]] + bound[t, ox0[t]]) + 1e-6, t
    assert (gx0 != ox0).sum() <= max(1, T // 50)
    # prob / entropy: the fp32 statistics tolerance plus what the logits'
    # own fp32 accumulation moves them by -- a random walk over d terms whose
    # partial sums stay within the row's largest |logit|: about
    # sqrt(d) 2^-24 max|z| in every exponent, twice that in prob or entropy.
    d = h.shape[1]
    rtol, atol = TOL["f32"]
    row_tol = rtol + 2.0 * np.sqrt(d) * 2.0**-24 * np.abs(z).max(axis=1)
    same = gx0 == ox0
    gp, ge = prob.cpu().numpy().astype(np.float64), ent.cpu().numpy().astype(np.float64)
    bad_p = np.abs(gp - op) > row_tol * np.abs(op) + atol
    bad_e = np.abs(ge - oe) > row_tol * np.abs(oe) + atol
    assert not (bad_p & same).any() and not (bad_e & same).any(), (
        np.flatnonzero(bad_p | bad_e), gp[bad_p | bad_e], op[bad_p | bad_e], row_tol[bad_p | bad_e])
    return gx0


@pytest.mark.parametrize("T,d,V", [(5, 64, 300), (130, 128, 1000), (32, 512, 5003), (257, 256, 33000)])
def test_small_shapes(cs, T, d, V):
    h, w, targets = W.lm_head_inputs(T + V, T, d, V)
    x0 = check(cs, h, w)
    assert np.mean(x0 == targets) > 0.9


def test_suppressed_ids_and_sampling(cs):
    T, d, V = 64, 256, 4096
    h, w, targets = W.lm_head_inputs(3, T, d, V, boost=3.0)
    sup = sorted(set(targets[:10].tolist()))          # the boosted targets of ten tokens
    x0 = check(cs, h, w, suppress=sup)
    assert not np.isin(x0, sup).any()
    check(cs, h, w, temperature=0.8, key=77, want_logits=False)
    check(cs, h, w, temperature=1.0, key=78, suppress=sup, want_logits=False)


def test_llada_lm_head_shape(cs):
    T, d, V = 32, 4096, 126464
    h, w, targets = W.lm_head_inputs(11, T, d, V)
    x0 = check(cs, h, w, suppress=[126336], want_logits=False)
    assert np.mean(x0 == targets) > 0.9


def test_argument_checks(cs):
    h = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")   # d not a multiple of 64
    w = torch.zeros((8, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cs.DllmError):
        cs.lm_head_stats(h, w)
