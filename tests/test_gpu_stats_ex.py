"""GPU parity of the extended statistics (dllm_token_stats_ex and the fused
step's dllm_stats_ex) against the oracle's orc_token_stats_ex.

Scaled logits z' = fp32(z * logit_scale), the margin confidence and the
greedy argmax beside a Gumbel-max sample.  x0 and argmax bit-exact; prob and
entropy within the tolerances of gpu_helpers; the margin within the same
relative tolerance of the two probabilities it subtracts.  Shapes cover the
cluster path (few rows) and the persistent path (many rows, rows split across
CTAs), ragged tails, ties, NaN, infinities and suppressed ids.
"""
import numpy as np
import pytest
import torch

import oracle
from dllm_workloads import f32_to_bf16_bits
from gpu_helpers import TOL, assert_stats_close, to_device

pytestmark = pytest.mark.gpu


def host_logits(z, dtype):
    return z if dtype == "f32" else f32_to_bf16_bits(z)


def check_ex(cs, host, dtype, temperature=0.0, key=0, scale=1.0, suppress=(), what=""):
    rows, V = host.shape
    per16 = 4 if dtype == "f32" else 8
    stride = -(-V // per16) * per16
    dev = to_device(host, dtype, stride=stride if stride != V else None)
    x0, prob, ent, mar, am = cs.token_stats_ex(dev, temperature=temperature, key=key, suppress_ids=suppress,
                                               logit_scale=scale)
    torch.cuda.synchronize()
    ox0, op, oe, om, oam = oracle.token_stats_ex(host, dtype=dtype, temperature=temperature, key=key,
                                                 logit_scale=scale, suppress_ids=suppress)
    g = lambda t: t.cpu().numpy().reshape(-1)
    gx0, gam = g(x0), g(am)
    bad = np.flatnonzero(gx0 != ox0)
    assert bad.size == 0, f"{what}: x0 differs in {bad.size} rows, first {bad[:4]}: {gx0[bad[:4]]} vs {ox0[bad[:4]]}"
    bad = np.flatnonzero(gam != oam)
    assert bad.size == 0, f"{what}: argmax differs in {bad.size} rows, first {bad[:4]}: {gam[bad[:4]]} vs {oam[bad[:4]]}"
    assert_stats_close(dtype, g(prob), g(ent), op, oe, what)
    rtol, atol = TOL[dtype]
    p2 = op - om                                   # the runner-up's probability
    gm = g(mar).astype(np.float64)
    bad = np.flatnonzero(np.abs(gm - om) > rtol * (op + np.abs(p2)) + atol)
    assert bad.size == 0, f"{what}: margin off in {bad.size} rows, first {bad[:4]}: {gm[bad[:4]]} vs {om[bad[:4]]}"
    return gx0, g(prob), g(ent), gm, gam


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scale", [1.0, 1 / 0.4, 0.75])
@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_cluster_path(cs, dtype, scale, temperature):
    rng = np.random.default_rng(int(scale * 1000) + int(temperature * 7))
    V = 33_001
    z = (rng.standard_normal((24, V)) * 2.5).astype(np.float32)
    z[0, 5] = z[0, 30_000] = 9.0                  # exact tie of the max: margin 0
    z[1, 100:110] = 7.0                           # a run of equal maxima
    z[2, ::5] = np.nan
    z[3, 11] = np.inf
    check_ex(cs, host_logits(z, dtype), dtype, temperature=temperature, key=77, scale=scale, suppress=[3, 12],
             what=f"cluster {dtype} s={scale:.3f} t={temperature}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_persistent_path_split_rows(cs, dtype):
    rng = np.random.default_rng(5)
    V = 150_001 if dtype == "bf16" else 90_001
    z = (rng.standard_normal((300, V)) * 1.5).astype(np.float32)
    z[7, 0] = z[7, V - 1] = 8.0                   # the tie straddles CTAs
    host = host_logits(z, dtype)
    for t, s in ((0.0, 1.25), (0.7, 1.0), (1.0, 2.5)):
        check_ex(cs, host, dtype, temperature=t, key=1234, scale=s, suppress=[V - 2],
                 what=f"persistent {dtype} t={t} s={s}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_token_and_uniform_rows(cs, dtype):
    V = 65                                        # 64 suppressed ids (the most a call takes) leave one token
    z = np.zeros((4, V), dtype=np.float32)
    z[1, :] = np.nan
    z[2, 17] = 3.0
    sup = [v for v in range(V) if v != 17]        # the token set is {17}: prob 1, margin 1
    x0, prob, ent, mar, am = check_ex(cs, host_logits(z, dtype), dtype, suppress=sup, what="single token")
    assert np.all(x0 == 17) and np.allclose(prob, 1.0) and np.allclose(mar, 1.0)
    V = 4099
    z = np.zeros((4, V), dtype=np.float32)
    z[1, :] = np.nan                              # uniform limit: margin 0
    z[2, 17] = 3.0
    x0, prob, ent, mar, am = check_ex(cs, host_logits(z, dtype), dtype, scale=3.0, what="uniform rows")
    assert mar[0] == 0.0 and mar[1] == 0.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unit_scale_options_match_the_plain_pass(cs, dtype):
    """Asking for margin/argmax at scale 1 changes no other output."""
    rng = np.random.default_rng(9)
    z = (rng.standard_normal((64, 20_000)) * 3).astype(np.float32)
    dev = to_device(host_logits(z, dtype), dtype)
    for t in (0.0, 0.8):
        a = cs.token_stats(dev, temperature=t, key=5)
        b = cs.token_stats_ex(dev, temperature=t, key=5)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0])
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
        if t == 0.0:
            assert torch.equal(b[4], b[0])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_entropy_bound_on_scaled_statistics(cs, dtype):
    """The uniform-noise step's acceptance: entropy bound over every position,
    on the entropy of z / T, with the categorical sample and the argmax."""
    rng = np.random.default_rng(21)
    B, L, V = 3, 96, 20_008                       # rows a multiple of 16 bytes in both dtypes
    z = (rng.standard_normal((B * L, V)) * 2.0).astype(np.float32)
    z[np.arange(0, B * L, 3), rng.integers(0, V, B * L // 3)] += 9.0   # some confident positions
    host = host_logits(z, dtype)
    dev = to_device(host, dtype).view(B, L, V)
    T = 0.55
    s = float(np.float32(1.0 / T))
    cand = torch.ones((B, L), dtype=torch.uint8, device="cuda")
    margin = torch.empty((B, L), dtype=torch.float32, device="cuda")
    argmax = torch.empty((B, L), dtype=torch.int32, device="cuda")
    x0, prob, ent, commit, _ = cs.commit_step(dev, rule=cs.RULE_ENTROPY_BOUND, gamma=0.1, temperature=1.0, key=31,
                                              cand=cand, logit_scale=s, margin=margin, argmax=argmax)
    torch.cuda.synchronize()
    ox0, op, oe, om, oam = oracle.token_stats_ex(host, dtype=dtype, temperature=1.0, key=31, logit_scale=s)
    assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
    assert np.array_equal(argmax.cpu().numpy().reshape(-1), oam)
    assert_stats_close(dtype, prob.cpu().numpy(), ent.cpu().numpy(), op, oe, "fused scaled")
    # the rule decides on the GPU's fp32 entropy, on both sides
    want = oracle.entropy_bound_transfer(ent.cpu().numpy(), np.ones((B, L), np.uint8), 0.1)
    assert np.array_equal(commit.cpu().numpy(), want)
    assert commit.cpu().numpy().sum(axis=1).min() >= 1


def test_scale_validation(cs):
    dev = torch.zeros((1, 2, 64), dtype=torch.float32, device="cuda")
    for bad in (0.0, -1.0, 300.0, float("nan")):
        with pytest.raises(cs.DllmError):
            cs.token_stats_ex(dev, logit_scale=bad)
