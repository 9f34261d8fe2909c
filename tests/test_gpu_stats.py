"""GPU parity of the statistics pass (dllm_token_stats) against the oracle.

x0 bit-exact; prob and entropy within the tolerances of gpu_helpers.  Shapes
span many units per row, rows shared by several CTAs, ragged tails (V not a
multiple of the 16-byte vector), padded row strides, suppressed ids, NaN and
infinite logits, exact ties, and both greedy and Gumbel-max selection.
"""
import numpy as np
import pytest
import torch

import oracle
from dllm_workloads import f32_to_bf16_bits
from gpu_helpers import assert_stats_close, to_device

pytestmark = pytest.mark.gpu


def run_case(cs, z_host, dtype, temperature=0.0, key=0, suppress=(), stride=None):
    rows, V = z_host.shape
    dev = to_device(z_host, dtype, stride=stride)
    x0, prob, ent = cs.token_stats(dev, temperature=temperature, key=key, suppress_ids=suppress)
    torch.cuda.synchronize()
    ox0, op, oe = oracle.token_stats(z_host, dtype=dtype, temperature=temperature, key=key, suppress_ids=suppress)
    gx0 = x0.cpu().numpy().reshape(-1)
    mism = np.flatnonzero(gx0 != ox0)
    assert mism.size == 0, f"x0 differs in {mism.size} rows, first {mism[:5]}: gpu {gx0[mism[:5]]} oracle {ox0[mism[:5]]}"
    assert_stats_close(dtype, prob.cpu().numpy(), ent.cpu().numpy(), op, oe, f"{dtype} V={V} t={temperature}")
    return gx0, prob.cpu().numpy().reshape(-1), ent.cpu().numpy().reshape(-1)


def gen(rng, rows, V, scale=3.0):
    return (rng.standard_normal((rows, V)) * scale).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 3, 8, 100, 4096, 4099, 33000])
def test_greedy_shapes(cs, dtype, V):
    rng = np.random.default_rng(100 + V)
    z = gen(rng, 37, V)
    host = z if dtype == "f32" else f32_to_bf16_bits(z)
    per16 = 4 if dtype == "f32" else 8
    stride = -(-V // per16) * per16
    run_case(cs, host, dtype, stride=stride if stride != V else None)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_few_long_rows_split_across_ctas(cs, dtype):
    rng = np.random.default_rng(7)
    z = gen(rng, 3, 1_000_003 if dtype == "bf16" else 600_001, scale=2.0)
    host = z if dtype == "f32" else f32_to_bf16_bits(z)
    V = host.shape[1]
    per16 = 4 if dtype == "f32" else 8
    run_case(cs, host, dtype, stride=-(-V // per16) * per16)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_persistent_path_rows_split_across_ctas(cs, dtype):
    """Too many rows for one cluster per row: the persistent grid, with rows
    shared by two or three CTAs and combined through the workspace."""
    rng = np.random.default_rng(71)
    V = 200_003 if dtype == "bf16" else 100_001
    z = gen(rng, 200, V, scale=1.5)
    host = z if dtype == "f32" else f32_to_bf16_bits(z)
    per16 = 4 if dtype == "f32" else 8
    run_case(cs, host, dtype, suppress=[3, V - 1], stride=-(-V // per16) * per16)
    run_case(cs, host, dtype, temperature=0.9, key=99, stride=-(-V // per16) * per16)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_suppress_nan_inf_and_ties(cs, dtype):
    rng = np.random.default_rng(8)
    V = 5000
    z = gen(rng, 12, V)
    z[0, 17] = z[0, 4000] = 50.0                  # exact tie: lower id wins
    z[1, :] = np.nan                              # all NaN: uniform limit
    z[2, ::3] = np.nan                            # scattered NaN
    z[3, 10] = np.inf                             # +inf dominates
    z[3, 20] = np.inf
    z[4, :] = -np.inf
    z[4, 999] = 0.0                               # a single finite logit
    z[5, 7] = 1e38                                # above the 2^100 clamp
    z[6, :] = 0.0                                 # flat row
    z[7, 123] = 80.0                              # suppressed argmax
    z[8, :] = -3e30                               # below the -2^100 clamp: uniform limit
    host = z if dtype == "f32" else f32_to_bf16_bits(z)
    sup = [123, 0, 4999, 2500]
    x0, p, h = run_case(cs, host, dtype, suppress=sup)
    assert x0[0] == 17 and x0[7] != 123
    assert x0[1] == 1                              # first id not suppressed
    assert not set(x0.tolist()) & set(sup)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [8, 1001, 152064])
def test_gumbel_matches_oracle(cs, dtype, V):
    rng = np.random.default_rng(9 + V)
    rows = 24 if V > 100000 else 64
    z = gen(rng, rows, V, scale=1.0)
    z[:, rng.integers(0, V, rows)] += 6.0
    host = z if dtype == "f32" else f32_to_bf16_bits(z)
    per16 = 4 if dtype == "f32" else 8
    stride = -(-V // per16) * per16
    for t, key in ((0.7, 0x123456789ABCDEF), (1.5, 42), (0.05, 2**64 - 1)):
        run_case(cs, host, dtype, temperature=t, key=key, suppress=[1, V - 1] if V > 2 else [],
                 stride=stride if stride != V else None)


def test_gumbel_sampling_frequency(cs):
    """Gumbel-max over many rows of the same logits samples softmax(z/t)."""
    import scipy.special
    import scipy.stats

    z = np.array([1.0, 0.0, -0.5, 2.0, 0.25, -1.0, 1.5, 0.0], dtype=np.float32)
    n = 200_000
    rows = np.ascontiguousarray(np.broadcast_to(z, (n, 8)))
    x0, _, _ = cs.token_stats(torch.from_numpy(rows).cuda(), temperature=0.7, key=5)
    counts = np.bincount(x0.cpu().numpy(), minlength=8)
    expect = scipy.special.softmax(z.astype(np.float64) / 0.7) * n
    assert scipy.stats.chisquare(counts, expect).pvalue > 1e-4


def test_batched_3d_and_repeat_calls_reuse_workspace(cs):
    rng = np.random.default_rng(10)
    B, L, V = 4, 33, 2056
    z = gen(rng, B * L, V)
    dev = torch.from_numpy(z).cuda().view(B, L, V)
    ox0, op, oe = oracle.token_stats(z)
    for _ in range(3):  # the workspace must come back zeroed after each call
        x0, p, h = cs.token_stats(dev, suppress_ids=[5])
        ox0, op, oe = oracle.token_stats(z, suppress_ids=[5])
        assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
        assert_stats_close("f32", p.cpu().numpy(), h.cpu().numpy(), op, oe)


def test_invalid_arguments_raise(cs):
    z = torch.zeros(4, 64, device="cuda")
    with pytest.raises(cs.DllmError):
        cs.token_stats(z, temperature=-1.0)
    with pytest.raises(cs.DllmError):
        cs.token_stats(z, suppress_ids=[64])
    with pytest.raises(cs.DllmError):
        cs.token_stats(z, suppress_ids=list(range(64)))          # empty token set
    with pytest.raises(cs.DllmError):
        cs.token_stats(z, suppress_ids=list(range(65)))          # too many
    zz = torch.zeros(4, 70, device="cuda")[:, 1:]                # misaligned rows
    with pytest.raises(cs.DllmError):
        cs.token_stats(zz)
    ws = cs.workspace(4, 1, 64, 0, z.device)
    assert cs.workspace_fault(ws) == 0


# Shapes that land on each unit size of the streaming loop (units of 1024,
# 512 and 256 vectors: 4, 2 or 1 vectors per consumer thread), on the
# cluster grid (8 rows: a cluster of 16 CTAs per row, a slice of 1200, 600 or
# 300 vectors per CTA) and on the persistent grid (600 rows dealt to the CTAs
# in unit ranges that cross rows), each with a ragged last unit.
UNIT_SHAPES = [  # rows, vectors per row
    (8, 19_200), (8, 9_600), (8, 4_800),
    (600, 4_000), (600, 2_400), (600, 1_000),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", UNIT_SHAPES, ids=[f"T{t}nvec{n}" for t, n in UNIT_SHAPES])
@pytest.mark.parametrize("temperature", [0.0, 0.8])
def test_every_unit_size(cs, dtype, shape, temperature):
    rows, nvec = shape
    V = nvec * (8 if dtype == "bf16" else 4)
    rng = np.random.default_rng(rows * 7 + nvec)
    z = gen(rng, rows, V, scale=2.5)
    z[np.arange(rows), rng.integers(0, V, rows)] += 7.0
    host = z if dtype == "f32" else f32_to_bf16_bits(z)
    run_case(cs, host, dtype, temperature=temperature, key=4242, suppress=[3, V - 5])
