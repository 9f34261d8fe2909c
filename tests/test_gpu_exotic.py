"""GPU parity of the statistics on rows with extreme logits, against the
oracle's reading ("dLLM block decoding", What mlx-arsenal ships: token_stats
is NaN-safe): a NaN has no mass, +inf entries share the mass, and every
finite logit, however large, takes the ordinary softmax.

Two kinds of rows:
  * rows the streaming pass does not finish itself (largest logit beyond
    about 1.8e8 in magnitude, +inf, or nothing above -2^100): one warp
    recomputes them from the logits;
  * rows it does finish at large offsets (1e3 .. 1.5e8) and rows whose
    threads see very negative maxima: the exponent references must keep
    the sums exact there.
Both grid kinds (a cluster per row; the persistent grid with rows split
across CTAs), both dtypes, greedy and Gumbel selection, scaled logits with
the margin, and the fused threshold rule on the emitted statistics.
"""
import numpy as np
import pytest
import torch

import oracle
from dllm_workloads import f32_to_bf16_bits
from gpu_helpers import TOL, assert_stats_close, to_device

pytestmark = pytest.mark.gpu


def extreme_rows(V, seed):
    rng = np.random.default_rng(seed)
    f = np.float32

    def base():
        return (rng.standard_normal(V) * 2).astype(np.float32)

    rows = []
    r = base(); r[[5, 9]] = [1e38, 1e37]; rows.append(r)                 # the larger takes all the mass
    r = np.full(V, np.nan, np.float32); r[0] = -1e31; rows.append(r)     # one finite logit among NaNs
    r = base(); r[[3, V // 2, V - 1]] = 3.0e38; r[7] = -3.0e38; rows.append(r)   # three maxima share
    r = base(); r[[10, 20]] = np.inf; rows.append(r)                     # the +inf entries share
    rows.append(np.full(V, np.nan, np.float32))                          # no mass: the uniform limit
    r = np.full(V, -np.inf, np.float32); r[V // 3] = np.nan; rows.append(r)
    rows.append(np.full(V, f(-2.0 ** 100), np.float32))                  # equal finite logits share
    r = base(); r[::7] = -2e30; r[4] = f(-2.0 ** 101); rows.append(r)    # very negative logits: no mass
    rows.append((f(1e9) - f(64) * rng.integers(0, 4, V)).astype(np.float32))   # gaps of the fp32 spacing
    rows.append((f(-3e8) - f(32) * rng.integers(0, 3, V)).astype(np.float32))
    # rows the streaming pass finishes itself, at large offsets
    rows.append((base() + f(1e3)).astype(np.float32))
    rows.append((base() + f(1e6)).astype(np.float32))
    rows.append((base() - f(1e7)).astype(np.float32))
    rows.append((base() * 40 + f(1.5e8)).astype(np.float32))
    r = base(); r[: V // 2] = f(-1e10); rows.append(r)                  # half the threads' maxima near -1e10
    r = base(); r[V // 4: 3 * V // 4] = f(-3.0e38); rows.append(r)
    return np.stack(rows)


def host_of(z, dtype):
    return z if dtype == "f32" else f32_to_bf16_bits(z)


def padded_stride(V, dtype):
    per16 = 4 if dtype == "f32" else 8
    s = -(-V // per16) * per16
    return s if s != V else None


def check_stats(cs, host, dtype, temperature, key, sup, what):
    dev = to_device(host, dtype, stride=padded_stride(host.shape[1], dtype))
    x0, prob, ent = cs.token_stats(dev, temperature=temperature, key=key, suppress_ids=sup)
    torch.cuda.synchronize()
    ox0, op, oe = oracle.token_stats(host, dtype=dtype, temperature=temperature, key=key, suppress_ids=sup)
    gx0 = x0.cpu().numpy().reshape(-1)
    bad = np.flatnonzero(gx0 != ox0)
    assert bad.size == 0, f"{what}: x0 differs in rows {bad[:6].tolist()}: {gx0[bad[:6]]} vs {ox0[bad[:6]]}"
    gp, ge = prob.cpu().numpy(), ent.cpu().numpy()
    assert np.all(np.isfinite(gp)) and np.all(np.isfinite(ge)), f"{what}: non-finite statistics"
    assert_stats_close(dtype, gp, ge, op, oe, what)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("temperature", [0.0, 0.8, 100.0])
def test_extreme_rows_cluster_grid(cs, dtype, temperature):
    """Few long rows: one thread-block cluster per row."""
    z = extreme_rows(40_003, 1)
    check_stats(cs, host_of(z, dtype), dtype, temperature, 0xC0FFEE, [2, 40_002],
                f"cluster {dtype} t={temperature}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("temperature", [0.0, 0.8])
def test_extreme_rows_persistent_grid(cs, dtype, temperature):
    """Many rows (the persistent grid, rows split across CTAs), the extreme
    rows among ordinary ones."""
    V = 50_001
    rng = np.random.default_rng(2)
    z = (rng.standard_normal((320, V)) * 2).astype(np.float32)
    ex = extreme_rows(V, 3)
    at = np.sort(rng.choice(z.shape[0], ex.shape[0], replace=False))
    z[at] = ex
    check_stats(cs, host_of(z, dtype), dtype, temperature, 99, [V - 3], f"persistent {dtype} t={temperature}")


def test_extreme_rows_short(cs):
    """Short rows (V = 37: one vector per thread or none, the tail path)."""
    z = extreme_rows(37, 4)
    for t in (0.0, 0.5):
        check_stats(cs, z, "f32", t, 5, [1], f"short t={t}")


@pytest.mark.parametrize("scale", [0.5, 2.5, 256.0])
@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_extreme_rows_scaled_with_margin(cs, scale, temperature):
    """Scaled logits z' = fp32(z s) (a product beyond the fp32 range is inf),
    the margin and the argmax beside a sample.  s = 256 with suppressed ids
    also checks that the suppressed entries' exponent stays finite."""
    for V, seed in ((40_003, 6), (997, 7)):
        host = extreme_rows(V, seed)
        dev = to_device(host, "f32", stride=padded_stride(V, "f32"))
        sup = [0, 11, V - 1]
        x0, prob, ent, mar, am = cs.token_stats_ex(dev, temperature=temperature, key=31, suppress_ids=sup,
                                                   logit_scale=scale)
        torch.cuda.synchronize()
        ox0, op, oe, om, oam = oracle.token_stats_ex(host, temperature=temperature, key=31, logit_scale=scale,
                                                     suppress_ids=sup)
        g = lambda t: t.cpu().numpy().reshape(-1)
        what = f"scaled V={V} s={scale} t={temperature}"
        assert np.array_equal(g(x0), ox0), what
        assert np.array_equal(g(am), oam), what
        assert_stats_close("f32", g(prob), g(ent), op, oe, what)
        rtol, atol = TOL["f32"]
        gm = g(mar).astype(np.float64)
        bad = np.flatnonzero(np.abs(gm - om) > rtol * (op + np.abs(op - om)) + atol)
        assert bad.size == 0, f"{what}: margin off in rows {bad[:6].tolist()}: {gm[bad[:6]]} vs {om[bad[:6]]}"


@pytest.mark.parametrize("scale", [0.5, 256.0])
def test_extreme_rows_scaled_plain_greedy(cs, scale):
    """Scaled statistics without the margin or a sample: the plain greedy
    mode's streaming loop (one running max per warp, the first vector of a
    new warp max looked for only where it is held), on the extreme rows,
    rows split across CTAs and the ties they hold; x0 bit for bit."""
    for V, rows, seed in ((40_003, 1, 6), (997, 40, 7)):
        host = np.tile(extreme_rows(V, seed), (rows, 1))
        dev = to_device(host, "f32", stride=padded_stride(V, "f32"))
        sup = [0, 11, V - 1]
        x0, prob, ent, mar, am = cs.token_stats_ex(dev, suppress_ids=sup, logit_scale=scale, margin=None,
                                                   argmax=None)
        torch.cuda.synchronize()
        assert mar is None and am is None
        ox0, op, oe, _, _ = oracle.token_stats_ex(host, logit_scale=scale, suppress_ids=sup)
        g = lambda t: t.cpu().numpy().reshape(-1)
        what = f"plain scaled V={V} s={scale}"
        assert np.array_equal(g(x0), ox0), what
        assert_stats_close("f32", g(prob), g(ent), op, oe, what)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_extreme_rows_fused_threshold(cs, dtype):
    """The fused step decides on the statistics the exact path emitted: the
    masks equal the oracle's threshold rule on them, bit for bit."""
    z = extreme_rows(20_011, 8)
    L = 8
    B = z.shape[0] // L
    host = host_of(z, dtype)
    cand = (np.random.default_rng(9).random((B, L)) < 0.7).astype(np.uint8)
    cand[:, 0] = 1
    dev = to_device(host, dtype, stride=padded_stride(z.shape[1], dtype)).view(B, L, -1)
    x0, prob, ent, commit, _ = cs.commit_step(dev, rule=1, tau=0.6, strict=True, suppress_ids=[3],
                                              cand=torch.from_numpy(cand).cuda())
    torch.cuda.synchronize()
    ox0, op, oe = oracle.token_stats(host, dtype=dtype, suppress_ids=[3])
    assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
    gp = prob.cpu().numpy()
    assert_stats_close(dtype, gp, ent.cpu().numpy(), op, oe, f"fused {dtype}")
    want = oracle.threshold_transfer(gp.reshape(B, L), cand, 0.6, True)
    assert np.array_equal(commit.cpu().numpy(), want)
