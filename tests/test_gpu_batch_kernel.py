"""GPU parity of the fused step's batch-row kernel: with DLLM_FLAG_INPUTS_READY
and few short batch rows, one thread-block cluster takes a whole batch row,
rank 0 gathers the rows' partials through distributed shared memory and runs
the rule in shared memory.  Checked against the oracle like every fused
path: x0 bit for bit, prob and entropy within the tolerances of gpu_helpers,
masks, canvas and counts bit for bit against the oracle's rule evaluated on
the statistics the GPU emitted ("dLLM block decoding", What mlx-arsenal
ships; Deviations from the references; Token editing (LLaDA2.1))."""
import numpy as np
import pytest
import torch

import oracle
from dllm_workloads import f32_to_bf16_bits
from gpu_helpers import TOL, assert_stats_close, to_device

pytestmark = pytest.mark.gpu

RULE = {"none": 0, "threshold": 1, "topk": 2, "factor": 3, "entropy_bound": 4}


def make(rng, B, L, V, dtype, scale=2.0, peak=9.0):
    z = (rng.standard_normal((B * L, V)) * scale).astype(np.float32)
    z[np.arange(B * L), rng.integers(0, V, B * L)] += rng.uniform(0, peak, B * L).astype(np.float32)
    host = f32_to_bf16_bits(z) if dtype == "bf16" else z
    per16 = 4 if dtype == "f32" else 8
    stride = -(-V // per16) * per16
    dev = to_device(host, dtype, stride=stride if stride != V else None).view(B, L, V)
    return host, dev


def oracle_rule(rule, p, h, cand, params):
    if rule == "threshold":
        return oracle.threshold_transfer(p, cand, params["tau"], params["strict"])
    if rule == "topk":
        return oracle.topk_transfer(p, cand, params["k"])
    if rule == "factor":
        return oracle.factor_transfer(p, cand, params["factor"])
    if rule == "entropy_bound":
        return oracle.entropy_bound_transfer(h, cand, params["gamma"])
    return np.zeros_like(cand)


SHAPES = [  # B, L, V, dtype
    (1, 32, 126464, "bf16"),     # the LLaDA-8B block step: 16 CTAs of 2 rows
    (2, 40, 30011, "f32"),       # L not a multiple of the cluster: 2 or 3 rows per CTA, ragged V
    (3, 5, 4099, "bf16"),        # L < 16: a cluster of 4, one or two rows per CTA
    (1, 256, 2053, "f32"),       # the largest L: 16 rows per CTA
    (4, 32, 7, "f32"),           # rows shorter than one 16-byte vector (tail only)
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}L{s[1]}V{s[2]}{s[3]}" for s in SHAPES])
@pytest.mark.parametrize("rule", ["threshold", "topk", "factor", "entropy_bound"])
def test_batch_kernel_rules(cs, shape, rule):
    B, L, V, dtype = shape
    rng = np.random.default_rng(B * 1000 + L * 10 + V % 97 + len(rule))
    host, dev = make(rng, B, L, V, dtype)
    cand = (rng.random((B, L)) < 0.6).astype(np.uint8)
    cand[:, 0] = 1
    k = rng.integers(0, L + 2, B).astype(np.int32)
    params = {"tau": 0.7, "strict": bool(L % 2), "k": k, "factor": 1.0, "gamma": 0.3}
    counts = torch.full((B, 3), -1, dtype=torch.int32, device="cuda")
    canvas0 = rng.integers(0, V, (B, L + 11)).astype(np.int32)
    canvas = torch.from_numpy(canvas0.copy()).cuda()
    x0, prob, ent, commit, _ = cs.commit_step(dev, rule=RULE[rule], tau=params["tau"], strict=params["strict"],
                                              k=torch.from_numpy(k).cuda(), factor=1.0, gamma=0.3,
                                              suppress_ids=[V - 1] if V > 1 else [], cand=torch.from_numpy(cand).cuda(),
                                              canvas=canvas, canvas_offset=11, counts=counts, inputs_ready=True)
    torch.cuda.synchronize()
    ox0, op, oe = oracle.token_stats(host, dtype=dtype, suppress_ids=[V - 1] if V > 1 else [])
    gx0, gp, ge = (t.cpu().numpy() for t in (x0, prob, ent))
    assert np.array_equal(gx0.reshape(-1), ox0)
    assert_stats_close(dtype, gp, ge, op, oe, f"{shape} {rule}")
    want = oracle_rule(rule, gp.reshape(B, L), ge.reshape(B, L), cand, params)
    assert np.array_equal(commit.cpu().numpy(), want)
    exp = canvas0.copy()
    exp[:, 11:] = np.where(want.astype(bool), gx0.reshape(B, L), canvas0[:, 11:])
    assert np.array_equal(canvas.cpu().numpy(), exp)
    assert counts.cpu().numpy().tolist() == [[int(cand[b].sum()), int(want[b].sum()), 0] for b in range(B)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_batch_kernel_edit_and_canvas_candidates(cs, dtype):
    """Candidates from the canvas (token == mask id), the edit rule on the
    other positions, the canvas update and the counts, as the editing loop
    uses them, with the inputs-ready launch."""
    rng = np.random.default_rng(5)
    B, L, V, N, off, MASK = 3, 32, 20_000, 80, 30, 19_999
    z = rng.standard_normal((B * L, V)).astype(np.float32)
    tgt = rng.integers(0, 19_000, (B, L))
    for b in range(B):
        for l in range(L):
            z[b * L + l, tgt[b, l]] += 18.0 if l % 3 else 4.0
    host = f32_to_bf16_bits(z) if dtype == "bf16" else z
    dev = to_device(host, dtype).view(B, L, V)
    canvas0 = rng.integers(0, 19_000, (B, N)).astype(np.int32)
    masked = rng.random((B, L)) < 0.5
    canvas0[:, off:off + L][masked] = MASK
    canvas = torch.from_numpy(canvas0.copy()).cuda()
    counts = torch.zeros((B, 3), dtype=torch.int32, device="cuda")
    x0, prob, ent, commit, edit = cs.commit_step(dev, rule=1, tau=0.95, strict=True, suppress_ids=[MASK],
                                                 mask_id=MASK, edit=True, tau_edit=0.9, canvas=canvas,
                                                 canvas_offset=off, counts=counts, inputs_ready=True)
    torch.cuda.synchronize()
    ox0, op, oe = oracle.token_stats(host, dtype=dtype, suppress_ids=[MASK])
    assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
    gp = prob.cpu().numpy()
    assert_stats_close(dtype, gp, ent.cpu().numpy(), op, oe, "edit")
    window = canvas0[:, off:off + L]
    want_c = oracle.threshold_transfer(gp, masked.astype(np.uint8), 0.95, True)
    want_e = oracle.edit_transfer(ox0.reshape(B, L), gp, window, (~masked).astype(np.uint8), 0.9)
    assert np.array_equal(commit.cpu().numpy(), want_c)
    assert np.array_equal(edit.cpu().numpy(), want_e)
    exp = canvas0.copy()
    exp[:, off:off + L] = np.where((want_c | want_e).astype(bool), ox0.reshape(B, L), window)
    assert np.array_equal(canvas.cpu().numpy(), exp)
    assert counts.cpu().numpy().tolist() == [[int(masked[b].sum()), int(want_c[b].sum()), int(want_e[b].sum())]
                                             for b in range(B)]


@pytest.mark.parametrize("scale", [1.0, 2.5])
def test_batch_kernel_gumbel_scaled_margin(cs, scale):
    """Gumbel-max sampling, scaled logits, margin and argmax outputs."""
    rng = np.random.default_rng(int(scale * 10))
    B, L, V = 2, 24, 33_001
    host, dev = make(rng, B, L, V, "bf16")
    cand = torch.ones((B, L), dtype=torch.uint8, device="cuda")
    margin = torch.empty((B, L), dtype=torch.float32, device="cuda")
    argmax = torch.empty((B, L), dtype=torch.int32, device="cuda")
    x0, prob, ent, commit, _ = cs.commit_step(dev, rule=2, k=3, temperature=0.8, key=12345, suppress_ids=[4],
                                              cand=cand, logit_scale=scale, margin=margin, argmax=argmax,
                                              inputs_ready=True)
    torch.cuda.synchronize()
    ox0, op, oe, om, oam = oracle.token_stats_ex(host, dtype="bf16", temperature=0.8, key=12345, logit_scale=scale,
                                                 suppress_ids=[4])
    assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
    assert np.array_equal(argmax.cpu().numpy().reshape(-1), oam)
    gp = prob.cpu().numpy()
    assert_stats_close("bf16", gp, ent.cpu().numpy(), op, oe, "gumbel")
    rtol, atol = TOL["bf16"]
    gm = margin.cpu().numpy().reshape(-1).astype(np.float64)
    assert np.all(np.abs(gm - om) <= rtol * (op + np.abs(op - om)) + atol)
    assert np.array_equal(commit.cpu().numpy(), oracle.topk_transfer(gp, np.ones((B, L), np.uint8), 3))


def test_batch_kernel_extreme_rows(cs):
    """Rows the streaming pass hands to the exact path, in the batch kernel."""
    from test_gpu_exotic import extreme_rows

    z = extreme_rows(20_011, 3)            # 16 rows
    B, L = 2, 8
    dev = to_device(z, "f32", stride=20_012).view(B, L, -1)
    cand = torch.ones((B, L), dtype=torch.uint8, device="cuda")
    x0, prob, ent, commit, _ = cs.commit_step(dev, rule=1, tau=0.5, suppress_ids=[1], cand=cand, inputs_ready=True)
    torch.cuda.synchronize()
    ox0, op, oe = oracle.token_stats(z, suppress_ids=[1])
    assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
    gp = prob.cpu().numpy()
    assert_stats_close("f32", gp, ent.cpu().numpy(), op, oe, "extreme")
    assert np.array_equal(commit.cpu().numpy(), oracle.threshold_transfer(gp, np.ones((B, L), np.uint8), 0.5, False))


def test_batch_kernel_back_to_back_steps(cs):
    """Many inputs-ready steps queued back to back over rotating buffers (the
    bench's launch, several steps in flight) give the results of plain calls."""
    rng = np.random.default_rng(44)
    B, L, V = 1, 32, 126464
    bufs, hosts = [], []
    for j in range(6):
        host, dev = make(rng, B, L, V, "bf16", scale=1.0 + j)
        bufs.append(dev)
        hosts.append(host)
    cand = torch.from_numpy((rng.random((B, L)) < 0.6).astype(np.uint8)).cuda()
    res = []
    for rep in range(4):
        for j in range(6):
            x0, prob, ent, commit, _ = cs.commit_step(bufs[j], rule=1, tau=0.9, strict=True, cand=cand,
                                                      suppress_ids=[126336], inputs_ready=True)
            res.append((j, x0, prob, ent, commit))
    torch.cuda.synchronize()
    oracle_stats = [oracle.token_stats(h, dtype="bf16", suppress_ids=[126336]) for h in hosts]
    for j, x0, prob, ent, commit in res:
        ox0, op, oe = oracle_stats[j]
        assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
        gp = prob.cpu().numpy()
        assert_stats_close("bf16", gp, ent.cpu().numpy(), op, oe, f"step {j}")
        assert np.array_equal(commit.cpu().numpy(), oracle.threshold_transfer(gp, cand.cpu().numpy(), 0.9, True))
