"""Edge cases of the C ABI on the GPU: empty inputs through every entry point
(DLLM_OK, nothing launched, nothing written), the largest sizes a call takes
(fused sorting rules at L = 1024, the fused threshold at L = 65535, 64
suppressed ids) and just past them (DLLM_ERR_UNSUPPORTED), and degenerate
inputs (one token, a vanishing temperature), each against the oracle."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_stats_close, to_device

pytestmark = pytest.mark.gpu

OK, UNSUPPORTED = 0, 2


def P(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def test_empty_inputs_touch_nothing(cs):
    lib = cs.lib_handle()
    s = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    sentinel = torch.full((16,), 7, dtype=torch.int32, device="cuda")
    sup = (C.c_int32 * 1)(0)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    for B, L in ((0, 5), (3, 0), (0, 0)):
        assert lib.dllm_token_stats(None, 1, B, L, 64, 64, 0.0, 0, sup, 0, None, None, None, P(ws), ws.numel(), s) == OK
        assert lib.dllm_token_stats_ex(None, 1, B, L, 64, 64, 0.7, 3, sup, 0, None, None, None, None, P(ws),
                                       ws.numel(), s) == OK
        p = cs.CommitParams()
        p.rule = cs.RULE_THRESHOLD
        assert lib.dllm_commit_step(None, 1, B, L, 64, 64, 0.0, 0, sup, 0, None, None, None, C.byref(p), P(ws),
                                    ws.numel(), s) == OK
        assert lib.dllm_threshold_transfer(None, None, B, L, C.c_float(0.5), 0, None, None, None, 0, 0, s) == OK
        assert lib.dllm_entropy_bound_transfer(None, None, B, L, C.c_float(0.1), None, None, None, 0, 0, s) == OK
        assert lib.dllm_renoise(None, None, None, None, B, L, None, s) == OK
        assert lib.dllm_uniform_canvas(B, L, 100, 1, None, L, s) == OK
    assert lib.dllm_edit_transfer(None, None, None, None, 0, 5, C.c_float(0.9), None, s) == OK
    assert lib.dllm_transfer_schedule(None, 0, 4, None, s) == OK
    assert lib.dllm_stable_confident_stop(None, None, 0, 8, 1, C.c_float(0.005), None, None, None, None, s) == OK
    assert lib.dllm_block_causal_mask(0, 0, 0, 0, 32, 0, None, 0, s) == OK
    torch.cuda.synchronize()
    assert torch.all(sentinel == 7)
    assert cs.workspace_fault(ws) == 0


def stats_and_rule_parity(cs, host, B, L, V, rule, **params):
    dev = to_device(host, "f32").view(B, L, V)
    cand = torch.ones((B, L), dtype=torch.uint8, device="cuda")
    kw = dict(cand=cand, suppress_ids=[0])
    if rule == "topk":
        kw["k"] = torch.full((B,), params["k"], dtype=torch.int32, device="cuda")
        r = cs.RULE_TOPK
    elif rule == "factor":
        kw["factor"] = params["factor"]
        r = cs.RULE_FACTOR
    elif rule == "entropy_bound":
        kw["gamma"] = params["gamma"]
        r = cs.RULE_ENTROPY_BOUND
    else:
        kw["tau"] = params["tau"]
        r = cs.RULE_THRESHOLD
    x0, prob, ent, commit, _ = cs.commit_step(dev, rule=r, **kw)
    torch.cuda.synchronize()
    ox0, op, oe = oracle.token_stats(host, suppress_ids=[0])
    assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
    assert_stats_close("f32", prob.cpu().numpy(), ent.cpu().numpy(), op, oe, f"{rule} L={L}")
    # the rule decides on the GPU's fp32 statistics, on both sides
    c = np.ones((B, L), np.uint8)
    g_prob, g_ent = prob.cpu().numpy().reshape(B, L), ent.cpu().numpy().reshape(B, L)
    if rule == "topk":
        want = oracle.topk_transfer(g_prob, c, np.full(B, params["k"], np.int32))
    elif rule == "factor":
        want = oracle.factor_transfer(g_prob, c, params["factor"])
    elif rule == "entropy_bound":
        want = oracle.entropy_bound_transfer(g_ent, c, params["gamma"])
    else:
        want = oracle.threshold_transfer(g_prob, c, params["tau"])
    assert np.array_equal(commit.cpu().numpy(), want), rule


@pytest.mark.parametrize("rule,params", [("topk", {"k": 700}), ("factor", {"factor": 3.0}),
                                         ("entropy_bound", {"gamma": 2.5})])
def test_fused_sorting_rules_at_their_largest_row(cs, rule, params):
    B, L, V = 2, 1024, 64
    rng = np.random.default_rng(1024)
    z = (rng.standard_normal((B * L, V)) * 2).astype(np.float32)
    z[np.arange(B * L), rng.integers(1, V, B * L)] += rng.uniform(0, 9, B * L).astype(np.float32)
    stats_and_rule_parity(cs, z, B, L, V, rule, **params)


def test_fused_threshold_at_its_largest_row(cs):
    B, L, V = 1, 65535, 16
    rng = np.random.default_rng(65535)
    z = (rng.standard_normal((B * L, V)) * 2).astype(np.float32)
    z[np.arange(L), rng.integers(1, V, L)] += rng.uniform(0, 9, L).astype(np.float32)
    stats_and_rule_parity(cs, z, B, L, V, "threshold", tau=0.9)


def test_sizes_just_past_the_limits(cs):
    dev = torch.zeros((1, 65536, 16), device="cuda")
    cand = torch.ones((1, 65536), dtype=torch.uint8, device="cuda")
    with pytest.raises(cs.DllmError) as e:
        cs.commit_step(dev, rule=cs.RULE_THRESHOLD, tau=0.5, cand=cand)
    assert e.value.status == UNSUPPORTED
    dev = torch.zeros((1, 1025, 16), device="cuda")
    cand = torch.ones((1, 1025), dtype=torch.uint8, device="cuda")
    with pytest.raises(cs.DllmError) as e:
        cs.commit_step(dev, rule=cs.RULE_ENTROPY_BOUND, gamma=0.1, cand=cand)
    assert e.value.status == UNSUPPORTED
    z = torch.zeros((1, 2, 128), device="cuda")
    with pytest.raises(cs.DllmError) as e:
        cs.token_stats(z, suppress_ids=list(range(65)))
    assert e.value.status == UNSUPPORTED


def test_sixty_four_suppressed_ids_with_duplicates(cs):
    rng = np.random.default_rng(64)
    V = 5000
    z = (rng.standard_normal((9, V)) * 3).astype(np.float32)
    sup = sorted(set(rng.integers(0, V, 60).tolist())) + [17, 17, 4999, 0]
    sup = sup[:64]
    z[:, sup] += 50.0                                        # suppressed ids would win otherwise
    x0, prob, ent = cs.token_stats(to_device(z, "f32"), suppress_ids=sup)
    ox0, op, oe = oracle.token_stats(z, suppress_ids=sup)
    assert np.array_equal(x0.cpu().numpy(), ox0)
    assert_stats_close("f32", prob.cpu().numpy(), ent.cpu().numpy(), op, oe, "64 suppressed")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_degenerate_rows(cs, dtype):
    rng = np.random.default_rng(5)
    from dllm_workloads import f32_to_bf16_bits
    one = np.array([[3.5], [-2.0], [np.nan]], np.float32)       # V = 1: prob 1, entropy 0
    h = one if dtype == "f32" else f32_to_bf16_bits(one)
    x0, prob, ent = cs.token_stats(to_device(h, dtype, stride=4 if dtype == "f32" else 8))
    assert np.all(x0.cpu().numpy() == 0) and np.allclose(prob.cpu().numpy(), 1) and np.allclose(ent.cpu().numpy(), 0)
    z = (rng.standard_normal((20, 3001)) * 2).astype(np.float32)
    h = z if dtype == "f32" else f32_to_bf16_bits(z)
    for t in (1e-30, 1e-3):                                  # sampling that degenerates to the argmax
        x0, prob, ent = cs.token_stats(to_device(h, dtype, stride=3004 if dtype == "f32" else 3008), temperature=t,
                                       key=11)
        ox0, op, oe = oracle.token_stats(h, dtype=dtype, temperature=t, key=11)
        assert np.array_equal(x0.cpu().numpy(), ox0)
        assert_stats_close(dtype, prob.cpu().numpy(), ent.cpu().numpy(), op, oe, f"t={t}")
