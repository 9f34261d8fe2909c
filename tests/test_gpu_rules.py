"""GPU parity of the commit rules, edit rule and schedule against the oracle,
bit for bit, on seeded confidences with exact ties, NaNs and ragged L."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def rand_conf(rng, B, L, ties=True, nan=True):
    c = rng.random((B, L)).astype(np.float32)
    if ties:
        c = np.round(c * 16) / 16                       # many exact ties
        c = c.astype(np.float32)
    if nan:
        c[rng.random((B, L)) < 0.03] = np.nan
    c[rng.random((B, L)) < 0.02] = -0.0
    return c


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


SHAPES = [(1, 1), (3, 7), (4, 32), (2, 64), (8, 256), (5, 513), (2, 1024), (3, 1500), (1, 4096), (2, 16384)]


@pytest.mark.parametrize("B,L", SHAPES)
def test_threshold(cs, B, L):
    rng = np.random.default_rng(B * 1000 + L)
    c = rand_conf(rng, B, L)
    cand = (rng.random((B, L)) < 0.6).astype(np.uint8)
    cand[0, :] = 0 if B > 1 else cand[0, :]             # a row without candidates
    for tau, strict in ((0.9, False), (0.9, True), (0.5, False), (1.5, False), (-1.0, True)):
        got = cs.threshold_transfer(dev(c), dev(cand), tau, strict).cpu().numpy()
        want = oracle.threshold_transfer(c, cand, tau, strict)
        assert np.array_equal(got, want), (tau, strict)


@pytest.mark.parametrize("B,L", SHAPES)
def test_topk(cs, B, L):
    rng = np.random.default_rng(B * 1001 + L)
    c = rand_conf(rng, B, L)
    cand = (rng.random((B, L)) < 0.5).astype(np.uint8)
    k = rng.integers(-1, L + 2, size=B).astype(np.int32)
    got = cs.topk_transfer(dev(c), dev(cand), dev(k)).cpu().numpy()
    assert np.array_equal(got, oracle.topk_transfer(c, cand, k))


@pytest.mark.parametrize("B,L", SHAPES)
def test_factor(cs, B, L):
    rng = np.random.default_rng(B * 1002 + L)
    c = rand_conf(rng, B, L, ties=False)
    c = np.where(np.isnan(c), c, 1 - (1 - c) ** 4).astype(np.float32)   # confident rows: long prefixes
    cand = (rng.random((B, L)) < 0.5).astype(np.uint8)
    for f in (1.0, 0.1, 3.0, 0.0):
        got = cs.factor_transfer(dev(c), dev(cand), f).cpu().numpy()
        assert np.array_equal(got, oracle.factor_transfer(c, cand, f)), f


@pytest.mark.parametrize("B,L", SHAPES)
def test_entropy_bound(cs, B, L):
    rng = np.random.default_rng(B * 1003 + L)
    h = (rng.exponential(0.05, (B, L))).astype(np.float32)
    h[rng.random((B, L)) < 0.02] = np.nan
    h[rng.random((B, L)) < 0.05] = 0.0
    cand = (rng.random((B, L)) < 0.5).astype(np.uint8)
    for g in (0.1, 0.0, 2.0, -1.0):
        got = cs.entropy_bound_transfer(dev(h), dev(cand), g).cpu().numpy()
        assert np.array_equal(got, oracle.entropy_bound_transfer(h, cand, g)), g


def test_rules_canvas_update(cs):
    rng = np.random.default_rng(77)
    B, L, N, off = 3, 40, 100, 17
    c = rand_conf(rng, B, L)
    cand = (rng.random((B, L)) < 0.7).astype(np.uint8)
    x0 = rng.integers(0, 1000, (B, L)).astype(np.int32)
    canvas0 = rng.integers(0, 1000, (B, N)).astype(np.int32)
    canvas = dev(canvas0)
    commit = cs.threshold_transfer(dev(c), dev(cand), 0.7, True, x0=dev(x0), canvas=canvas, canvas_offset=off)
    want = oracle.threshold_transfer(c, cand, 0.7, True).astype(bool)
    exp = canvas0.copy()
    exp[:, off:off + L] = np.where(want, x0, canvas0[:, off:off + L])
    assert np.array_equal(commit.cpu().numpy().astype(bool), want)
    assert np.array_equal(canvas.cpu().numpy(), exp)


@pytest.mark.parametrize("n", [1, 37, 100_000])
def test_edit(cs, n):
    rng = np.random.default_rng(n)
    x0 = rng.integers(0, 5, n).astype(np.int32)
    tok = rng.integers(0, 5, n).astype(np.int32)
    p = rng.random(n).astype(np.float32)
    p[rng.random(n) < 0.05] = np.nan
    p[rng.random(n) < 0.05] = 0.9
    ed = (rng.random(n) < 0.7).astype(np.uint8)
    got = cs.edit_transfer(dev(x0[None]), dev(p[None]), dev(tok[None]), dev(ed[None]), 0.9).cpu().numpy()[0]
    assert np.array_equal(got, oracle.edit_transfer(x0, p, tok, ed, 0.9))


def test_transfer_schedule(cs):
    rng = np.random.default_rng(5)
    for steps in (1, 4, 32, 77):
        counts = rng.integers(-3, 3000, size=9).astype(np.int32)
        got = cs.transfer_schedule(dev(counts), steps).cpu().numpy()
        assert np.array_equal(got, oracle.transfer_schedule(counts, steps))


def test_block_ranges_host_entry(cs):
    for args in ((128, 1024, 32, False), (128, 1024, 32, True), (5, 11, 4, True), (7, 0, 4, False)):
        assert cs.block_ranges(*args) == oracle.block_ranges(*args)


def test_rule_argument_errors(cs):
    import ctypes

    lib = cs.lib_handle()
    c = torch.zeros(2, 8, device="cuda")
    m = torch.ones(2, 8, dtype=torch.uint8, device="cuda")
    out = torch.zeros(2, 8, dtype=torch.uint8, device="cuda")
    x0 = torch.zeros(2, 8, dtype=torch.int32, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # negative sizes, missing pointers, x0 without canvas, overlapping canvas rows, NaN tau
    assert lib.dllm_threshold_transfer(P(c), P(m), -1, 8, ctypes.c_float(0.5), 0, P(out), None, None, 0, 0, s) == 1
    assert lib.dllm_threshold_transfer(None, P(m), 2, 8, ctypes.c_float(0.5), 0, P(out), None, None, 0, 0, s) == 1
    assert lib.dllm_threshold_transfer(P(c), P(m), 2, 8, ctypes.c_float(0.5), 0, P(out), P(x0), None, 0, 0, s) == 1
    assert lib.dllm_threshold_transfer(P(c), P(m), 2, 8, ctypes.c_float(0.5), 0, P(out), P(x0), P(x0), 4, 0, s) == 1
    with pytest.raises(cs.DllmError):
        cs.threshold_transfer(c, m, float("nan"))
    assert lib.dllm_topk_transfer(P(c), P(m), 2, 8, None, P(out), None, None, 0, 0, s) == 1   # k missing
    with pytest.raises(ValueError):
        cs.topk_transfer(c, m, torch.zeros(0, dtype=torch.int32, device="cuda"))
    big = torch.zeros(1, 16385, device="cuda")
    with pytest.raises(cs.DllmError):
        cs.topk_transfer(big, torch.ones(1, 16385, dtype=torch.uint8, device="cuda"), 3)
    # empty calls are valid and launch nothing
    e = torch.zeros(0, 8, device="cuda")
    cs.threshold_transfer(e, torch.zeros(0, 8, dtype=torch.uint8, device="cuda"), 0.5)
