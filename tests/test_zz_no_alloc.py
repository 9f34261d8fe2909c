"""dllm_token_stats_noalloc: the statistics pass for callers that may not
allocate device memory (its scratch is a fixed array inside the library).

Called through the C ABI with ctypes, on two calls in a row per case, and
checked against the oracle (x0 bit for bit, prob and entropy within the
statistics tolerance of the other GPU tests) and against dllm_token_stats
(the entry point with a caller workspace).  After every call the array's
fault word is read back with dllm_noalloc_fault and must be 0.  Shapes cover
the cluster grid (few rows), the persistent grid with rows split across CTAs
(the partials and per-row counters inside the array), and a shape just under
the array's size.  This file is collected last so that a run stopping at the
first failure has already run every other test; it passes alone in a fresh
process as well.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from dllm_workloads import f32_to_bf16_bits
from gpu_helpers import assert_stats_close

pytestmark = pytest.mark.gpu


def call_noalloc(lib, logits, dtype_code, B, L, V, temperature, key, sup, outs):
    x0, prob, ent = outs
    arr = (C.c_int32 * max(1, len(sup)))(*sup)
    f = lib.dllm_token_stats_noalloc
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.c_int, C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_float, C.c_uint64,
                  C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    return f(logits.data_ptr(), dtype_code, B, L, V, V, temperature, key, arr, len(sup),
             x0.data_ptr(), prob.data_ptr(), ent.data_ptr(), torch.cuda.current_stream().cuda_stream)


def read_fault(lib):
    f = lib.dllm_noalloc_fault
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.POINTER(C.c_int32)]
    code = C.c_int32(-1)
    assert f(torch.cuda.current_stream().cuda_stream, C.byref(code)) == 0
    return code.value


CASES = [
    # (B, L, V, dtype, temperature, key, suppress): cluster grid, greedy and Gumbel
    (2, 32, 126464, "bf16", 0.0, 0, [126336, 5]),
    (2, 32, 126464, "bf16", 0.7, 0xABCDEF, [126336, 5]),
    # persistent grid, rows split across CTAs (the Dream-7B shape)
    (8, 256, 152064, "bf16", 0.7, 0x5EED, []),
    # 250,000 short rows: the row counters fill the array almost to its size
    (1, 250_000, 8, "f32", 0.0, 0, [3]),
]


@pytest.mark.parametrize("case", CASES, ids=["cluster-greedy", "cluster-gumbel", "persistent-gumbel", "near-limit"])
def test_noalloc_matches_oracle_twice(cs, case):
    lib = cs.lib_handle()
    B, L, V, dtype, temperature, key, sup = case
    rng = np.random.default_rng(B * L + V)
    code = 1 if dtype == "bf16" else 0
    for call in range(2):
        z = (rng.standard_normal((B * L, V)) * (2.0 + call)).astype(np.float32)
        z[np.arange(B * L), rng.integers(0, V, B * L)] += 6.0
        host = f32_to_bf16_bits(z) if dtype == "bf16" else z
        t = torch.from_numpy(host.view(np.int16) if dtype == "bf16" else host).cuda()
        logits = (t.view(torch.bfloat16) if dtype == "bf16" else t).view(B, L, V)
        outs = tuple(torch.empty((B, L), dtype=dt, device="cuda")
                     for dt in (torch.int32, torch.float32, torch.float32))
        st = call_noalloc(lib, logits, code, B, L, V, temperature, key, sup, outs)
        assert st == 0, cs.status_string(st)
        assert read_fault(lib) == 0
        ox0, op, oe = oracle.token_stats(host, dtype=dtype, temperature=temperature, key=key, suppress_ids=sup)
        gx0 = outs[0].cpu().numpy().reshape(-1)
        bad = np.flatnonzero(gx0 != ox0)
        assert bad.size == 0, f"call {call}: x0 differs from the oracle in rows {bad[:5].tolist()}"
        assert_stats_close(dtype, outs[1].cpu().numpy(), outs[2].cpu().numpy(), op, oe, f"no-alloc call {call}")
        # and the workspace entry point gives the same x0 and statistics within the tolerance
        rx0, rp, re = cs.token_stats(logits, temperature=temperature, key=key, suppress_ids=sup)
        torch.cuda.synchronize()
        assert np.array_equal(gx0, rx0.cpu().numpy().reshape(-1)), f"call {call}: x0 differs from token_stats"
        assert_stats_close(dtype, outs[1].cpu().numpy(), outs[2].cpu().numpy(),
                           rp.cpu().numpy().astype(np.float64), re.cpu().numpy().astype(np.float64),
                           f"no-alloc vs token_stats, call {call}")


def test_noalloc_through_the_binding(cs):
    rng = np.random.default_rng(77)
    z = (rng.standard_normal((48, 5000)) * 3).astype(np.float32)
    logits = torch.from_numpy(z).cuda()
    for _ in range(2):
        x0, prob, ent = cs.token_stats_noalloc(logits, suppress_ids=[1])
        assert cs.noalloc_fault() == 0
        ox0, op, oe = oracle.token_stats(z, suppress_ids=[1])
        assert np.array_equal(x0.cpu().numpy(), ox0)
        assert_stats_close("f32", prob.cpu().numpy(), ent.cpu().numpy(), op, oe, "binding")


def test_noalloc_rejects_shapes_beyond_its_scratch(cs):
    lib = cs.lib_handle()
    B, L, V = 1, 300_000, 8                    # needs more than the fixed scratch
    logits = torch.zeros((B * L, V), dtype=torch.float32, device="cuda")
    outs = tuple(torch.empty((B * L,), dtype=dt, device="cuda") for dt in (torch.int32, torch.float32, torch.float32))
    st = call_noalloc(lib, logits, 0, B, L, V, 0.0, 0, [], outs)
    assert st == 2, cs.status_string(st)      # DLLM_ERR_UNSUPPORTED, nothing launched
