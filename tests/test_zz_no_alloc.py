"""dllm_token_stats_noalloc: the statistics pass for callers that may not
allocate device memory (its scratch is a fixed array inside the library).

Called through the C ABI with ctypes and checked against dllm_token_stats (the
entry point with a caller workspace) on two calls in a row, within the
statistics tolerance of the other GPU tests.  This file is collected last so
that a run stopping at the first failure has already run every other test;
it passes alone in a fresh process as well.
"""
import ctypes as C

import numpy as np
import pytest
import torch

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


def test_noalloc_matches_workspace_entry_point_twice(cs):
    lib = cs.lib_handle()
    rng = np.random.default_rng(2024)
    B, L, V = 2, 32, 126464
    for call, (temperature, key) in enumerate(((0.0, 0), (0.7, 0xABCDEF))):
        z = (rng.standard_normal((B * L, V)) * (2.0 + call)).astype(np.float32)
        bits = f32_to_bf16_bits(z)
        logits = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16).view(B, L, V)
        sup = [126336, 5]
        outs = tuple(torch.empty((B, L), dtype=dt, device="cuda")
                     for dt in (torch.int32, torch.float32, torch.float32))
        st = call_noalloc(lib, logits, 1, B, L, V, temperature, key, sup, outs)
        assert st == 0, cs.status_string(st)
        rx0, rp, re = cs.token_stats(logits, temperature=temperature, key=key, suppress_ids=sup)
        torch.cuda.synchronize()
        assert np.array_equal(outs[0].cpu().numpy(), rx0.cpu().numpy()), f"call {call}: x0 differs"
        assert_stats_close("bf16", outs[1].cpu().numpy(), outs[2].cpu().numpy(),
                           rp.cpu().numpy().astype(np.float64), re.cpu().numpy().astype(np.float64),
                           f"no-alloc call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch(cs):
    lib = cs.lib_handle()
    B, L, V = 1, 300_000, 8                    # needs more than the fixed scratch
    logits = torch.zeros((B * L, V), dtype=torch.float32, device="cuda")
    outs = tuple(torch.empty((B * L,), dtype=dt, device="cuda") for dt in (torch.int32, torch.float32, torch.float32))
    st = call_noalloc(lib, logits, 0, B, L, V, 0.0, 0, [], outs)
    assert st == 2, cs.status_string(st)      # DLLM_ERR_UNSUPPORTED, nothing launched
