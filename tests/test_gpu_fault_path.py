"""The fault path of the statistics kernel, exercised without a real fault.

Every mbarrier wait in the kernel is bounded (about one second); a wait that
runs out records a fault code in the workspace and the CTA stops in order
(its issued copies drained first).  DLLM_FLAG_TEST_DROP_COPY makes the first
CTA skip one bulk copy, so that its consumers' wait for it runs out: the call
must come back, dllm_workspace_fault must report the code, and the workspace,
once zeroed, must serve a correct call.  Both grid kinds: a cluster per row
and the persistent grid with rows split across CTAs.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from dllm_workloads import f32_to_bf16_bits
from gpu_helpers import assert_stats_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,L,V,dtype", [(1, 32, 126464, "bf16"), (4, 96, 50_000, "f32")],
                         ids=["cluster", "persistent"])
def test_wait_that_runs_out_is_reported_and_the_workspace_recovers(cs, B, L, V, dtype):
    rng = np.random.default_rng(B + V)
    z = (rng.standard_normal((B * L, V)) * 2).astype(np.float32)
    host = f32_to_bf16_bits(z) if dtype == "bf16" else z
    t = torch.from_numpy(host.view(np.int16) if dtype == "bf16" else host).cuda()
    logits = (t.view(torch.bfloat16) if dtype == "bf16" else t).view(B, L, V)
    cand = torch.ones((B, L), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(int(cs.lib_handle().dllm_token_stats_workspace_size(B, L, V, 1 if dtype == "bf16" else 0)),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    cs.commit_step(logits, rule=cs.RULE_NONE, cand=cand, suppress_ids=[7], ws=ws,
                   _test_flags=cs.FLAG_TEST_DROP_COPY)
    code = cs.workspace_fault(ws)             # synchronises; zeroes the workspace when a fault is reported
    elapsed = time.perf_counter() - t0
    assert code in (1, 2), f"expected a bounded-wait fault code, got {code}"
    assert 0.3 < elapsed < 30, elapsed       # the wait ran out (about a second), and the call came back
    # the device is still usable and the zeroed workspace serves a correct call
    x0, prob, ent, _, _ = cs.commit_step(logits, rule=cs.RULE_NONE, cand=cand, suppress_ids=[7], ws=ws)
    torch.cuda.synchronize()
    assert cs.workspace_fault(ws) == 0
    ox0, op, oe = oracle.token_stats(host, dtype=dtype, suppress_ids=[7])
    assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
    assert_stats_close(dtype, prob.cpu().numpy(), ent.cpu().numpy(), op, oe, "after the fault")
