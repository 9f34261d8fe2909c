"""The block-decode loop with editing on the GPU (fused commit steps) against
the oracle's loop on the same generator: the full loop workload (B=4, P=128,
gen_len=1024, block_len=32, V=126464 bf16) and a small one."""
import numpy as np
import pytest
import torch

import dllm_workloads as W
from oracle.loop import decode_with_editing as oracle_loop

pytestmark = pytest.mark.gpu


def run_both(cs, spec):
    from commit_step_gb300.decode import decode_with_editing as gpu_loop

    gen = W.LoopGenerator(spec)
    prompt = torch.from_numpy(gen.prompt).cuda()
    gtrace, otrace = [], []
    out_g, fw_g = gpu_loop(lambda bi, st, c0, n: gen.device_logits(bi, st, c0, n), prompt, gen_len=spec.gen_len,
                           block_len=spec.block_len, mask_id=spec.mask_id, threshold=spec.tau,
                           editing_threshold=spec.tau_edit, max_post_steps=spec.max_post_steps,
                           suppress_ids=[spec.mask_id], trace=gtrace)
    out_o, fw_o = oracle_loop(lambda bi, st, c0, n: gen.host_logits(bi, st, c0, n), gen.prompt,
                              gen_len=spec.gen_len, block_len=spec.block_len, mask_id=spec.mask_id,
                              threshold=spec.tau, editing_threshold=spec.tau_edit,
                              max_post_steps=spec.max_post_steps, suppress_ids=[spec.mask_id], trace=otrace)
    for i, (a, b) in enumerate(zip(gtrace, otrace)):
        assert a == b, f"step {i} differs: gpu {a} oracle {b}"
    assert fw_g == fw_o
    assert np.array_equal(out_g.cpu().numpy(), out_o)
    return gtrace


def test_small_loop(cs):
    spec = W.LoopSpec(B=2, P=5, gen_len=40, block_len=8, V=4096, mask_id=4000, bank_rows=16, max_post_steps=3)
    trace = run_both(cs, spec)
    assert any(t[3] > 0 for t in trace)        # the edit path fired


def test_full_loop_workload(cs):
    trace = run_both(cs, W.loop_spec())
    assert len(trace) >= 32 and any(t[3] > 0 for t in trace)
