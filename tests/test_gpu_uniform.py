"""GPU parity of the uniform-noise decoding helpers and loop against the
oracle: linear_temperature (bit-exact fp32), uniform_canvas (bit-exact
tokens), renoise (with frozen rows), the stopping criterion over call
sequences (state and flags bit-exact), and whole loops (argmax canvas, step
count and per-step done counts identical)."""
import numpy as np
import pytest
import torch

import dllm_workloads as W
import oracle
from oracle.loop import decode_uniform as oracle_decode_uniform

pytestmark = pytest.mark.gpu


def test_linear_temperature_matches(cs):
    for num_steps in (1, 7, 48, 1000):
        for remaining in sorted({0, 1, num_steps // 3, num_steps - 1, num_steps}):
            for t_min, t_max in ((0.4, 0.8), (0.05, 3.0), (1.0, 1.0)):
                assert np.float32(cs.linear_temperature(remaining, num_steps, t_min, t_max)) == \
                    oracle.linear_temperature(remaining, num_steps, t_min, t_max)
    with pytest.raises(cs.DllmError):
        cs.linear_temperature(5, 4)


@pytest.mark.parametrize("B,N,V", [(1, 1, 7), (3, 257, 262144), (4, 1022, 4096), (2, 10_001, 151_936)])
def test_uniform_canvas_matches(cs, B, N, V):
    key = 0xFEEDFACE12345678 + N
    got = cs.uniform_canvas(B, N, V, key).cpu().numpy()
    assert np.array_equal(got, oracle.uniform_canvas(B, N, V, key))
    wide = torch.full((B, N + 13), -5, dtype=torch.int32, device="cuda")
    cs.uniform_canvas(B, N, V, key, out=wide[:, :N])
    w = wide.cpu().numpy()
    assert np.array_equal(w[:, :N], got) and np.all(w[:, N:] == -5)


def test_renoise_matches_with_frozen_rows(cs):
    rng = np.random.default_rng(3)
    B, N = 5, 700
    sample = rng.integers(0, 1000, (B, N)).astype(np.int32)
    noise = rng.integers(0, 1000, (B, N)).astype(np.int32)
    acc = (rng.random((B, N)) < 0.3).astype(np.uint8)
    old = rng.integers(0, 1000, (B, N)).astype(np.int32)
    frozen = np.array([0, 1, 0, 0, 1], np.uint8)
    d = lambda a: torch.from_numpy(a).cuda()
    out = d(old.copy())
    cs.renoise(d(sample), d(acc), d(noise), out=out, frozen=d(frozen))
    want = oracle.renoise(sample, acc, noise)
    want[frozen == 1] = old[frozen == 1]
    assert np.array_equal(out.cpu().numpy(), want)
    out2 = cs.renoise(d(sample), None, None)
    assert np.array_equal(out2.cpu().numpy(), sample)


@pytest.mark.parametrize("L", [300, 2500])
def test_stopping_criterion_sequence_matches(cs, L):
    rng = np.random.default_rng(L)
    B = 6
    thr = 0.005
    ref = oracle.StableConfidentStopping(B, L, 1, thr)
    gpu = cs.StableConfidentStopping(B, L, 1, thr)
    done = torch.zeros(B, dtype=torch.uint8, device="cuda")
    done_ref = np.zeros(B, np.uint8)
    canvas = rng.integers(0, 50, (B, L)).astype(np.int32)
    for call in range(8):
        change = rng.random(B) < 0.4
        canvas[change, rng.integers(0, L)] += 1
        ent = np.where(rng.random((B, 1)) < 0.5, 1e-4, 0.05) * rng.random((B, L)) * 2
        ent = ent.astype(np.float32)
        ent[0, :] = thr                                     # a mean exactly at the threshold: not confident
        ent[1, 0] = np.nan                                  # NaN counts as 64
        want = ref(canvas, ent)
        got = gpu(torch.from_numpy(canvas).cuda(), torch.from_numpy(ent).cuda(), done=done)
        done_ref |= want
        assert np.array_equal(got.cpu().numpy(), want), call
        assert np.array_equal(done.cpu().numpy(), done_ref), call
        assert np.array_equal(gpu.count.cpu().numpy(), ref.count), call
        assert np.array_equal(gpu.prev.cpu().numpy(), ref.prev), call


@pytest.mark.parametrize("dtype,B,N,V,onset", [("f32", 2, 32, 4096, 10), ("bf16", 2, 64, 32768, 14),
                                               ("bf16", 1, 256, 262144, 8)])
def test_uniform_loop_matches_oracle_loop(cs, dtype, B, N, V, onset):
    from commit_step_gb300.decode import decode_uniform

    spec = W.uniform_spec(B=B, N=N, V=V, dtype=dtype, max_onset=onset)
    gen = W.UniformGenerator(spec)
    trace_ref = []
    want, steps_ref = oracle_decode_uniform(lambda st, c: gen.host_logits(st), batch=B, canvas_len=N, vocab_size=V,
                                            key=spec.key, dtype=dtype, trace=trace_ref)
    trace = []
    got, steps = decode_uniform(lambda st, c: gen.device_logits(st), batch=B, canvas_len=N, vocab_size=V,
                                key=spec.key, trace=trace)
    assert steps == steps_ref
    assert [t[1] for t in trace] == [t[2] for t in trace_ref]
    assert np.array_equal(got.cpu().numpy(), want)
    assert np.array_equal(want, gen.targets)


def test_fused_update_equals_the_four_calls(cs):
    """dllm_uniform_update gives what uniform_canvas, renoise (twice, done
    rows frozen) and the stopping criterion give in that order."""
    rng = np.random.default_rng(9)
    B, N, V = 5, 700, 262144
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sample = d(rng.integers(0, V, (B, N)).astype(np.int32))
    accepted = d((rng.random((B, N)) < 0.3).astype(np.uint8))
    step_am = d(rng.integers(0, V, (B, N)).astype(np.int32))
    canvas0 = rng.integers(0, V, (B, N)).astype(np.int32)
    argmax0 = rng.integers(0, V, (B, N)).astype(np.int32)
    step_np = step_am.cpu().numpy()
    argmax0[1] = step_np[1]                                    # row 1 will be stable
    done0 = np.array([0, 0, 1, 0, 1], np.uint8)
    for call in range(3):
        ent = d(np.where(rng.random((B, 1)) < 0.5, 1e-4, 0.05).astype(np.float32) * np.ones((B, N), np.float32))
        # the composition
        ref_stop = cs.StableConfidentStopping(B, N, 1, 0.005)
        c_ref, a_ref, done_ref = d(canvas0.copy()), d(argmax0.copy()), d(done0.copy())
        ref_stop.prev.copy_(d(argmax0)); ref_stop.count.fill_(call - 1)
        noise = cs.uniform_canvas(B, N, V, 1234 + call)
        cs.renoise(sample, accepted, noise, out=c_ref, frozen=done_ref)
        cs.renoise(step_am, None, None, out=a_ref, frozen=done_ref)
        ref_stop(a_ref, ent, done=done_ref)
        # one launch
        stop = cs.StableConfidentStopping(B, N, 1, 0.005)
        c, a, done = d(canvas0.copy()), d(argmax0.copy()), d(done0.copy())
        stop.prev.copy_(d(argmax0)); stop.count.fill_(call - 1)
        cs.uniform_update(sample, accepted, step_am, ent, V, 1234 + call, stop, c, a, done)
        torch.cuda.synchronize()
        for x, y in ((c, c_ref), (a, a_ref), (done, done_ref), (stop.prev, ref_stop.prev), (stop.count, ref_stop.count)):
            assert torch.equal(x, y), call
