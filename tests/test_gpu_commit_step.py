"""GPU parity of the fused commit step (statistics + rule + canvas update in
one launch) against the oracle, on the five workloads, every one in full:
x0 bit for bit, prob and entropy within the tolerances of gpu_helpers, and
the commit masks bit for bit against the oracle's rule evaluated on the
statistics the GPU emitted ("dLLM block decoding", Deviations from the
references: the rules decide on fp32 confidences)."""
import numpy as np
import pytest
import torch

import dllm_workloads as W
import oracle
from gpu_helpers import TOL, assert_stats_close, to_device

pytestmark = pytest.mark.gpu

RULES = {"threshold": 1, "topk": 2, "factor": 3, "entropy_bound": 4}


def fused(cs, w, logits_dev, rule, **kw):
    cand = torch.from_numpy(w.candidates).cuda()
    return cs.commit_step(logits_dev.view(w.B, w.L, w.V), rule=RULES[rule], temperature=w.temperature, key=w.key,
                          suppress_ids=w.suppress_ids, cand=cand, **kw)


def oracle_rule(rule, scores, cand, params):
    """The oracle's rule on the given fp32 scores (prob, or entropy for the entropy bound)."""
    s32 = np.asarray(scores, dtype=np.float32)
    if rule == "threshold":
        return oracle.threshold_transfer(s32, cand, params["tau"], params["strict"])
    if rule == "topk":
        return oracle.topk_transfer(s32, cand, params["k"])
    if rule == "factor":
        return oracle.factor_transfer(s32, cand, params["factor"])
    return oracle.entropy_bound_transfer(s32, cand, params["gamma"])


def assert_mask_equal(got, want, what):
    bad = np.flatnonzero((np.asarray(got) != np.asarray(want)).any(axis=1))
    assert bad.size == 0, f"{what}: commit masks differ in batch rows {bad[:8].tolist()}"


def check_full(cs, w, rule, params, canvas=False, **kw):
    """One fused call over the whole workload, checked element by element.
    With canvas=True the call also writes x0 into a canvas where it commits
    (the bench's launch), and the canvas is checked too."""
    dev = to_device(w.logits, w.dtype)
    cv = None
    if canvas:
        cv = torch.full((w.B, 128 + w.L), -7, dtype=torch.int32, device="cuda")
        kw = dict(kw, canvas=cv, canvas_offset=128)
    x0, prob, ent, commit, _ = fused(cs, w, dev, rule, **kw)
    torch.cuda.synchronize()
    gx0, gp, ge, got = (t.cpu().numpy() for t in (x0, prob, ent, commit))
    ox0, op, oe = oracle.token_stats(w.logits, dtype=w.dtype, temperature=w.temperature, key=w.key,
                                     suppress_ids=w.suppress_ids)
    bad = np.flatnonzero(gx0.reshape(-1) != ox0)
    assert bad.size == 0, f"{w.name}: x0 differs in {bad.size} rows, first {bad[:5].tolist()}"
    assert_stats_close(w.dtype, gp, ge, op, oe, w.name)
    scores = (ge if rule == "entropy_bound" else gp).reshape(w.B, w.L)
    want = oracle_rule(rule, scores, w.candidates, params)
    assert_mask_equal(got, want, f"{w.name}/{rule}")
    if canvas:
        exp = np.full((w.B, 128 + w.L), -7, dtype=np.int32)
        exp[:, 128:] = np.where(want.astype(bool), gx0.reshape(w.B, w.L), -7)
        assert np.array_equal(cv.cpu().numpy(), exp), f"{w.name}: canvas differs"
    return got, gx0.reshape(w.B, w.L), gp.reshape(w.B, w.L), ge.reshape(w.B, w.L)


@pytest.mark.parametrize("bench_launch", [False, True])
def test_tiny_threshold(cs, bench_launch):
    w = W.tiny()
    kw = {"inputs_ready": True} if bench_launch else {}
    got, *_ = check_full(cs, w, "threshold", w.params, canvas=bench_launch, tau=0.9, strict=False, **kw)
    assert got.sum() >= 1


@pytest.mark.parametrize("bench_launch", [False, True])
def test_llada_threshold_strict(cs, bench_launch):
    """The LLaDA-8B-shaped block step; bench_launch: as bench.py times it
    (DLLM_FLAG_INPUTS_READY, which plans a smaller cluster grid, and the
    canvas update)."""
    w = W.llada()
    kw = {"inputs_ready": True} if bench_launch else {}
    got, *_ = check_full(cs, w, "threshold", w.params, canvas=bench_launch, tau=0.95, strict=True, **kw)
    assert 1 <= got.sum() <= 19 and np.all(got <= w.candidates)


@pytest.mark.parametrize("seed", [1, 2])
def test_small_rules_all_kinds(cs, seed):
    """Every rule on a reduced LLaDA-like shape (B=3, L=40, V=3000, ragged)."""
    rng = np.random.default_rng(seed)
    B, L, V = 3, 40, 3000
    z = (rng.standard_normal((B * L, V)) * 2).astype(np.float32)
    for r in range(B * L):
        z[r, rng.integers(0, V)] += rng.uniform(0, 14)
    cand = (rng.random((B, L)) < 0.6).astype(np.uint8)
    w = W.Workload("small", B, L, V, "f32", z, None, [7], 0.0, 0, "", cand, {})
    k = np.array([3, 0, 50], dtype=np.int32)
    check_full(cs, w, "threshold", {"tau": 0.6, "strict": False}, tau=0.6)
    check_full(cs, w, "threshold", {"tau": 0.999, "strict": True}, tau=0.999, strict=True)   # forced commits
    check_full(cs, w, "topk", {"k": k}, k=torch.from_numpy(k).cuda())
    check_full(cs, w, "factor", {"factor": 1.0}, factor=1.0)
    check_full(cs, w, "entropy_bound", {"gamma": 0.3}, gamma=0.3)


def test_fused_canvas_candidates_edit_counts(cs):
    """Candidates from the canvas (token == mask id), edit rule, canvas update
    and per-row counts, as the block-decode loop uses them."""
    rng = np.random.default_rng(3)
    B, L, V, N, off, MASK = 2, 32, 2048, 96, 40, 2047
    z = (rng.standard_normal((B * L, V))).astype(np.float32)
    tgt = rng.integers(0, 2000, (B, L))
    for b in range(B):
        for l in range(L):
            z[b * L + l, tgt[b, l]] += 18.0 if l % 3 else 5.0
    canvas0 = rng.integers(0, 2000, (B, N)).astype(np.int32)
    masked = rng.random((B, L)) < 0.5
    canvas0[:, off:off + L][masked] = MASK
    canvas = torch.from_numpy(canvas0.copy()).cuda()
    counts = torch.zeros((B, 3), dtype=torch.int32, device="cuda")
    dev = torch.from_numpy(z).cuda().view(B, L, V)
    x0, prob, ent, commit, edit = cs.commit_step(dev, rule=1, tau=0.95, strict=True, suppress_ids=[MASK],
                                                 mask_id=MASK, edit=True, tau_edit=0.9, canvas=canvas,
                                                 canvas_offset=off, counts=counts)
    ox0, op, _ = oracle.token_stats(z, suppress_ids=[MASK])
    assert np.array_equal(x0.cpu().numpy().reshape(-1), ox0)
    p32 = op.astype(np.float32).reshape(B, L)
    window = canvas0[:, off:off + L]
    want_c = oracle.threshold_transfer(p32, masked.astype(np.uint8), 0.95, True)
    want_e = oracle.edit_transfer(ox0.reshape(B, L), p32, window, (~masked).astype(np.uint8), 0.9)
    assert np.array_equal(commit.cpu().numpy(), want_c)
    assert np.array_equal(edit.cpu().numpy(), want_e)
    exp = canvas0.copy()
    exp[:, off:off + L] = np.where((want_c | want_e).astype(bool), ox0.reshape(B, L), window)
    assert np.array_equal(canvas.cpu().numpy(), exp)
    assert counts.cpu().numpy().tolist() == [[int(masked[b].sum()), int(want_c[b].sum()), int(want_e[b].sum())]
                                             for b in range(B)]


def test_inputs_ready_pipelining_matches_plain_calls(cs):
    """Back-to-back fused steps over independent buffers with
    DLLM_FLAG_INPUTS_READY give the same results as plain calls."""
    rng = np.random.default_rng(12)
    B, L, V = 2, 32, 50_000
    bufs, outs_plain = [], []
    cand = torch.from_numpy((rng.random((B, L)) < 0.6).astype(np.uint8)).cuda()
    for j in range(4):
        z = (rng.standard_normal((B * L, V)) * (1 + j)).astype(np.float32)
        bufs.append(torch.from_numpy(z).cuda().view(B, L, V))
    for j in range(4):
        x0, prob, ent, commit, _ = cs.commit_step(bufs[j], rule=1, tau=0.5, cand=cand, suppress_ids=[0])
        outs_plain.append((x0.clone(), prob.clone(), commit.clone()))
    res = []
    for rep in range(3):
        for j in range(4):
            x0, prob, ent, commit, _ = cs.commit_step(bufs[j], rule=1, tau=0.5, cand=cand, suppress_ids=[0],
                                                      inputs_ready=True)
            res.append((j, x0, prob, commit))
    torch.cuda.synchronize()
    for j, x0, prob, commit in res:
        # x0 and the masks are exact; prob may differ in the last bits because an
        # overlapping call sizes its grid differently (another fp32 summation order)
        assert torch.equal(x0, outs_plain[j][0]) and torch.equal(commit, outs_plain[j][2])
        assert torch.allclose(prob, outs_plain[j][1], rtol=TOL["f32"][0], atol=TOL["f32"][1])


def test_host_buffer_step_matches_device_call(cs):
    """dllm_commit_step_host (host logits in, one packed host read out) gives
    the device call's results bit for bit, over repeated steps whose host
    logits are refilled between steps, for a greedy and a sampled rule."""
    rng = np.random.default_rng(21)
    B, L, V = 2, 24, 40_000
    cand = torch.from_numpy((rng.random((B, L)) < 0.7).astype(np.uint8)).cuda()
    host = torch.empty((B, L, V), dtype=torch.bfloat16).pin_memory()
    for kw in ({"rule": 1, "tau": 0.6, "strict": True},
               {"rule": 2, "k": 3, "temperature": 0.8, "key": 77}):
        step = cs.HostStep(host, cand=cand, suppress_ids=[5, 17], **kw)
        for j in range(3):
            z = (rng.standard_normal((B * L, V)) * (2 + j)).astype(np.float32)
            z[np.arange(B * L), rng.integers(0, V, B * L)] += 9
            host.copy_(torch.from_numpy(z).view(B, L, V).to(torch.bfloat16))
            x0, prob, ent, commit = step()
            torch.cuda.synchronize()
            dx0, dprob, dent, dcommit, _ = cs.commit_step(host.cuda(), cand=cand, suppress_ids=[5, 17], **kw)
            torch.cuda.synchronize()
            assert torch.equal(x0, dx0.cpu()) and torch.equal(commit, dcommit.cpu())
            assert torch.equal(prob, dprob.cpu()) and torch.equal(ent, dent.cpu())
    with pytest.raises(ValueError):
        cs.HostStep(host.cuda(), rule=1, cand=cand)


def test_repeated_fused_calls_leave_workspace_clean(cs):
    w = W.tiny()
    dev = to_device(w.logits, w.dtype)
    first = None
    for _ in range(5):
        x0, prob, ent, commit, _ = fused(cs, w, dev, "threshold", tau=0.9)
        cur = (x0.cpu().numpy(), commit.cpu().numpy())
        if first is None:
            first = cur
        assert np.array_equal(cur[0], first[0]) and np.array_equal(cur[1], first[1])


# ---------------- full-size workloads, every row ----------------

def invariants(w, x0, prob, ent, commit):
    veff = w.V - len(set(w.suppress_ids))
    assert np.all(prob > 0) and np.all(prob <= 1 + 1e-6)
    assert np.all(ent >= 0) and np.all(ent <= np.log(veff) + 1e-4)
    assert not np.isin(x0, w.suppress_ids).any()
    assert np.all(commit <= w.candidates)


def test_full_dream_topk(cs):
    """Dream-7B-shaped canvas step, all 2048 rows and all 8 batch rows' masks,
    in the bench's launch configuration (canvas update, DLLM_FLAG_INPUTS_READY)."""
    w = W.dream()
    k = np.full(w.B, 8, dtype=np.int32)
    got, x0, prob, ent = check_full(cs, w, "topk", {"k": k}, canvas=True, k=torch.from_numpy(k).cuda(),
                                    inputs_ready=True)
    invariants(w, x0, prob, ent, got)
    assert np.all(got.sum(axis=1) == 8)


def test_full_large_factor_and_entropy_bound(cs):
    """Large batch, all 16384 rows; the factor rule fused, the entropy bound
    on the same statistics, all 32 batch rows' masks of both rules."""
    w = W.large()
    got, x0, prob, ent = check_full(cs, w, "factor", {"factor": 1.0}, canvas=True, factor=1.0, inputs_ready=True)
    cand = torch.from_numpy(w.candidates).cuda()
    eb = cs.entropy_bound_transfer(torch.from_numpy(np.ascontiguousarray(ent)).cuda(), cand, 0.1).cpu().numpy()
    invariants(w, x0, prob, ent, got)
    assert np.all(got.sum(axis=1) >= 1) and np.all(eb.sum(axis=1) >= 1) and np.all(eb <= w.candidates)
    assert_mask_equal(eb, oracle.entropy_bound_transfer(ent, w.candidates, 0.1), "large/entropy_bound")
