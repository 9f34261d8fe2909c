"""Seeded synthetic inputs for the commit step of masked diffusion-LM decoding.

This module only builds inputs: logit rows, candidate masks, per-row quotas,
Philox keys and the block-decode loop's per-step logits.  It serves both the
CUDA path (tests, bench) and the CPU oracle, and it holds none of the commit
step's arithmetic (no softmax, no ranking, no rule).

Every array comes from ``numpy.random.default_rng`` seeded with a tuple
``(seed, stream tag, indices...)``, so any single row can be rebuilt on its own
(the full-size parity checks rebuild only the rows they sample).

The five workloads follow the shapes the mlx-arsenal "dLLM block decoding"
research notes and the mojo-dllm manual describe:

* ``tiny``  -- B=1, L=64, V=4096 fp32, N(0, 3^2) with a +8 peak in 16 rows.
* ``llada`` -- one LLaDA-8B block step: B=1, L=32, V=126464 bf16.
* ``dream`` -- one Dream-7B canvas step: B=8, L=256, V=152064 bf16, Gumbel.
* ``large`` -- B=32, L=512, V=126464 fp32 N(0, 2^2) with a peak in every row.
* ``loop``  -- B=4, P=128, gen_len=1024, block_len=32, V=126464 bf16; a
  generator emits the active block's rows at every step.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

LLADA_VOCAB = 126464
LLADA_MASK_ID = 126336
DREAM_VOCAB = 152064

_TAGS = {"tiny": 1, "llada": 2, "dream": 3, "large": 4, "loop": 5, "uniform": 6}


def _rng(*entropy: int) -> np.random.Generator:
    return np.random.default_rng([int(e) for e in entropy])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the raw uint16 bits.

    Input construction only: it decides which bf16 values the workload holds.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    nan = np.isnan(x)
    # below 2^32 for every non-NaN pattern (at most 0xFF800000 + 0x8000)
    bb = np.where(nan, np.uint32(0), b)
    bb += np.uint32(0x7FFF)
    bb += (b >> np.uint32(16)) & np.uint32(1)
    rounded = (bb >> np.uint32(16)).astype(np.uint16)
    if nan.any():
        rounded[nan] = ((b[nan] >> 16) | 0x40).astype(np.uint16)  # keep it a quiet NaN
    return rounded


@dataclasses.dataclass
class Workload:
    """One commit-step workload.

    ``logits`` is (B*L, V): float32, or uint16 holding bf16 bits when
    ``dtype == "bf16"``.  ``rows`` lists which global rows ``logits`` holds when
    only a sample was built (None = all B*L rows, in order).
    """

    name: str
    B: int
    L: int
    V: int
    dtype: str
    logits: Optional[np.ndarray]
    rows: Optional[np.ndarray]
    suppress_ids: list
    temperature: float
    key: int
    rule: str                      # threshold | topk | factor+entropy_bound
    candidates: np.ndarray         # (B, L) uint8
    params: dict

    @property
    def T(self) -> int:
        return self.B * self.L

    def logit_bytes(self) -> int:
        return self.T * self.V * (2 if self.dtype == "bf16" else 4)


def _fill_rows(make_row, rows: Sequence[int], V: int, dtype, threads: int = 0) -> np.ndarray:
    out = np.empty((len(rows), V), dtype=dtype)

    def work(i):
        out[i] = make_row(int(rows[i]))

    n = threads or min(16, max(1, len(rows) // 64 + 1))
    if n == 1 or len(rows) < 64:
        for i in range(len(rows)):
            work(i)
    else:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(work, range(len(rows)), chunksize=max(1, len(rows) // (4 * n))))
    return out


def _choose_rows(B: int, L: int, rows):
    if rows is None:
        return np.arange(B * L, dtype=np.int64), None
    rows = np.asarray(rows, dtype=np.int64)
    return rows, rows


def _candidates_fraction(seed: int, tag: int, B: int, L: int, n_cand: int) -> np.ndarray:
    cand = np.zeros((B, L), dtype=np.uint8)
    for b in range(B):
        perm = _rng(seed, tag, 7, b).permutation(L)
        cand[b, perm[:n_cand]] = 1
    return cand


def tiny(seed: int = 0, rows=None) -> Workload:
    """B=1, L=64, V=4096 fp32 z ~ N(0, 3^2); 16 rows get +8 at an id in [0, 4095)."""
    B, L, V = 1, 64, 4096
    tag = _TAGS["tiny"]
    pick = _rng(seed, tag, 1)
    peak_rows = pick.choice(B * L, size=16, replace=False)
    peak_ids = pick.integers(0, V - 1, size=16)
    peaks = dict(zip(peak_rows.tolist(), peak_ids.tolist()))

    def make_row(r):
        z = _rng(seed, tag, 2, r).normal(0.0, 3.0, size=V).astype(np.float32)
        if r in peaks:
            z[peaks[r]] += np.float32(8.0)
        return z

    rows_idx, rows_out = _choose_rows(B, L, rows)
    logits = _fill_rows(make_row, rows_idx, V, np.float32)
    return Workload("tiny", B, L, V, "f32", logits, rows_out, [V - 1], 0.0, 0,
                    "threshold", np.ones((B, L), dtype=np.uint8),
                    {"tau": 0.9, "strict": False})


# Inverse-temperature range for the LLaDA-shaped rows: log-uniform in
# [3, 60] gives top-1 probabilities from about 0.02 to above 0.999 on rows of
# 126464 N(0,1) logits (the spread is checked against the oracle in the tests).
LLADA_SCALE_RANGE = (3.0, 60.0)


def llada(seed: int = 0, rows=None) -> Workload:
    """B=1, L=32 active block rows, V=126464 bf16: N(0,1) times a per-row scale."""
    B, L, V = 1, 32, LLADA_VOCAB
    tag = _TAGS["llada"]
    lo, hi = (math.log(s) for s in LLADA_SCALE_RANGE)

    def make_row(r):
        g = _rng(seed, tag, 2, r)
        scale = np.float32(math.exp(g.uniform(lo, hi)))
        n = g.standard_normal(V, dtype=np.float32)
        return f32_to_bf16_bits(n * scale)

    rows_idx, rows_out = _choose_rows(B, L, rows)
    logits = _fill_rows(make_row, rows_idx, V, np.uint16)
    cand = _candidates_fraction(seed, tag, B, L, 19)       # 60 % of 32
    return Workload("llada", B, L, V, "bf16", logits, rows_out, [LLADA_MASK_ID], 0.0, 0,
                    "threshold", cand, {"tau": 0.95, "strict": True})


def dream(seed: int = 0, rows=None) -> Workload:
    """B=8, L=256, V=152064 bf16; half the rows of each batch row carry a +10 peak.

    Gumbel-max at temperature 0.7 with a per-step key; top-k with the step-0
    quota of a 256-position canvas over 32 steps.
    """
    B, L, V = 8, 256, DREAM_VOCAB
    tag = _TAGS["dream"]
    sharp = {}
    for b in range(B):
        g = _rng(seed, tag, 1, b)
        perm = g.permutation(L)[: L // 2]
        ids = g.integers(0, V, size=L // 2)
        for l, v in zip(perm.tolist(), ids.tolist()):
            sharp[b * L + l] = v

    def make_row(r):
        z = _rng(seed, tag, 2, r).standard_normal(V, dtype=np.float32)
        if r in sharp:
            z[sharp[r]] += np.float32(10.0)
        return f32_to_bf16_bits(z)

    rows_idx, rows_out = _choose_rows(B, L, rows)
    logits = _fill_rows(make_row, rows_idx, V, np.uint16)
    key = int(_rng(seed, tag, 3).integers(0, 2**63 - 1)) * 2 + 1
    return Workload("dream", B, L, V, "bf16", logits, rows_out, [], 0.7, key,
                    "topk", np.ones((B, L), dtype=np.uint8),
                    {"masked_count": L, "steps": 32})


def large(seed: int = 0, rows=None) -> Workload:
    """B=32, L=512, V=126464 fp32 N(0, 2^2); every row gets a U(0,12) peak."""
    B, L, V = 32, 512, LLADA_VOCAB
    tag = _TAGS["large"]

    def make_row(r):
        g = _rng(seed, tag, 2, r)
        h = np.float32(g.uniform(0.0, 12.0))
        pid = int(g.integers(0, V - 1))
        if pid >= LLADA_MASK_ID:
            pid += 1                      # never the suppressed mask id
        z = g.normal(0.0, 2.0, size=V).astype(np.float32)
        z[pid] += h
        return z

    rows_idx, rows_out = _choose_rows(B, L, rows)
    logits = _fill_rows(make_row, rows_idx, V, np.float32)
    cand = _candidates_fraction(seed, tag, B, L, 256)
    return Workload("large", B, L, V, "f32", logits, rows_out, [LLADA_MASK_ID], 0.0, 0,
                    "factor+entropy_bound", cand, {"factor": 1.0, "gamma": 0.1})


def build(name: str, seed: int = 0, rows=None) -> Workload:
    return {"tiny": tiny, "llada": llada, "dream": dream, "large": large}[name](seed, rows)


# --------------------------------------------------------------------------
# Block-decode loop (LLaDA2.1-style decoding with editing).
#
# Every canvas position p of batch row b has a target id T[b, p] (never the
# mask id) and a base peak height h0[b, p] ~ U(0, 4).  At step s of a block,
# the row emitted for position p is a background row from a bank of seeded
# N(0,1) rows plus a peak of height h0 + s at T[b, p].  The peak starts below
# the background's maximum (about 4.4 over 126464 ids), so the commits forced
# in early steps take background tokens, and the editing rule rewrites them
# once their target's peak has grown.  The bank keeps per-step generation
# cheap on both sides; which bank row a position gets is drawn afresh at every
# step.
# --------------------------------------------------------------------------

@dataclasses.dataclass
class LoopSpec:
    B: int = 4
    P: int = 128
    gen_len: int = 1024
    block_len: int = 32
    V: int = LLADA_VOCAB
    mask_id: int = LLADA_MASK_ID
    tau: float = 0.95
    tau_edit: float = 0.9
    max_post_steps: int = 4
    seed: int = 0
    bank_rows: int = 64
    delta: float = 1.0


class LoopGenerator:
    """Per-step logits for the block-decode loop (host numpy and device torch forms)."""

    def __init__(self, spec: LoopSpec):
        self.spec = spec
        s = spec
        tag = _TAGS["loop"]
        total = -(-(s.P + s.gen_len) // s.block_len) * s.block_len
        self.total = total
        g = _rng(s.seed, tag, 1)
        t = g.integers(0, s.V - 1, size=(s.B, total))
        t[t >= s.mask_id] += 1
        self.targets = t.astype(np.int64)
        self.h0 = g.uniform(0.0, 4.0, size=(s.B, total)).astype(np.float32)
        self.prompt = _rng(s.seed, tag, 2).integers(0, s.mask_id, size=(s.B, s.P)).astype(np.int32)

        def make_row(r):
            return _rng(s.seed, tag, 3, r).standard_normal(s.V, dtype=np.float32)

        self.bank_src = _fill_rows(make_row, np.arange(s.bank_rows), s.V, np.float32)
        self.bank_bits = f32_to_bf16_bits(self.bank_src)        # (bank_rows, V) uint16
        self._dev = None

    def _pick(self, block: int, step: int, n_cols: int) -> np.ndarray:
        s = self.spec
        return _rng(s.seed, _TAGS["loop"], 4, block, step).integers(0, s.bank_rows, size=(s.B, n_cols))

    def _peaks(self, block: int, step: int, col0: int, n_cols: int):
        s = self.spec
        pick = self._pick(block, step, n_cols)
        cols = np.arange(col0, col0 + n_cols)
        tgt = self.targets[:, cols]                                  # (B, n)
        h = self.h0[:, cols] + np.float32(s.delta * step)            # (B, n) f32
        base = self.bank_src[pick, tgt]                              # (B, n) f32
        val = f32_to_bf16_bits((base + h).astype(np.float32))       # f32 add, then bf16
        return pick, tgt, val

    def host_logits(self, block: int, step: int, col0: int, n_cols: int) -> np.ndarray:
        """(B*n_cols, V) uint16 bf16 bits of the rows for canvas columns [col0, col0+n_cols)."""
        s = self.spec
        pick, tgt, val = self._peaks(block, step, col0, n_cols)
        out = self.bank_bits[pick.reshape(-1)].copy()
        out[np.arange(s.B * n_cols), tgt.reshape(-1)] = val.reshape(-1)
        return out

    def device_logits(self, block: int, step: int, col0: int, n_cols: int, out=None):
        """The same rows as :meth:`host_logits`, assembled on the GPU with torch."""
        import torch

        s = self.spec
        if self._dev is None:
            self._dev = torch.from_numpy(self.bank_bits.view(np.int16)).cuda().view(torch.bfloat16)
        pick, tgt, val = self._peaks(block, step, col0, n_cols)
        idx = torch.from_numpy(pick.reshape(-1)).cuda()
        rows = torch.index_select(self._dev, 0, idx)
        if out is not None:
            out[: rows.shape[0]].copy_(rows)
            rows = out[: rows.shape[0]]
        flat = rows.view(torch.int16).view(-1)
        pos = torch.from_numpy((np.arange(s.B * n_cols) * s.V + tgt.reshape(-1)).astype(np.int64)).cuda()
        flat.index_copy_(0, pos, torch.from_numpy(val.reshape(-1).view(np.int16)).cuda())
        return rows


def loop_spec(seed: int = 0) -> LoopSpec:
    return LoopSpec(seed=seed)


# --------------------------------------------------------------------------
# Uniform-noise decoding (DiffusionGemma-style canvas denoising).
#
# A stand-in for the model: every canvas position (b, j) has a target id and
# an onset step.  Before its onset the position's logits are a background row
# (one of a bank of seeded N(0, 1) rows, drawn afresh at every step), so its
# prediction is uncertain (entropy near ln V) and its argmax wanders; from its
# onset on, the row also carries a peak of height `peak` at the target, so the
# prediction is confident and stable.  The canvas the loop feeds back is not
# read (self-conditioning stays with a real model).  Entropies are thus
# either tiny or large, far from the acceptance budget and the stopping
# threshold, which keeps every decision of the loop away from rounding.
# --------------------------------------------------------------------------

GEMMA_VOCAB = 262144


@dataclasses.dataclass
class UniformSpec:
    B: int = 1
    N: int = 256                 # canvas length
    V: int = GEMMA_VOCAB
    dtype: str = "bf16"
    num_steps: int = 48
    entropy_bound: float = 0.1
    t_min: float = 0.4
    t_max: float = 0.8
    stability_threshold: int = 1
    confidence_threshold: float = 0.005
    key: int = 0x5EED_0001
    seed: int = 0
    bank_rows: int = 64
    peak: float = 24.0
    max_onset: int = 24          # onsets are uniform in [0, max_onset]


class UniformGenerator:
    """Per-step logits of the uniform-noise loop (host numpy and device torch forms)."""

    def __init__(self, spec: UniformSpec):
        self.spec = s = spec
        tag = _TAGS["uniform"]
        g = _rng(s.seed, tag, 1)
        self.targets = g.integers(0, s.V, size=(s.B, s.N)).astype(np.int64)
        self.onset = g.integers(0, s.max_onset + 1, size=(s.B, s.N)).astype(np.int64)

        def make_row(r):
            return _rng(s.seed, tag, 3, r).standard_normal(s.V, dtype=np.float32)

        self.bank_src = _fill_rows(make_row, np.arange(s.bank_rows), s.V, np.float32)
        self.bank = f32_to_bf16_bits(self.bank_src) if s.dtype == "bf16" else self.bank_src
        self._dev = None

    def _rows(self, step: int):
        s = self.spec
        pick = _rng(s.seed, _TAGS["uniform"], 4, step).integers(0, s.bank_rows, size=(s.B, s.N))
        on = self.onset <= step                                        # (B, N) confident positions
        flat = np.flatnonzero(on.reshape(-1))
        tgt = self.targets.reshape(-1)[flat]
        val = (self.bank_src[pick.reshape(-1)[flat], tgt] + np.float32(s.peak)).astype(np.float32)
        if s.dtype == "bf16":
            val = f32_to_bf16_bits(val)
        return pick.reshape(-1), flat, tgt, val

    def host_logits(self, step: int) -> np.ndarray:
        """(B*N, V) logits of step `step` (uint16 bf16 bits, or float32)."""
        pick, flat, tgt, val = self._rows(step)
        out = self.bank[pick].copy()
        out[flat, tgt] = val
        return out

    def device_logits(self, step: int, out=None):
        """The same rows as :meth:`host_logits`, assembled on the GPU with torch."""
        import torch

        s = self.spec
        if self._dev is None:
            if s.dtype == "bf16":
                self._dev = torch.from_numpy(self.bank.view(np.int16)).cuda().view(torch.bfloat16)
            else:
                self._dev = torch.from_numpy(self.bank).cuda()
        pick, flat, tgt, val = self._rows(step)
        rows = torch.index_select(self._dev, 0, torch.from_numpy(pick).cuda())
        if out is not None:
            out.copy_(rows)
            rows = out
        if flat.size:
            pos = torch.from_numpy((flat * s.V + tgt).astype(np.int64)).cuda()
            if s.dtype == "bf16":
                rows.view(torch.int16).view(-1).index_copy_(0, pos, torch.from_numpy(val.view(np.int16)).cuda())
            else:
                rows.view(-1).index_copy_(0, pos, torch.from_numpy(val).cuda())
        return rows


def uniform_spec(**kw) -> UniformSpec:
    return UniformSpec(**kw)


# --------------------------------------------------------------------------
# Fused LM head + statistics: hidden states and an LM-head weight.
#
# hidden ~ N(0, 1) per element; weight ~ N(0, 1/d), so the logits are about
# N(0, 1); then for every token t the weight row of a seeded target id gets
# + boost h_t / |h_t|^2 added, which raises that token's logit at the target
# by about `boost` (its argmax is then the target unless the boost is small).
# Both returned as bf16 bits; generated in row chunks so any V fits.
# --------------------------------------------------------------------------

def lm_head_inputs(seed: int, T: int, d: int, V: int, boost: float = 8.0):
    tag = 7
    g = _rng(seed, tag, 1)
    hidden = g.standard_normal((T, d), dtype=np.float32)
    weight = np.empty((V, d), dtype=np.uint16)
    targets = _rng(seed, tag, 2).integers(0, V, size=T)
    chunk = 8192
    for c0 in range(0, V, chunk):
        c1 = min(V, c0 + chunk)
        wc = _rng(seed, tag, 3, c0).standard_normal((c1 - c0, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(d))
        for t in np.flatnonzero((targets >= c0) & (targets < c1)):
            h = hidden[t]
            wc[targets[t] - c0] += np.float32(boost) * h / np.float32(h @ h)
        weight[c0:c1] = f32_to_bf16_bits(wc)
    return f32_to_bf16_bits(hidden), weight, targets
