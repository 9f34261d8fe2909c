"""CPU oracle of the diffusion-LM commit step -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct C++ implementation (``dllm_oracle.cpp``) of
what the GPU library computes, with numpy wrappers.  Only ``tests/``, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it; the library path never does.  It shares no code with the GPU
library.

Parity pins: see ``tests/test_oracle_*.py`` (worked examples, closed forms,
invariants, brute force, Philox and the Gumbel chain against independent
implementations and statistics).
"""
from __future__ import annotations

import ctypes as C
import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P, i64, i32, f32, u64 = C.c_void_p, C.c_int64, C.c_int32, C.c_float, C.c_uint64
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_philox4x32_10.restype = None
        L.orc_ln_p.argtypes = [f32]
        L.orc_ln_p.restype = f32
        L.orc_ln_p_many.argtypes = [P, i64, P]
        L.orc_ln_p_many.restype = None
        L.orc_gumbel_score.argtypes = [f32, f32, u64, i64, i64]
        L.orc_gumbel_score.restype = f32
        L.orc_token_stats.argtypes = [P, C.c_int, i64, i64, i64, P, f32, u64, P, i32, P, P, P, C.c_int]
        L.orc_token_stats_ex.argtypes = [P, C.c_int, i64, i64, i64, P, f32, u64, f32, P, i32, P, P, P, P, P,
                                         C.c_int]
        for name in ("orc_threshold_transfer",):
            getattr(L, name).argtypes = [P, P, i64, i64, f32, C.c_int, P]
        L.orc_topk_transfer.argtypes = [P, P, i64, i64, P, P]
        L.orc_factor_transfer.argtypes = [P, P, i64, i64, f32, P]
        L.orc_entropy_bound_transfer.argtypes = [P, P, i64, i64, f32, P]
        L.orc_edit_transfer.argtypes = [P, P, P, P, i64, f32, P]
        L.orc_transfer_schedule.argtypes = [P, i64, i32, P]
        L.orc_block_ranges.argtypes = [i64, i64, i64, C.c_int, P, i64, P]
        L.orc_default_threads.argtypes = []
        L.orc_linear_temperature.argtypes = [i32, i32, f32, f32, P]
        L.orc_uniform_canvas.argtypes = [i64, i64, i64, u64, P]
        L.orc_renoise.argtypes = [P, P, P, i64, P]
        L.orc_stable_confident_stop.argtypes = [P, P, i64, i64, i32, f32, P, P, P]
        L.orc_block_causal_mask.argtypes = [i64, i64, i64, i64, i64, P]
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data if a is not None else None


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def default_threads() -> int:
    return lib().orc_default_threads()


def philox4x32_10(counter, key):
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def ln_p(x: float) -> np.float32:
    return np.float32(lib().orc_ln_p(float(np.float32(x))))


def ln_p_many(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(a)
    lib().orc_ln_p_many(_p(a), a.size, _p(out))
    return out


def gumbel_score(z, temperature, key, row, v) -> np.float32:
    return np.float32(lib().orc_gumbel_score(float(np.float32(z)), float(np.float32(temperature)),
                                             int(key), int(row), int(v)))


def token_stats(logits: np.ndarray, dtype: str = "f32", temperature: float = 0.0, key: int = 0,
                suppress_ids=(), row_ids=None, n_threads: int = 0):
    """(x0 int32, prob float64, entropy float64) per row of ``logits``.

    ``logits``: (n_rows, V) float32, or uint16 bf16 bits with ``dtype="bf16"``.
    ``row_ids``: global row index of each row (feeds the Gumbel counter).
    """
    dt = {"f32": 0, "bf16": 1}[dtype]
    want = np.float32 if dt == 0 else np.uint16
    z = np.ascontiguousarray(logits, dtype=want)
    if z.ndim != 2:
        raise ValueError("logits must be 2-D (rows, V)")
    n, V = z.shape
    rid = None if row_ids is None else np.ascontiguousarray(row_ids, dtype=np.int64)
    sup = np.ascontiguousarray(list(suppress_ids), dtype=np.int32)
    x0 = np.zeros(n, dtype=np.int32)
    prob = np.zeros(n, dtype=np.float64)
    ent = np.zeros(n, dtype=np.float64)
    rc = lib().orc_token_stats(_p(z), dt, n, V, V, _p(rid), float(temperature), int(key) & (2**64 - 1),
                               _p(sup) if sup.size else None, int(sup.size),
                               _p(x0), _p(prob), _p(ent), int(n_threads))
    _check(rc, "token_stats")
    return x0, prob, ent


def token_stats_ex(logits: np.ndarray, dtype: str = "f32", temperature: float = 0.0, key: int = 0,
                   logit_scale: float = 1.0, suppress_ids=(), row_ids=None, n_threads: int = 0):
    """(x0, prob, entropy, margin, argmax) per row of the scaled logits
    z' = fp32(z * logit_scale); margin = prob(x0) - prob(runner-up), argmax
    = the first id of the largest z' (the greedy proposal when sampling)."""
    dt = {"f32": 0, "bf16": 1}[dtype]
    want = np.float32 if dt == 0 else np.uint16
    z = np.ascontiguousarray(logits, dtype=want)
    if z.ndim != 2:
        raise ValueError("logits must be 2-D (rows, V)")
    n, V = z.shape
    rid = None if row_ids is None else np.ascontiguousarray(row_ids, dtype=np.int64)
    sup = np.ascontiguousarray(list(suppress_ids), dtype=np.int32)
    x0 = np.zeros(n, dtype=np.int32)
    am = np.zeros(n, dtype=np.int32)
    prob = np.zeros(n, dtype=np.float64)
    ent = np.zeros(n, dtype=np.float64)
    mar = np.zeros(n, dtype=np.float64)
    rc = lib().orc_token_stats_ex(_p(z), dt, n, V, V, _p(rid), float(temperature), int(key) & (2**64 - 1),
                                  float(np.float32(logit_scale)), _p(sup) if sup.size else None, int(sup.size),
                                  _p(x0), _p(prob), _p(ent), _p(mar), _p(am), int(n_threads))
    _check(rc, "token_stats_ex")
    return x0, prob, ent, mar, am


def _rule_inputs(conf, cand):
    c = np.ascontiguousarray(conf, dtype=np.float32)
    m = np.ascontiguousarray(cand, dtype=np.uint8)
    if c.ndim == 1:
        c, m = c[None], m[None]
    if c.shape != m.shape:
        raise ValueError("conf and candidates differ in shape")
    return c, m, np.zeros(c.shape, dtype=np.uint8)


def threshold_transfer(conf, cand, tau, strict=False):
    c, m, out = _rule_inputs(conf, cand)
    _check(lib().orc_threshold_transfer(_p(c), _p(m), c.shape[0], c.shape[1], float(tau), int(bool(strict)), _p(out)), "threshold")
    return out


def topk_transfer(conf, cand, k):
    c, m, out = _rule_inputs(conf, cand)
    kk = np.ascontiguousarray(np.broadcast_to(np.asarray(k, dtype=np.int32), (c.shape[0],)))
    _check(lib().orc_topk_transfer(_p(c), _p(m), c.shape[0], c.shape[1], _p(kk), _p(out)), "topk")
    return out


def factor_transfer(conf, cand, factor):
    c, m, out = _rule_inputs(conf, cand)
    _check(lib().orc_factor_transfer(_p(c), _p(m), c.shape[0], c.shape[1], float(factor), _p(out)), "factor")
    return out


def entropy_bound_transfer(entropy, cand, gamma):
    c, m, out = _rule_inputs(entropy, cand)
    _check(lib().orc_entropy_bound_transfer(_p(c), _p(m), c.shape[0], c.shape[1], float(gamma), _p(out)), "entropy_bound")
    return out


def edit_transfer(x0, prob, tokens, editable, tau_edit):
    a = np.ascontiguousarray(x0, dtype=np.int32)
    p = np.ascontiguousarray(prob, dtype=np.float32)
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    e = np.ascontiguousarray(editable, dtype=np.uint8)
    if not (a.shape == p.shape == t.shape == e.shape):
        raise ValueError("edit_transfer inputs differ in shape")
    out = np.zeros(a.shape, dtype=np.uint8)
    _check(lib().orc_edit_transfer(_p(a), _p(p), _p(t), _p(e), a.size, float(tau_edit), _p(out)), "edit")
    return out


def transfer_schedule(counts, steps):
    c = np.ascontiguousarray(np.atleast_1d(counts), dtype=np.int32)
    out = np.zeros((c.size, steps), dtype=np.int32) if steps > 0 else np.zeros((c.size, 0), np.int32)
    _check(lib().orc_transfer_schedule(_p(c), c.size, int(steps), _p(out)), "transfer_schedule")
    return out


def block_ranges(P, gen_len, block_len, align=False):
    n = np.zeros(1, dtype=np.int64)
    rc = lib().orc_block_ranges(int(P), int(gen_len), int(block_len), int(bool(align)), None, 0, _p(n))
    if rc not in (0, -2):
        _check(rc, "block_ranges")
    out = np.zeros((int(n[0]), 2), dtype=np.int64)
    _check(lib().orc_block_ranges(int(P), int(gen_len), int(block_len), int(bool(align)), _p(out), out.shape[0], _p(n)), "block_ranges")
    return [tuple(map(int, r)) for r in out]


# ---------------------------------------------------------------------------
# uniform-noise decoding helpers
# ---------------------------------------------------------------------------
def linear_temperature(remaining: int, num_steps: int, t_min: float = 0.4, t_max: float = 0.8) -> np.float32:
    T = C.c_float(0.0)
    _check(lib().orc_linear_temperature(int(remaining), int(num_steps), float(t_min), float(t_max), C.byref(T)),
           "linear_temperature")
    return np.float32(T.value)


def uniform_canvas(B: int, N: int, V: int, key: int) -> np.ndarray:
    out = np.zeros((B, N), dtype=np.int32)
    _check(lib().orc_uniform_canvas(int(B), int(N), int(V), int(key) & (2**64 - 1), _p(out)), "uniform_canvas")
    return out


def renoise(sample, accepted, noise) -> np.ndarray:
    s = np.ascontiguousarray(sample, dtype=np.int32)
    a = np.ascontiguousarray(accepted, dtype=np.uint8)
    n = np.ascontiguousarray(noise, dtype=np.int32)
    if not (s.shape == a.shape == n.shape):
        raise ValueError("renoise: shapes differ")
    out = np.zeros_like(s)
    _check(lib().orc_renoise(_p(s), _p(a), _p(n), s.size, _p(out)), "renoise")
    return out


class StableConfidentStopping:
    """The oracle's stopping criterion with its state (prev canvas, count)."""

    def __init__(self, B: int, L: int, stability_threshold: int = 1, confidence_threshold: float = 0.005):
        self.prev = np.zeros((B, L), dtype=np.int32)
        self.count = np.full(B, -1, dtype=np.int32)
        self.stability_threshold = int(stability_threshold)
        self.confidence_threshold = float(confidence_threshold)

    def __call__(self, argmax, entropy) -> np.ndarray:
        am = np.ascontiguousarray(argmax, dtype=np.int32)
        en = np.ascontiguousarray(entropy, dtype=np.float32)
        B, L = am.shape
        stop = np.zeros(B, dtype=np.uint8)
        _check(lib().orc_stable_confident_stop(_p(am), _p(en), B, L, self.stability_threshold,
                                               self.confidence_threshold, _p(self.prev), _p(self.count), _p(stop)),
               "stable_confident_stop")
        return stop


def block_causal_mask(Lq: int, block_len: int, Lk: int = None, q_offset: int = 0, k_offset: int = 0) -> np.ndarray:
    """(Lq, Lk) additive mask in float64: 0 where query block >= key block, -inf elsewhere."""
    Lk = Lq if Lk is None else Lk
    out = np.zeros((Lq, Lk), dtype=np.float64)
    _check(lib().orc_block_causal_mask(int(Lq), int(Lk), int(q_offset), int(k_offset), int(block_len), _p(out)),
           "block_causal_mask")
    return out


# ---------------------------------------------------------------------------
# fused LM head + statistics
# ---------------------------------------------------------------------------
def lm_head_logits(hidden_bits: np.ndarray, weight_bits: np.ndarray) -> np.ndarray:
    """logits = hidden @ weight^T from bf16 bit arrays, (T, d) and (V, d): the
    exact products summed in double (a library matmul in float64), rounded
    once to fp32 -- what an fp32-accumulating GEMM approximates."""
    h = (np.ascontiguousarray(hidden_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    w = (np.ascontiguousarray(weight_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return (h.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32)


def lm_head_stats(hidden_bits, weight_bits, temperature: float = 0.0, key: int = 0, suppress_ids=(),
                  n_threads: int = 0):
    """token_stats of the LM head's logits (lm_head_logits): x0, prob, entropy per row of hidden."""
    return token_stats(lm_head_logits(hidden_bits, weight_bits), dtype="f32", temperature=temperature, key=key,
                       suppress_ids=suppress_ids, n_threads=n_threads)
