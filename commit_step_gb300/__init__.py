"""Python binding of libdllmcommit, the GB300 commit step of diffusion-LM decoding.

Argument marshalling only: every step runs in the library's CUDA kernels
(``libdllmcommit.so``, built in-tree by ``commit_step_gb300.build``).  PyTorch
supplies device memory and streams.  The functions carry the names of the C
entry points without their ``dllm_`` prefix (``token_stats`` calls
``dllm_token_stats`` and so on); see ``include/dllmcommit.h`` for the contract
of each.

Importing this package raises if the library is missing: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdllmcommit.so")

DLLM_OK = 0
DLLM_F32, DLLM_BF16 = 0, 1
RULE_NONE, RULE_THRESHOLD, RULE_TOPK, RULE_FACTOR, RULE_ENTROPY_BOUND = 0, 1, 2, 3, 4
MAX_SUPPRESS = 64
MAX_SORT_L = 16384
FUSED_SORT_CAP = 1024
FLAG_INPUTS_READY = 1
FLAG_TEST_DROP_COPY = 2   # tests only: see DLLM_FLAG_TEST_DROP_COPY

EXPORTS = (
    "dllm_status_string", "dllm_version", "dllm_token_stats_workspace_size", "dllm_token_stats",
    "dllm_threshold_transfer", "dllm_topk_transfer", "dllm_factor_transfer", "dllm_entropy_bound_transfer",
    "dllm_edit_transfer", "dllm_transfer_schedule", "dllm_block_ranges", "dllm_commit_step",
    "dllm_workspace_fault", "dllm_token_stats_noalloc", "dllm_token_stats_ex", "dllm_linear_temperature",
    "dllm_uniform_canvas", "dllm_renoise", "dllm_stable_confident_stop", "dllm_block_causal_mask",
    "dllm_lm_head_stats_workspace_size", "dllm_lm_head_stats", "dllm_uniform_update", "dllm_commit_step_host",
    "dllm_noalloc_fault",
)


class DllmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


class StatsEx(C.Structure):
    """Mirror of ``dllm_stats_ex``."""

    _fields_ = [("logit_scale", C.c_float), ("margin", C.c_void_p), ("argmax", C.c_void_p)]


class CommitParams(C.Structure):
    """Mirror of ``dllm_commit_params``."""

    _fields_ = [
        ("rule", C.c_int32), ("strict", C.c_int32), ("tau", C.c_float), ("factor", C.c_float),
        ("gamma", C.c_float), ("k", C.c_void_p), ("cand", C.c_void_p), ("mask_id", C.c_int32),
        ("edit", C.c_int32), ("tau_edit", C.c_float), ("commit", C.c_void_p), ("edit_mask", C.c_void_p),
        ("canvas", C.c_void_p), ("canvas_stride", C.c_int64), ("canvas_offset", C.c_int64),
        ("counts", C.c_void_p), ("flags", C.c_int32), ("ex", C.POINTER(StatsEx)),
    ]


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = C.CDLL(LIB_PATH)
    P, i64, i32, f32, u64, sz = C.c_void_p, C.c_int64, C.c_int32, C.c_float, C.c_uint64, C.c_size_t
    lib.dllm_status_string.argtypes = [C.c_int]
    lib.dllm_status_string.restype = C.c_char_p
    lib.dllm_version.restype = C.c_char_p
    lib.dllm_token_stats_workspace_size.argtypes = [i64, i64, i64, C.c_int]
    lib.dllm_token_stats_workspace_size.restype = sz
    stats_args = [P, C.c_int, i64, i64, i64, i64, f32, u64, P, i32, P, P, P]
    lib.dllm_token_stats.argtypes = stats_args + [P, sz, P]
    lib.dllm_commit_step.argtypes = stats_args + [C.POINTER(CommitParams), P, sz, P]
    lib.dllm_commit_step_host.argtypes = [P, P, C.c_int, i64, i64, i64, f32, u64, P, i32, C.POINTER(CommitParams),
                                          P, P, P, sz, P]
    tail = [P, P, i64, i64, P]
    lib.dllm_threshold_transfer.argtypes = [P, P, i64, i64, f32, C.c_int, P] + tail
    lib.dllm_topk_transfer.argtypes = [P, P, i64, i64, P, P] + tail
    lib.dllm_factor_transfer.argtypes = [P, P, i64, i64, f32, P] + tail
    lib.dllm_entropy_bound_transfer.argtypes = [P, P, i64, i64, f32, P] + tail
    lib.dllm_edit_transfer.argtypes = [P, P, P, P, i64, i64, f32, P, P]
    lib.dllm_transfer_schedule.argtypes = [P, i64, i32, P, P]
    lib.dllm_block_ranges.argtypes = [i64, i64, i64, C.c_int, P, i64, P]
    lib.dllm_workspace_fault.argtypes = [P, P, C.POINTER(C.c_int32)]
    lib.dllm_token_stats_noalloc.argtypes = stats_args + [P]
    lib.dllm_noalloc_fault.argtypes = [P, C.POINTER(C.c_int32)]
    lib.dllm_token_stats_ex.argtypes = stats_args[:10] + [C.POINTER(StatsEx)] + stats_args[10:] + [P, sz, P]
    lib.dllm_linear_temperature.argtypes = [i32, i32, f32, f32, C.POINTER(C.c_float)]
    lib.dllm_uniform_canvas.argtypes = [i64, i64, i64, u64, P, i64, P]
    lib.dllm_renoise.argtypes = [P, P, P, P, i64, i64, P, P]
    lib.dllm_stable_confident_stop.argtypes = [P, P, i64, i64, i32, f32, P, P, P, P, P]
    lib.dllm_block_causal_mask.argtypes = [i64, i64, i64, i64, i64, C.c_int, P, i64, P]
    lib.dllm_uniform_update.argtypes = [P, P, P, P, i64, i64, i64, u64, i32, f32, P, P, P, P, P, P]
    lib.dllm_lm_head_stats_workspace_size.argtypes = [i64, i64, i64]
    lib.dllm_lm_head_stats_workspace_size.restype = sz
    lib.dllm_lm_head_stats.argtypes = [P, i64, i64, i64, P, i64, i64, f32, u64, P, i32, P, P, P, P, i64, P, sz, P]
    for name in EXPORTS[3:]:
        if name not in ("dllm_token_stats_workspace_size", "dllm_lm_head_stats_workspace_size"):
            getattr(lib, name).restype = C.c_int
    return lib


_lib = _load()


def status_string(status: int) -> str:
    return _lib.dllm_status_string(int(status)).decode()


def version() -> str:
    return _lib.dllm_version().decode()


def _check(status: int, what: str) -> None:
    if status != DLLM_OK:
        raise DllmError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DLLM_BF16
    if t.dtype == torch.float32:
        return DLLM_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _need_cuda(*ts):
    for t in ts:  # (non-tensors, e.g. an integer k, are converted by the caller)
        if torch.is_tensor(t) and not t.is_cuda:
            raise ValueError("device tensors are required")


_I32, _F32, _MASK = (torch.int32,), (torch.float32,), (torch.uint8, torch.bool)


def _arg(t, name: str, numel: int, dtypes, device) -> None:
    """Checks a tensor the library reads or writes through a raw pointer: on
    ``device``, contiguous, ``numel`` elements of one of ``dtypes`` (the
    kernels index it by row, so anything else would be read or written out
    of bounds).  None passes: the argument is optional."""
    if t is None:
        return
    if not torch.is_tensor(t):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}; the call runs on {device}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must be {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if t.numel() != numel or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor of {numel} elements, got shape {tuple(t.shape)}")


def _canvas_check(canvas, B: int, L: int, canvas_offset: int, device) -> None:
    """A canvas updated at columns canvas_offset .. canvas_offset + L - 1 of
    its first B rows."""
    if canvas is None:
        return
    if not torch.is_tensor(canvas) or canvas.device != device:
        raise ValueError(f"canvas must be a tensor on {device}")
    if canvas.dim() != 2 or canvas.stride(1) != 1 or canvas.dtype != torch.int32:
        raise ValueError("canvas must be a (B, N) int32 tensor with unit column stride")
    off = int(canvas_offset)
    if canvas.shape[0] < B or off < 0 or canvas.shape[1] < off + L:
        raise ValueError(f"canvas {tuple(canvas.shape)} does not hold {B} rows of columns {off} .. {off + L - 1}")


def _stats_out(out, T: int, device) -> None:
    x0, prob, ent = out[:3]
    _arg(x0, "x0", T, _I32, device)
    _arg(prob, "prob", T, _F32, device)
    _arg(ent, "entropy", T, _F32, device)


_WS = {}


def workspace(B: int, L: int, V: int, dtype_code: int, device: torch.device, stream=None) -> torch.Tensor:
    """A zero-filled workspace for the statistics pass, cached per device and stream."""
    need = int(_lib.dllm_token_stats_workspace_size(B, L, V, dtype_code))
    s = torch.cuda.current_stream(device) if stream is None else stream
    key = (device.index, s.cuda_stream)
    ws = _WS.get(key)
    if ws is None or ws.numel() < need:
        with torch.cuda.stream(s):
            ws = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=device)
        _WS[key] = ws
    return ws


def _logits_view(logits: torch.Tensor):
    if logits.dim() == 3:
        B, L, V = logits.shape
        if logits.stride(2) != 1 or logits.stride(0) != L * logits.stride(1):
            raise ValueError("logits must be (B, L, V) with unit stride over V and rows evenly spaced")
        return B, L, V, logits.stride(1)
    if logits.dim() == 2:
        T, V = logits.shape
        if logits.stride(1) != 1:
            raise ValueError("logits must have unit stride over V")
        return 1, T, V, logits.stride(0)
    raise ValueError("logits must be (B, L, V) or (T, V)")


def token_stats(logits: torch.Tensor, temperature: float = 0.0, key: int = 0, suppress_ids: Sequence[int] = (),
                out=None, ws: Optional[torch.Tensor] = None, stream=None):
    """(x0 int32, prob float32, entropy float32), each shaped like logits without V."""
    _need_cuda(logits)
    B, L, V, stride = _logits_view(logits)
    dt = _dtype_code(logits)
    shape = logits.shape[:-1]
    if out is None:
        x0 = torch.empty(shape, dtype=torch.int32, device=logits.device)
        prob = torch.empty(shape, dtype=torch.float32, device=logits.device)
        ent = torch.empty(shape, dtype=torch.float32, device=logits.device)
    else:
        x0, prob, ent = out
        _stats_out(out, B * L, logits.device)
    sup = (C.c_int32 * max(1, len(suppress_ids)))(*[int(v) for v in suppress_ids])
    if ws is None:
        ws = workspace(B, L, V, dt, logits.device, stream)
    _check(_lib.dllm_token_stats(_ptr(logits), dt, B, L, V, stride, float(temperature), int(key) & (2**64 - 1),
                                 sup, len(suppress_ids), _ptr(x0), _ptr(prob), _ptr(ent), _ptr(ws), ws.numel(),
                                 _stream(stream)), "dllm_token_stats")
    return x0, prob, ent


def _stats_ex(shape, device, logit_scale, margin, argmax):
    """The dllm_stats_ex of a call (None when no option departs from the
    plain pass) and the margin / argmax tensors it writes.  ``margin`` and
    ``argmax``: True (allocate), a tensor (write there) or None/False."""
    if margin is True:
        margin = torch.empty(shape, dtype=torch.float32, device=device)
    if argmax is True:
        argmax = torch.empty(shape, dtype=torch.int32, device=device)
    margin = margin if torch.is_tensor(margin) else None
    argmax = argmax if torch.is_tensor(argmax) else None
    n = 1
    for d in shape:
        n *= int(d)
    _arg(margin, "margin", n, _F32, device)
    _arg(argmax, "argmax", n, _I32, device)
    if float(logit_scale) == 1.0 and margin is None and argmax is None:
        return None, None, None
    ex = StatsEx()
    ex.logit_scale = float(logit_scale)
    ex.margin = None if margin is None else margin.data_ptr()
    ex.argmax = None if argmax is None else argmax.data_ptr()
    return ex, margin, argmax


def token_stats_ex(logits: torch.Tensor, temperature: float = 0.0, key: int = 0, suppress_ids: Sequence[int] = (),
                   logit_scale: float = 1.0, margin=True, argmax=True, out=None, ws: Optional[torch.Tensor] = None,
                   stream=None):
    """Statistics of the scaled logits z' = fp32(z * logit_scale), with the
    margin confidence (prob(x0) - prob(runner-up)) and the greedy argmax
    beside a sample.  Returns (x0, prob, entropy, margin, argmax); margin /
    argmax are None when not requested."""
    _need_cuda(logits)
    B, L, V, stride = _logits_view(logits)
    dt = _dtype_code(logits)
    shape = logits.shape[:-1]
    if out is None:
        x0 = torch.empty(shape, dtype=torch.int32, device=logits.device)
        prob = torch.empty(shape, dtype=torch.float32, device=logits.device)
        ent = torch.empty(shape, dtype=torch.float32, device=logits.device)
    else:
        x0, prob, ent = out
        _stats_out(out, B * L, logits.device)
    ex, margin, argmax = _stats_ex(shape, logits.device, logit_scale, margin, argmax)
    sup = (C.c_int32 * max(1, len(suppress_ids)))(*[int(v) for v in suppress_ids])
    if ws is None:
        ws = workspace(B, L, V, dt, logits.device, stream)
    _check(_lib.dllm_token_stats_ex(_ptr(logits), dt, B, L, V, stride, float(temperature), int(key) & (2**64 - 1),
                                    sup, len(suppress_ids), None if ex is None else C.byref(ex), _ptr(x0),
                                    _ptr(prob), _ptr(ent), _ptr(ws), ws.numel(), _stream(stream)),
           "dllm_token_stats_ex")
    return x0, prob, ent, margin, argmax


def _canvas_args(x0, canvas, canvas_offset, B: int, L: int, device):
    if canvas is None:
        return None, None, 0, 0
    if x0 is None:
        raise ValueError("a canvas update needs x0")
    _arg(x0, "x0", B * L, _I32, device)
    _canvas_check(canvas, B, L, canvas_offset, device)
    return _ptr(x0), _ptr(canvas), canvas.stride(0), int(canvas_offset)


def _rule_io(conf, cand, commit):
    _need_cuda(conf, cand)
    if conf.dtype != torch.float32 or conf.dim() != 2 or not conf.is_contiguous():
        raise ValueError("scores must be a contiguous (B, L) float32 tensor")
    if cand.shape != conf.shape or cand.dtype not in (torch.uint8, torch.bool) or not cand.is_contiguous():
        raise ValueError("candidates must be a contiguous (B, L) bool/uint8 tensor")
    if cand.device != conf.device:
        raise ValueError("scores and candidates must be on one device")
    if commit is None:
        commit = torch.empty(conf.shape, dtype=torch.uint8, device=conf.device)
    _arg(commit, "commit", conf.numel(), _MASK, conf.device)
    return conf.shape[0], conf.shape[1], commit


def threshold_transfer(conf, cand, tau: float, strict: bool = False, commit=None, x0=None, canvas=None,
                       canvas_offset: int = 0, stream=None):
    B, L, commit = _rule_io(conf, cand, commit)
    a = _canvas_args(x0, canvas, canvas_offset, B, L, commit.device)
    _check(_lib.dllm_threshold_transfer(_ptr(conf), _ptr(cand), B, L, float(tau), int(bool(strict)), _ptr(commit),
                                        *a, _stream(stream)), "dllm_threshold_transfer")
    return commit


def topk_transfer(conf, cand, k, commit=None, x0=None, canvas=None, canvas_offset: int = 0, stream=None):
    B, L, commit = _rule_io(conf, cand, commit)
    if not torch.is_tensor(k):
        k = torch.full((B,), int(k), dtype=torch.int32, device=conf.device)
    _arg(k, "k", B, _I32, conf.device)
    a = _canvas_args(x0, canvas, canvas_offset, B, L, commit.device)
    _check(_lib.dllm_topk_transfer(_ptr(conf), _ptr(cand), B, L, _ptr(k), _ptr(commit), *a, _stream(stream)),
           "dllm_topk_transfer")
    return commit


def factor_transfer(conf, cand, factor: float, commit=None, x0=None, canvas=None, canvas_offset: int = 0, stream=None):
    B, L, commit = _rule_io(conf, cand, commit)
    a = _canvas_args(x0, canvas, canvas_offset, B, L, commit.device)
    _check(_lib.dllm_factor_transfer(_ptr(conf), _ptr(cand), B, L, float(factor), _ptr(commit), *a, _stream(stream)),
           "dllm_factor_transfer")
    return commit


def entropy_bound_transfer(entropy, cand, gamma: float, commit=None, x0=None, canvas=None, canvas_offset: int = 0,
                           stream=None):
    B, L, commit = _rule_io(entropy, cand, commit)
    a = _canvas_args(x0, canvas, canvas_offset, B, L, commit.device)
    _check(_lib.dllm_entropy_bound_transfer(_ptr(entropy), _ptr(cand), B, L, float(gamma), _ptr(commit), *a,
                                            _stream(stream)), "dllm_entropy_bound_transfer")
    return commit


def edit_transfer(x0, prob, tokens, editable, tau_edit: float, edit=None, stream=None):
    _need_cuda(x0, prob, tokens, editable)
    if not (x0.shape == prob.shape == tokens.shape == editable.shape) or x0.dim() != 2:
        raise ValueError("edit_transfer inputs must share one (B, L) shape")
    for t, dt in ((x0, torch.int32), (prob, torch.float32), (tokens, torch.int32)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError("edit_transfer: x0/tokens int32, prob float32, all contiguous")
    _arg(editable, "editable", x0.numel(), _MASK, x0.device)
    for t in (prob, tokens):
        if t.device != x0.device:
            raise ValueError("edit_transfer inputs must be on one device")
    if edit is None:
        edit = torch.empty(x0.shape, dtype=torch.uint8, device=x0.device)
    _arg(edit, "edit", x0.numel(), _MASK, x0.device)
    B, L = x0.shape
    _check(_lib.dllm_edit_transfer(_ptr(x0), _ptr(prob), _ptr(tokens), _ptr(editable), B, L, float(tau_edit),
                                   _ptr(edit), _stream(stream)), "dllm_edit_transfer")
    return edit


def transfer_schedule(counts, steps: int, quotas=None, stream=None):
    _need_cuda(counts)
    if counts.dtype != torch.int32 or counts.dim() != 1 or not counts.is_contiguous():
        raise ValueError("counts must be a contiguous (B,) int32 tensor")
    B = counts.numel()
    if quotas is None:
        quotas = torch.empty((B, max(int(steps), 0)), dtype=torch.int32, device=counts.device)
    _arg(quotas, "quotas", B * max(int(steps), 0), _I32, counts.device)
    _check(_lib.dllm_transfer_schedule(_ptr(counts), B, int(steps), _ptr(quotas), _stream(stream)),
           "dllm_transfer_schedule")
    return quotas


def block_ranges(P: int, gen_len: int, block_len: int, align: bool = False):
    n = C.c_int64(0)
    st = _lib.dllm_block_ranges(int(P), int(gen_len), int(block_len), int(bool(align)), None, 0, C.byref(n))
    if st not in (DLLM_OK, 3):
        _check(st, "dllm_block_ranges")
    buf = (C.c_int64 * max(1, 2 * n.value))()
    _check(_lib.dllm_block_ranges(int(P), int(gen_len), int(block_len), int(bool(align)), buf, n.value, C.byref(n)),
           "dllm_block_ranges")
    return [(buf[2 * i], buf[2 * i + 1]) for i in range(n.value)]


def _fused_args(B: int, L: int, device, rule, edit, k, cand, canvas, canvas_offset, counts, commit=None,
                edit_mask=None, check_commit=False) -> None:
    """Checks the device tensors of a fused step (dllm_commit_step and its
    host-buffer form)."""
    T = B * L
    _arg(cand, "cand", T, _MASK, device)
    _arg(k, "k", B, _I32, device)
    _arg(counts, "counts", 3 * B, _I32, device)
    _canvas_check(canvas, B, L, canvas_offset, device)
    if check_commit and rule != RULE_NONE:
        if commit is None:
            raise ValueError("a commit rule needs a commit mask")
        _arg(commit, "commit", T, _MASK, device)
    if edit:
        if edit_mask is None:
            raise ValueError("the edit rule needs an edit mask")
        _arg(edit_mask, "edit_mask", T, _MASK, device)


def _commit_params(rule, strict, tau, factor, gamma, k, cand, mask_id, edit, tau_edit, commit, edit_mask, canvas,
                   canvas_offset, counts, inputs_ready, ex) -> CommitParams:
    """The dllm_commit_params of a call (device tensors or None)."""
    p = CommitParams()
    p.rule, p.strict, p.tau, p.factor, p.gamma = int(rule), int(bool(strict)), float(tau), float(factor), float(gamma)
    p.k = None if k is None else k.data_ptr()
    p.cand = None if cand is None else cand.data_ptr()
    p.mask_id = int(mask_id)
    p.edit, p.tau_edit = int(bool(edit)), float(tau_edit)
    p.commit = None if commit is None else commit.data_ptr()
    p.edit_mask = None if edit_mask is None else edit_mask.data_ptr()
    if canvas is not None:   # checked by the caller (_fused_args)
        p.canvas, p.canvas_stride, p.canvas_offset = canvas.data_ptr(), canvas.stride(0), int(canvas_offset)
    p.counts = None if counts is None else counts.data_ptr()
    p.flags = FLAG_INPUTS_READY if inputs_ready else 0
    if ex is not None:
        p.ex = C.pointer(ex)
    return p


def commit_step(logits, *, rule: int, temperature: float = 0.0, key: int = 0, suppress_ids: Sequence[int] = (),
                cand=None, mask_id: int = -1, tau: float = 0.0, strict: bool = False, k=None, factor: float = 0.0,
                gamma: float = 0.0, edit: bool = False, tau_edit: float = 1.0, canvas=None, canvas_offset: int = 0,
                out=None, counts=None, ws=None, stream=None, inputs_ready: bool = False,
                logit_scale: float = 1.0, margin: Optional[torch.Tensor] = None,
                argmax: Optional[torch.Tensor] = None, _test_flags: int = 0):
    """Fused statistics pass + commit rule (+ edit rule and canvas update) in one launch.

    ``logit_scale``, ``margin`` and ``argmax`` (preallocated (B, L) float32 /
    int32 tensors) are the extended statistics of ``token_stats_ex``; the
    rules then decide on the statistics of the scaled logits.

    ``inputs_ready`` sets DLLM_FLAG_INPUTS_READY: only when neither the logits
    nor ``cand`` were written by the kernel that precedes this call in the
    stream.

    Returns (x0, prob, entropy, commit, edit_mask); commit/edit_mask are None
    when not requested.
    """
    _need_cuda(logits, cand, canvas, k, counts)
    B, L, V, stride = _logits_view(logits)
    dt = _dtype_code(logits)
    dev = logits.device
    if out is None:
        x0 = torch.empty((B, L), dtype=torch.int32, device=dev)
        prob = torch.empty((B, L), dtype=torch.float32, device=dev)
        ent = torch.empty((B, L), dtype=torch.float32, device=dev)
        commit = torch.empty((B, L), dtype=torch.uint8, device=dev) if rule != RULE_NONE else None
        edit_mask = torch.empty((B, L), dtype=torch.uint8, device=dev) if edit else None
    else:
        x0, prob, ent, commit, edit_mask = out
        _stats_out(out, B * L, dev)
    if rule == RULE_TOPK and not torch.is_tensor(k):
        k = torch.full((B,), int(k), dtype=torch.int32, device=dev)
    _fused_args(B, L, dev, rule, edit, k, cand, canvas, canvas_offset, counts, commit, edit_mask, check_commit=True)
    ex, _, _ = _stats_ex((B, L), dev, logit_scale, margin, argmax)
    p = _commit_params(rule, strict, tau, factor, gamma, k, cand, mask_id, edit, tau_edit, commit, edit_mask, canvas,
                       canvas_offset, counts, inputs_ready, ex)
    p.flags |= int(_test_flags)
    sup = (C.c_int32 * max(1, len(suppress_ids)))(*[int(v) for v in suppress_ids])
    if ws is None:
        ws = workspace(B, L, V, dt, dev, stream)
    _check(_lib.dllm_commit_step(_ptr(logits), dt, B, L, V, stride, float(temperature), int(key) & (2**64 - 1),
                                 sup, len(suppress_ids), _ptr(x0), _ptr(prob), _ptr(ent), C.byref(p), _ptr(ws),
                                 ws.numel(), _stream(stream)), "dllm_commit_step")
    return x0, prob, ent, commit, edit_mask


class HostStep:
    """A commit step on logits held in host memory, prepared once and queued
    with one C call (dllm_commit_step_host) each time it is called: the copy
    of the logits to the device, the fused statistics pass + commit rule, and
    one copy of x0 / prob / entropy / commit back to host memory, in order on
    one stream (fixed at construction).

    ``host_logits``: a contiguous CPU tensor (B, L, V) or (T, V), bf16 or
    fp32; pin it for the copies to run asynchronously.  Its contents are read
    when the stream reaches the step, so a caller may refill it between
    steps once the previous step has finished.  After the stream reaches the
    step, ``x0``, ``prob``, ``entropy`` and ``commit`` (views of one pinned
    host buffer) hold the results.  ``cand``, ``k``, ``canvas``, ``counts``,
    ``margin`` and ``argmax`` are device tensors as in commit_step; an edit
    mask, when ``edit`` is set, is written to the device tensor ``edit_mask``.
    """

    def __init__(self, host_logits: torch.Tensor, *, rule: int, temperature: float = 0.0, key: int = 0,
                 suppress_ids: Sequence[int] = (), cand=None, mask_id: int = -1, tau: float = 0.0,
                 strict: bool = False, k=None, factor: float = 0.0, gamma: float = 0.0, edit: bool = False,
                 edit_mask=None, tau_edit: float = 1.0, canvas=None, canvas_offset: int = 0, counts=None,
                 device=None, ws=None, stream=None, logit_scale: float = 1.0, margin=None, argmax=None):
        if host_logits.is_cuda or not host_logits.is_contiguous():
            raise ValueError("host_logits must be a contiguous CPU tensor")
        B, L, V, _ = _logits_view(host_logits)
        dt = _dtype_code(host_logits)
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        if dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        _need_cuda(cand, canvas, k, counts, edit_mask)
        T = B * L
        self.dev_logits = torch.empty(host_logits.shape, dtype=host_logits.dtype, device=dev)
        self.dev_out = torch.empty(max(1, 13 * T), dtype=torch.uint8, device=dev)
        self.host_out = torch.empty(max(1, 13 * T), dtype=torch.uint8).pin_memory()
        self.x0 = self.host_out[0:4 * T].view(torch.int32).view(B, L)
        self.prob = self.host_out[4 * T:8 * T].view(torch.float32).view(B, L)
        self.entropy = self.host_out[8 * T:12 * T].view(torch.float32).view(B, L)
        self.commit = self.host_out[12 * T:13 * T].view(B, L) if rule != RULE_NONE else None
        if rule == RULE_TOPK and not torch.is_tensor(k):
            k = torch.full((B,), int(k), dtype=torch.int32, device=dev)
        if edit and edit_mask is None:
            edit_mask = torch.empty((B, L), dtype=torch.uint8, device=dev)
        self.edit_mask = edit_mask if edit else None
        _fused_args(B, L, dev, rule, edit, k, cand, canvas, canvas_offset, counts, None, self.edit_mask)
        ex, _, _ = _stats_ex((B, L), dev, logit_scale, margin, argmax)
        self._ex = ex
        self._p = _commit_params(rule, strict, tau, factor, gamma, k, cand, mask_id, edit, tau_edit, None,
                                 self.edit_mask, canvas, canvas_offset, counts, False, ex)
        self._sup = (C.c_int32 * max(1, len(suppress_ids)))(*[int(v) for v in suppress_ids])
        if ws is None:
            ws = workspace(B, L, V, dt, dev, stream)
        self._keep = (host_logits, cand, k, canvas, counts, margin, argmax, ws)
        self._args = (C.c_void_p(host_logits.data_ptr()), _ptr(self.dev_logits), dt, B, L, V, float(temperature),
                      int(key) & (2**64 - 1), self._sup, len(suppress_ids), C.byref(self._p), _ptr(self.dev_out),
                      C.c_void_p(self.host_out.data_ptr()), _ptr(ws), ws.numel(), _stream(stream))

    def __call__(self):
        _check(_lib.dllm_commit_step_host(*self._args), "dllm_commit_step_host")
        return self.x0, self.prob, self.entropy, self.commit


def commit_step_host(host_logits: torch.Tensor, **kw):
    """One commit step on host-resident logits (see HostStep); returns host
    tensors (x0, prob, entropy, commit), valid once the stream reaches the
    step."""
    return HostStep(host_logits, **kw)()


def _on_current_device(device: torch.device, current: int, stream_device=None) -> None:
    """The allocation-free entry takes its scratch array, the device's launch
    limits and (without a stream) the default stream from the current CUDA
    device, so its tensors (and a given stream) must be on that device."""
    if device.type != "cuda" or device.index != current:
        raise ValueError(f"tensors on {device} but the current CUDA device is cuda:{current}: "
                         "make their device current first")
    if stream_device is not None and stream_device != current:
        raise ValueError(f"stream on cuda:{stream_device} but the current CUDA device is cuda:{current}")


def token_stats_noalloc(logits: torch.Tensor, temperature: float = 0.0, key: int = 0,
                        suppress_ids: Sequence[int] = (), out=None, stream=None):
    """token_stats without a workspace: the library's fixed scratch array is
    used instead (see dllm_token_stats_noalloc); calls must not overlap.  The
    tensors must be on the current CUDA device.  A kernel fault of the call
    is read with noalloc_fault() before the next call."""
    _need_cuda(logits)
    _on_current_device(logits.device, torch.cuda.current_device(),
                       None if stream is None else stream.device.index)
    B, L, V, stride = _logits_view(logits)
    dt = _dtype_code(logits)
    shape = logits.shape[:-1]
    if out is None:
        out = (torch.empty(shape, dtype=torch.int32, device=logits.device),
               torch.empty(shape, dtype=torch.float32, device=logits.device),
               torch.empty(shape, dtype=torch.float32, device=logits.device))
    x0, prob, ent = out
    _stats_out(out, B * L, logits.device)
    sup = (C.c_int32 * max(1, len(suppress_ids)))(*[int(v) for v in suppress_ids])
    _check(_lib.dllm_token_stats_noalloc(_ptr(logits), dt, B, L, V, stride, float(temperature),
                                         int(key) & (2**64 - 1), sup, len(suppress_ids), _ptr(x0), _ptr(prob),
                                         _ptr(ent), _stream(stream)), "dllm_token_stats_noalloc")
    return x0, prob, ent


def noalloc_fault(stream=None) -> int:
    """The fault code the last token_stats_noalloc call on the current device
    left in the library's array (0: none); synchronises the stream and clears
    the code."""
    f = C.c_int32(0)
    _check(_lib.dllm_noalloc_fault(_stream(stream), C.byref(f)), "dllm_noalloc_fault")
    return f.value


def workspace_fault(ws: torch.Tensor, stream=None) -> int:
    """The fault code a kernel left in ``ws`` (0: none).  After a fault the
    workspace's counters may be left non-zero, so the whole tensor is zeroed
    here, on the same stream, before it can be used again."""
    f = C.c_int32(0)
    _check(_lib.dllm_workspace_fault(_ptr(ws), _stream(stream), C.byref(f)), "dllm_workspace_fault")
    if f.value != 0:
        with torch.cuda.stream(torch.cuda.current_stream(ws.device) if stream is None else stream):
            ws.zero_()
    return f.value


def lib_handle() -> C.CDLL:
    return _lib


# ---------------------------------------------------------------------------
# uniform-noise decoding helpers
# ---------------------------------------------------------------------------
def linear_temperature(remaining: int, num_steps: int, t_min: float = 0.4, t_max: float = 0.8) -> float:
    """fp32(t_min + (t_max - t_min) * remaining / num_steps) (host)."""
    T = C.c_float(0.0)
    _check(_lib.dllm_linear_temperature(int(remaining), int(num_steps), float(t_min), float(t_max), C.byref(T)),
           "dllm_linear_temperature")
    return T.value


def uniform_canvas(B: int, N: int, V: int, key: int, out: Optional[torch.Tensor] = None, device=None,
                   stream=None) -> torch.Tensor:
    """(B, N) int32 uniformly random tokens of [0, V) keyed by ``key``."""
    if out is None:
        out = torch.empty((B, N), dtype=torch.int32, device=device or "cuda")
    _need_cuda(out)
    if out.shape != (B, N) or out.dtype != torch.int32 or out.stride(1) != 1:
        raise ValueError("out must be a (B, N) int32 tensor with unit column stride")
    _check(_lib.dllm_uniform_canvas(B, N, V, int(key) & (2**64 - 1), _ptr(out), out.stride(0), _stream(stream)),
           "dllm_uniform_canvas")
    return out


def renoise(sample: torch.Tensor, accepted: Optional[torch.Tensor], noise: Optional[torch.Tensor],
            out: Optional[torch.Tensor] = None, frozen: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out = accepted ? sample : noise over a contiguous (B, N) canvas; rows
    with frozen[b] != 0 keep ``out``."""
    _need_cuda(sample, accepted, noise, out, frozen)
    if sample.dim() != 2 or sample.dtype != torch.int32 or not sample.is_contiguous():
        raise ValueError("sample must be a contiguous (B, N) int32 tensor")
    B, N = sample.shape
    for t, dt in ((accepted, (torch.uint8, torch.bool)), (noise, (torch.int32,))):
        if t is not None and (t.shape != sample.shape or t.dtype not in dt or not t.is_contiguous()):
            raise ValueError("accepted / noise must be contiguous and shaped like sample")
    for t in (accepted, noise):
        if t is not None and t.device != sample.device:
            raise ValueError("renoise inputs must be on one device")
    _arg(frozen, "frozen", B, _MASK, sample.device)
    if out is None:
        out = torch.empty_like(sample)
    _arg(out, "out", B * N, _I32, sample.device)
    _check(_lib.dllm_renoise(_ptr(sample), _ptr(accepted), _ptr(noise), _ptr(frozen), B, N, _ptr(out),
                             _stream(stream)), "dllm_renoise")
    return out


class StableConfidentStopping:
    """The stable-and-confident stopping criterion with its device state
    (the previous argmax canvas and the count of consecutive stable calls)."""

    def __init__(self, B: int, L: int, stability_threshold: int = 1, confidence_threshold: float = 0.005,
                 device=None):
        dev = device or "cuda"
        self.prev = torch.zeros((B, L), dtype=torch.int32, device=dev)
        self.count = torch.full((B,), -1, dtype=torch.int32, device=dev)
        self.stability_threshold = int(stability_threshold)
        self.confidence_threshold = float(confidence_threshold)

    def __call__(self, argmax: torch.Tensor, entropy: torch.Tensor, done: Optional[torch.Tensor] = None,
                 stop: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        _need_cuda(argmax, entropy, done, stop)
        B, L = self.prev.shape
        if argmax.shape != (B, L) or entropy.shape != (B, L) or not argmax.is_contiguous() or \
                not entropy.is_contiguous() or argmax.dtype != torch.int32 or entropy.dtype != torch.float32:
            raise ValueError("argmax / entropy must be contiguous (B, L) int32 / float32 tensors")
        dev = self.prev.device
        if argmax.device != dev or entropy.device != dev:
            raise ValueError(f"argmax / entropy must be on the criterion's device {dev}")
        _arg(done, "done", B, _MASK, dev)
        if stop is None:
            stop = torch.empty((B,), dtype=torch.uint8, device=dev)
        _arg(stop, "stop", B, _MASK, dev)
        _check(_lib.dllm_stable_confident_stop(_ptr(argmax), _ptr(entropy), B, L, self.stability_threshold,
                                               self.confidence_threshold, _ptr(self.prev), _ptr(self.count),
                                               _ptr(stop), _ptr(done), _stream(stream)),
               "dllm_stable_confident_stop")
        return stop


MASK_F32, MASK_BF16, MASK_KEEP_U8 = 0, 1, 2


def block_causal_mask(L: int, block_len: int, Lk: Optional[int] = None, q_offset: int = 0, k_offset: int = 0,
                      dtype=torch.float32, out: Optional[torch.Tensor] = None, device=None,
                      stream=None) -> torch.Tensor:
    """(L, Lk) block-causal attention mask: additive (float32 / bfloat16: 0
    attend, -inf blocked) or, with dtype=torch.bool / torch.uint8, the keep
    mask (True / 1 attend)."""
    Lk = L if Lk is None else Lk
    kinds = {torch.float32: MASK_F32, torch.bfloat16: MASK_BF16, torch.uint8: MASK_KEEP_U8, torch.bool: MASK_KEEP_U8}
    if out is None:
        out = torch.empty((L, Lk), dtype=dtype, device=device or "cuda")
    _need_cuda(out)
    if out.dim() != 2 or out.shape != (L, Lk) or out.stride(1) != 1 or out.dtype not in kinds:
        raise ValueError("out must be an (L, Lk) float32 / bfloat16 / uint8 / bool tensor with unit column stride")
    _check(_lib.dllm_block_causal_mask(L, Lk, q_offset, k_offset, block_len, kinds[out.dtype], _ptr(out),
                                       out.stride(0), _stream(stream)), "dllm_block_causal_mask")
    return out


_WS_LH = {}


def lm_head_stats(hidden: torch.Tensor, weight: torch.Tensor, temperature: float = 0.0, key: int = 0,
                  suppress_ids: Sequence[int] = (), out=None, logits: Optional[torch.Tensor] = None,
                  ws: Optional[torch.Tensor] = None, stream=None):
    """The LM head fused with the statistics pass: x0, prob, entropy of the
    logits hidden @ weight^T (bf16 in, fp32 tensor-core accumulation) without
    storing them.  hidden (T, d) and weight (V, d) bf16 with unit column
    stride; ``logits`` (T, V) float32, if given, receives the logits too."""
    _need_cuda(hidden, weight, logits)
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16 or hidden.dim() != 2 or weight.dim() != 2:
        raise TypeError("hidden and weight must be 2-D bfloat16 tensors")
    if hidden.stride(1) != 1 or weight.stride(1) != 1 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden (T, d) and weight (V, d) need unit column stride and the same d")
    T, d = hidden.shape
    V = weight.shape[0]
    if weight.device != hidden.device or (logits is not None and logits.device != hidden.device):
        raise ValueError("hidden, weight and logits must be on one device")
    if out is None:
        out = (torch.empty((T,), dtype=torch.int32, device=hidden.device),
               torch.empty((T,), dtype=torch.float32, device=hidden.device),
               torch.empty((T,), dtype=torch.float32, device=hidden.device))
    x0, prob, ent = out
    _stats_out(out, T, hidden.device)
    if logits is not None and (logits.dtype != torch.float32 or logits.shape != (T, V) or logits.stride(1) != 1):
        raise ValueError("logits must be a (T, V) float32 tensor with unit column stride")
    if ws is None:
        need = int(_lib.dllm_lm_head_stats_workspace_size(T, V, d))
        key_ = (hidden.device.index,)
        ws = _WS_LH.get(key_)
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device=hidden.device)
            _WS_LH[key_] = ws
    sup = (C.c_int32 * max(1, len(suppress_ids)))(*[int(v) for v in suppress_ids])
    _check(_lib.dllm_lm_head_stats(_ptr(hidden), T, d, hidden.stride(0), _ptr(weight), V, weight.stride(0),
                                   float(temperature), int(key) & (2**64 - 1), sup, len(suppress_ids), _ptr(x0),
                                   _ptr(prob), _ptr(ent), _ptr(logits), 0 if logits is None else logits.stride(0),
                                   _ptr(ws), ws.numel(), _stream(stream)), "dllm_lm_head_stats")
    return x0, prob, ent


def uniform_update(sample: torch.Tensor, accepted: torch.Tensor, step_argmax: torch.Tensor, entropy: torch.Tensor,
                   V: int, noise_key: int, stop: "StableConfidentStopping", canvas: torch.Tensor,
                   argmax: torch.Tensor, done: torch.Tensor, stream=None) -> None:
    """The rest of one uniform-noise step in one launch: re-noise the canvas
    (rows not done), take the step's argmax into ``argmax`` (rows not done),
    and update ``stop``'s state and the done flags (dllm_uniform_update)."""
    B, N = sample.shape
    _need_cuda(sample, accepted, step_argmax, entropy, canvas, argmax, done)
    dev = sample.device
    for t, name, dts in ((sample, "sample", _I32), (accepted, "accepted", _MASK), (step_argmax, "step_argmax", _I32),
                         (entropy, "entropy", _F32), (canvas, "canvas", _I32), (argmax, "argmax", _I32)):
        if t.shape != (B, N):
            raise ValueError("uniform_update takes contiguous (B, N) tensors")
        _arg(t, name, B * N, dts, dev)
    _arg(done, "done", B, _MASK, dev)
    if stop.prev.shape != (B, N) or stop.prev.device != dev:
        raise ValueError("the stopping criterion's state must be (B, N) on the same device")
    _check(_lib.dllm_uniform_update(_ptr(sample), _ptr(accepted), _ptr(step_argmax), _ptr(entropy), B, N, V,
                                    int(noise_key) & (2**64 - 1), stop.stability_threshold,
                                    stop.confidence_threshold, _ptr(canvas), _ptr(argmax), _ptr(stop.prev),
                                    _ptr(stop.count), _ptr(done), _stream(stream)), "dllm_uniform_update")
