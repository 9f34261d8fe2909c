"""The C-ABI library loads and exports every function include/dllmcommit.h
declares; host-only entry points agree with the oracle.  CPU only (no kernel
is launched)."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "dllmcommit.h")


@pytest.fixture(scope="module")
def lib():
    import importlib.util

    spec = importlib.util.spec_from_file_location("_b", os.path.join(ROOT, "commit_step_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    path = b.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HDR).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dllm_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n


def test_status_and_version(lib):
    lib.dllm_status_string.restype = ctypes.c_char_p
    lib.dllm_version.restype = ctypes.c_char_p
    assert lib.dllm_status_string(0) == b"DLLM_OK"
    assert b"INVALID" in lib.dllm_status_string(1)
    assert b"sm_103a" in lib.dllm_version()


def _ranges(lib, P, gen, bl, align):
    n = ctypes.c_int64(0)
    lib.dllm_block_ranges.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                                                             ctypes.c_void_p]
    st = lib.dllm_block_ranges(P, gen, bl, align, None, 0, ctypes.byref(n))
    assert st in (0, 3)
    buf = (ctypes.c_int64 * max(1, 2 * n.value))()
    assert lib.dllm_block_ranges(P, gen, bl, align, buf, n.value, ctypes.byref(n)) == 0
    return [(buf[2 * i], buf[2 * i + 1]) for i in range(n.value)]


def test_block_ranges_matches_oracle(lib):
    import numpy as np

    rng = np.random.default_rng(41)
    for _ in range(500):
        P, gen, bl = int(rng.integers(0, 400)), int(rng.integers(0, 700)), int(rng.integers(1, 90))
        for align in (0, 1):
            assert _ranges(lib, P, gen, bl, align) == oracle.block_ranges(P, gen, bl, bool(align))


def test_block_ranges_errors(lib):
    n = ctypes.c_int64(0)
    assert lib.dllm_block_ranges(5, 10, 0, 0, None, 0, ctypes.byref(n)) == 1     # block_len <= 0
    assert lib.dllm_block_ranges(-1, 10, 4, 0, None, 0, ctypes.byref(n)) == 1    # P < 0
    assert lib.dllm_block_ranges(5, 10, 4, 0, None, 0, None) == 1                # no n_out
    assert lib.dllm_block_ranges(5, 10, 4, 0, None, 0, ctypes.byref(n)) == 3 and n.value == 3


def test_linear_temperature_matches_oracle(lib):
    """dllm_linear_temperature is host-only: the library's value equals the
    oracle's bit for bit, and bad schedules are rejected."""
    import numpy as np

    f = lib.dllm_linear_temperature
    f.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_float, ctypes.POINTER(ctypes.c_float)]
    f.restype = ctypes.c_int
    out = ctypes.c_float(0.0)
    for num_steps in (1, 7, 48, 1000):
        for remaining in sorted({0, 1, num_steps // 3, num_steps - 1, num_steps}):
            for t_min, t_max in ((0.4, 0.8), (0.05, 3.0), (1.0, 1.0)):
                assert f(remaining, num_steps, t_min, t_max, ctypes.byref(out)) == 0
                assert np.float32(out.value) == oracle.linear_temperature(remaining, num_steps, t_min, t_max)
    assert f(5, 4, 0.4, 0.8, ctypes.byref(out)) == 1       # remaining > num_steps
    assert f(1, 0, 0.4, 0.8, ctypes.byref(out)) == 1       # num_steps <= 0
    assert f(1, 4, 0.0, 0.8, ctypes.byref(out)) == 1       # t_min <= 0
    assert f(1, 4, 0.9, 0.8, ctypes.byref(out)) == 1       # t_max < t_min
    assert f(1, 4, 0.4, 0.8, None) == 1                    # no output


def test_workspace_size_without_device(lib):
    lib.dllm_token_stats_workspace_size.restype = ctypes.c_size_t
    lib.dllm_token_stats_workspace_size.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int]
    a = lib.dllm_token_stats_workspace_size(1, 32, 126464, 1)
    b = lib.dllm_token_stats_workspace_size(32, 512, 126464, 0)
    assert 0 < a < b < (1 << 24)


def test_commit_step_host_checks_arguments_before_any_device_work(lib):
    """dllm_commit_step_host validates on the host and returns before queuing
    anything: an empty shape is a no-op, bad pointers, dtype, alignment or
    rule parameters are DLLM_ERR_INVALID_ARGUMENT (1)."""
    P, i64, i32, f32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_uint64
    fn = lib.dllm_commit_step_host
    fn.argtypes = [P, P, ctypes.c_int, i64, i64, i64, f32, u64, P, i32, P, P, P, P, ctypes.c_size_t, P]
    fn.restype = ctypes.c_int
    params = (ctypes.c_char * 256)()           # a zeroed dllm_commit_params: rule NONE, no candidates
    cp = ctypes.cast(params, P)
    fake = P(4096)                              # never dereferenced: every call below fails its checks
    # empty shape: nothing to do
    assert fn(None, None, 1, 0, 32, 1000, 0.0, 0, None, 0, cp, None, None, None, 0, None) == 0
    # missing pointers / params
    assert fn(None, fake, 1, 1, 32, 1000, 0.0, 0, None, 0, cp, fake, fake, fake, 1 << 20, None) == 1
    assert fn(fake, fake, 1, 1, 32, 1000, 0.0, 0, None, 0, None, fake, fake, fake, 1 << 20, None) == 1
    # bad dtype, misaligned packed output, negative temperature
    assert fn(fake, fake, 7, 1, 32, 1000, 0.0, 0, None, 0, cp, fake, fake, fake, 1 << 20, None) == 1
    assert fn(fake, fake, 1, 1, 32, 1000, 0.0, 0, None, 0, cp, P(4098), fake, fake, 1 << 20, None) == 1
    assert fn(fake, fake, 1, 1, 32, 1000, -1.0, 0, None, 0, cp, fake, fake, fake, 1 << 20, None) == 1
    # temperatures above 2^64 (and inf, NaN) are outside the range the statistics accept
    for t in (2.0 ** 65, float("inf"), float("nan")):
        assert fn(fake, fake, 1, 1, 32, 1000, t, 0, None, 0, cp, fake, fake, fake, 1 << 20, None) == 1
    # rule NONE with neither candidates nor a canvas is invalid (as for dllm_commit_step)
    assert fn(fake, fake, 1, 1, 32, 1000, 0.0, 0, None, 0, cp, fake, fake, fake, 1 << 20, None) == 1


def test_overflowing_shapes_are_rejected_on_the_host(lib):
    """Shapes whose row count, element count or byte count does not fit in
    int64 describe no buffer: the entry points return
    DLLM_ERR_INVALID_ARGUMENT (1) before any other arithmetic on them (a
    wrapped product could otherwise pass as an empty shape).  Nothing is
    launched, so no device is needed."""
    P, i64, i32, f32, u64, c_int = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                    ctypes.c_uint64, ctypes.c_int)
    fake = P(4096)                              # never dereferenced
    big = 1 << 40                               # big * big wraps to 0 in int64
    ts = lib.dllm_token_stats
    ts.argtypes = [P, c_int, i64, i64, i64, i64, f32, u64, P, i32, P, P, P, P, ctypes.c_size_t, P]
    ts.restype = c_int
    assert ts(fake, 1, big, big, 1000, 1000, 0.0, 0, None, 0, fake, fake, fake, fake, 1 << 20, None) == 1
    # rows fit, elements do not: 2^41 rows of stride 2^30
    assert ts(fake, 0, 1 << 31, 1 << 10, 1000, 1 << 30, 0.0, 0, None, 0, fake, fake, fake, fake, 1 << 20, None) == 1
    ws = lib.dllm_token_stats_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [i64, i64, i64, c_int]
    assert ws(big, big, 1000, 1) == 0
    assert ws(1 << 60, 0, 1000, 1) == 0
    assert ws(1, 32, 1000, 1) > 0
    edit = lib.dllm_edit_transfer
    edit.argtypes = [P, P, P, P, i64, i64, f32, P, P]
    edit.restype = c_int
    assert edit(fake, fake, fake, fake, big, big, 0.5, fake, None) == 1
    ren = lib.dllm_renoise
    ren.argtypes = [P, P, P, P, i64, i64, P, P]
    ren.restype = c_int
    assert ren(fake, None, None, None, big, big, fake, None) == 1
    uc = lib.dllm_uniform_canvas
    uc.argtypes = [i64, i64, i64, u64, P, i64, P]
    uc.restype = c_int
    assert uc(big, 10, 1000, 0, fake, big, None) == 1
    sched = lib.dllm_transfer_schedule
    sched.argtypes = [P, i64, i32, P, P]
    sched.restype = c_int
    assert sched(fake, 1 << 40, 1 << 30, fake, None) == 1
    mask = lib.dllm_block_causal_mask
    mask.argtypes = [i64, i64, i64, i64, i64, c_int, P, i64, P]
    mask.restype = c_int
    assert mask(big, big, 0, 0, 32, 0, fake, big, None) == 1
    host = lib.dllm_commit_step_host
    host.argtypes = [P, P, c_int, i64, i64, i64, f32, u64, P, i32, P, P, P, P, ctypes.c_size_t, P]
    host.restype = c_int
    params = (ctypes.c_char * 256)()
    assert host(fake, fake, 1, big, big, 1000, 0.0, 0, None, 0, ctypes.cast(params, P), fake, fake, fake,
                1 << 20, None) == 1
