"""A C99 program (tests/c_abi_host.c) compiles against include/dllmcommit.h
with every warning an error, links against the in-tree library and calls its
host-side entry points; what it prints agrees with the oracle.  CPU only."""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    import importlib.util

    spec = importlib.util.spec_from_file_location("_b", os.path.join(ROOT, "commit_step_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    lib = os.path.abspath(b.build())
    exe = str(tmp_path_factory.mktemp("c_caller") / "c_abi_host")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_host.c"), lib, f"-Wl,-rpath,{os.path.dirname(lib)}",
           "-Wl,--allow-shlib-undefined", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    return [line.split() for line in out.stdout.splitlines()]


def _lines(program, tag):
    return [f[1:] for f in program if f[0] == tag]


def test_version_and_every_status_has_a_string(program):
    (version,) = _lines(program, "version")
    assert version and version[0]
    status = _lines(program, "status")
    assert [int(s[0]) for s in status] == [0, 1, 2, 3, 4, 5]
    assert all(len(s) > 1 and s[1] != "(null)" for s in status)


def test_block_ranges_from_c_match_the_oracle(program):
    got = _lines(program, "ranges")
    assert len(got) == 5
    for f in got:
        P, gen, bl, align, st, n = (int(x) for x in f[:6])
        want = oracle.block_ranges(P, gen, bl, bool(align))
        assert st == 0 and n == len(want)
        pairs = [int(x) for x in f[6:]]
        assert [tuple(pairs[i:i + 2]) for i in range(0, len(pairs), 2)] == [tuple(r) for r in want]


def test_linear_temperature_from_c_is_the_oracle_bit_for_bit(program):
    got = _lines(program, "temperature")
    assert len(got) == 3
    for remaining, num_steps, st, bits in got:
        assert int(st) == 0
        want = np.float32(oracle.linear_temperature(int(remaining), int(num_steps), 0.4, 0.8))
        assert struct.unpack("<I", want.tobytes())[0] == int(bits, 16)


def test_host_queries_and_argument_errors_from_c(program):
    (ws,) = _lines(program, "workspace")
    assert 0 < int(ws[4]) < (1 << 24)
    (mask,) = _lines(program, "mask_bad_block_len")
    assert int(mask[0]) == 1          # DLLM_ERR_INVALID_ARGUMENT, found before any device work
