"""The C-ABI library builds, loads and exports every symbol include/sp_api.h
declares; host-only entry points agree with the oracle.  No GPU needed (no
device call is made)."""
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from sequence_video_dit_gb300 import build

    build.build()
    import sequence_video_dit_gb300 as sp

    return sp


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^SP_API\s+[\w\s\*]+?\b(sp_\w+)\s*\(", src, flags=re.M))
    return names


def test_header_declares_the_step_entry_points():
    names = _declared_symbols()
    for n in ("sp_pad", "sp_partition", "sp_send_recv_heads", "sp_attention", "sp_gather_heads",
              "sp_gather_output", "sp_unpad"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    import ctypes

    from sequence_video_dit_gb300 import _lib

    lib = ctypes.CDLL(_lib.LIB_PATH)
    for name in sorted(_declared_symbols()):
        assert hasattr(lib, name), f"{name} not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


def test_library_exports_nothing_else(L):
    import subprocess

    from sequence_video_dit_gb300 import _lib

    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.split() and line.split()[-1].startswith("sp_")}
    assert exported == _declared_symbols()


def test_padded_len_and_partition(L):
    assert L.sp_padded_len(37, 2) == 38
    assert L.sp_padded_len(49155, 8) == 49160
    assert L.sp_padded_len(24576, 8) == 24576
    assert L.sp_partition(38, 2) == [(0, 19), (19, 19)]
    with pytest.raises(ValueError):
        L.sp_partition(37, 2)
    with pytest.raises(ValueError):
        L.sp_padded_len(-1, 2)
    for T, W in [(0, 1), (1, 8), (1001, 4), (6149, 8), (7, 3)]:
        assert L.sp_padded_len(T, W) == oracle.padded_len(T, W)
        assert L.sp_partition(L.sp_padded_len(T, W), W) == oracle.partition(oracle.padded_len(T, W), W)


@pytest.mark.parametrize("n,W", [(132, 8), (152, 8), (608, 8), (7, 8), (152, 3), (5, 1)])
def test_sm_rotation_counts_match_oracle(L, n, W):
    assert L.sp_sm_rotation_counts(n, W) == oracle.sm_rotation_counts(n, W)


def test_status_strings(L):
    from sequence_video_dit_gb300 import _lib

    lib = _lib.lib()
    assert lib.sp_status_string(0) == b"SP_OK"
    assert lib.sp_status_string(_lib.SP_ERR_NOT_DIVISIBLE) == b"SP_ERR_NOT_DIVISIBLE"
    assert lib.sp_status_string(_lib.SP_ERR_TIMEOUT) == b"SP_ERR_TIMEOUT"
    assert lib.sp_version() >= 1
    # the error message of the last failing call is kept per thread
    with pytest.raises(ValueError):
        L.sp_partition(5, 2)
    assert b"not divisible" in lib.sp_last_error()


@pytest.mark.parametrize("W", list(range(1, 33)))
def test_optimal_split_matches_oracle(L, W):
    assert L.sp_optimal_split(W) == oracle.optimal_split(W)


def test_optimal_split_rejects_zero(L):
    with pytest.raises(ValueError):
        L.sp_optimal_split(0)


def test_header_constants_match_the_binding():
    src = open(os.path.join(ROOT, "include", "sp_api.h")).read()
    from sequence_video_dit_gb300 import _lib

    for name in ("SP_WORKSPACE_HEADER_BYTES", "SP_WORKSPACE_KV_STALL_OFFSET"):
        m = re.search(rf"#define\s+{name}\s+(\d+)", src)
        assert m and int(m.group(1)) == getattr(_lib, name)


def test_missing_library_fails_loudly():
    # No CPU fallback: without the built CUDA library every entry point raises.
    import subprocess
    import sys

    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import sequence_video_dit_gb300._lib as L\n"
        "L.LIB_PATH = '/nonexistent/libsp_gb300.so'\n"
        "import sequence_video_dit_gb300 as sp\n"
        "try:\n"
        "    sp.sp_padded_len(37, 2)\n"
        "except ImportError as e:\n"
        "    print('raised:', e)\n"
        "    sys.exit(0)\n"
        "sys.exit(3)\n" % ROOT
    )
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "raised" in p.stdout
