"""The C-ABI library without a GPU: it loads, exports every function that
include/pkv.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import subprocess

import pytest

import paged_kv_cache_311_gb300 as pkv
from paged_kv_cache_311_gb300.build import build, library_path


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(library_path()):
        build()
    return pkv.load_library()


def test_header_declares_the_boundary():
    names = pkv.declared_functions()
    for n in ["pkv_paged_attention_decode", "pkv_reshape_and_cache", "pkv_copy_blocks",
              "pkv_paged_attention_workspace_bytes", "pkv_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in pkv.declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    assert pkv.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5):
        assert pkv.status_string(code) != "unknown status"
    assert pkv.status_string(99) == "unknown status"


def test_workspace_bytes(lib):
    # single pass: no workspace
    assert pkv.paged_attention_workspace_bytes(64, 32, 512, 128, 0) == 0
    # split path at 512-token partitions: (max, sum) pairs then fp32 accumulators
    B, H, L, D = 16, 64, 32768, 128
    np_ = L // 512
    ml = B * H * np_ * 2 * 4
    expect = ((ml + 255) // 256) * 256 + B * H * np_ * D * 4
    assert pkv.paged_attention_workspace_bytes(B, H, L, D, 0) == expect
    assert pkv.paged_attention_workspace_bytes(B, H, L, D, 512) == expect
    assert pkv.paged_attention_workspace_bytes(0, H, L, D, 0) == 0
    # sizes whose byte count passes 64 bits report 0 (the decode call then
    # refuses them) instead of a wrapped-around size
    assert pkv.paged_attention_workspace_bytes(65535, 65535, 1 << 30, 128, 32) == 0


def _decode(lib, **kw):
    a = dict(out=1 << 20, out_dtype=0, q=1 << 20, k=1 << 20, v=1 << 20, kv_dtype=1, bt=1 << 20, mb=8,
             cl=1 << 20, B=2, H=4, Hk=2, D=128, bs=16, NB=64, maxL=100, scale=0.1, P=0, ws=None,
             wsb=0, st=None, stream=None)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.pkv_paged_attention_decode(
        vp(a["out"]), a["out_dtype"], vp(a["q"]), vp(a["k"]), vp(a["v"]), a["kv_dtype"], vp(a["bt"]),
        a["mb"], vp(a["cl"]), a["B"], a["H"], a["Hk"], a["D"], a["bs"], a["NB"], a["maxL"],
        ctypes.c_float(a["scale"]), a["P"], a["ws"], a["wsb"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(H=5, Hk=2), -1),              # heads not a multiple of kv heads
    (dict(kv_dtype=7), -1),             # unknown dtype
    (dict(maxL=8 * 16 + 1), -1),        # longer than the table can cover
    (dict(out=0), -1),                  # null pointer
    (dict(k=(1 << 20) + 8), -1),        # cache not 16-byte aligned
    (dict(P=48), None),                 # partition not a multiple of 32 (checked after device query)
    (dict(D=96), -2),                   # head_dim outside {64, 128}
    (dict(bs=24), -2),                  # block size outside {8, 16, 32}
    (dict(H=6, Hk=2), -2),              # group of 3
])
def test_decode_host_validation(lib, kw, code):
    rc = _decode(lib, **kw)
    if code is None:
        assert rc in (-1, -3)            # -3 only because this host has no GPU
    else:
        assert rc == code


def test_zero_sequences_is_ok(lib):
    assert _decode(lib, B=0, out=0, q=0, k=0, v=0, bt=0, cl=0) == 0


def test_cache_ops_host_validation(lib):
    vp = ctypes.c_void_p
    A = vp(1 << 20)
    # head_dim * element size not a multiple of 16 bytes
    assert lib.pkv_reshape_and_cache(A, A, A, A, 1, A, 4, 2, 4, 16, 8, None, None) == -1
    assert lib.pkv_reshape_and_cache(A, A, A, A, 1, A, 0, 2, 64, 16, 8, None, None) == 0
    arr = (ctypes.c_void_p * 1)(1 << 20)
    assert lib.pkv_copy_blocks(arr, arr, 1, A, 3, 100, 8, None, None) == -1   # block bytes % 16
    assert lib.pkv_copy_blocks(arr, arr, 1, A, 0, 128, 8, None, None) == 0
    bad = (ctypes.c_void_p * 1)(0)
    assert lib.pkv_copy_blocks(bad, arr, 1, A, 3, 128, 8, None, None) == -1


def test_package_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        pkv.load_library(str(tmp_path / "missing.so"))


def test_bounded_wait_hook_checks_its_arguments_on_the_host(lib):
    """The test hook rejects a missing status word and a limit outside
    (0, 2 s] before any CUDA call."""
    lib.pkv_test_bounded_wait.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p,
                                          ctypes.c_void_p]
    assert lib.pkv_test_bounded_wait(1_000_000, 0, None, None) == -1
    fake = ctypes.c_void_p(1 << 20)
    assert lib.pkv_test_bounded_wait(0, 0, fake, None) == -1
    assert lib.pkv_test_bounded_wait(2_000_000_001, 0, fake, None) == -1
