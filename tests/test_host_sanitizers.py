"""The library's host code (shared-prefix planner, block pool, cache-usage
accounting) built with AddressSanitizer and UndefinedBehaviorSanitizer and
run on random inputs by tests/sanitize/host_driver.cpp.  CPU only."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_311_gb300", "csrc")
HOST_SOURCES = ["pkv_plan.cu", "pkv_block_pool.cu", "pkv_usage.cu"]


def _cuda_root():
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_host_code_is_clean_under_asan_and_ubsan(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    cuda = _cuda_root()
    exe = tmp_path / "host_driver"
    cmd = [cxx, "-std=c++17", "-O1", "-g", "-fno-omit-frame-pointer",
           "-fsanitize=address,undefined", f"-I{cuda}/include"]
    for src in HOST_SOURCES:   # plain host C++ in .cu files
        cmd += ["-x", "c++", os.path.join(CSRC, src)]
    cmd += ["-x", "c++", os.path.join(ROOT, "tests", "sanitize", "host_driver.cpp"),
            "-o", str(exe), f"-L{cuda}/lib64", "-lcudart"]
    b = subprocess.run(cmd, capture_output=True, text=True)
    if b.returncode != 0 and "sanitize" in b.stderr and "cannot find" in b.stderr:
        pytest.skip("no sanitizer runtime for this compiler")
    assert b.returncode == 0, b.stderr[-3000:]
    env = dict(os.environ,
               LD_LIBRARY_PATH=f"{cuda}/lib64:" + os.environ.get("LD_LIBRARY_PATH", ""),
               # an allocation too large to serve fails as it would without ASan
               ASAN_OPTIONS="detect_leaks=1:protect_shadow_gap=0:allocator_may_return_null=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=600)
    report = r.stdout[-3000:] + r.stderr[-3000:]
    assert r.returncode == 0, report
    assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, report
    assert r.stdout.startswith("planned ")


def test_oracle_pins_are_clean_under_asan_and_ubsan(tmp_path):
    """The oracle's C source built with both sanitizers: its pin suite runs
    against it (the sanitizer runtimes preloaded into the interpreter)
    without a report."""
    import sys
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    rt = []
    for name in ("libasan.so", "libubsan.so"):
        p = subprocess.run([gcc, f"-print-file-name={name}"], capture_output=True,
                           text=True).stdout.strip()
        if not os.path.isabs(p):
            pytest.skip(f"no {name} for this compiler")
        rt.append(p)
    lib = tmp_path / "liboracle_san.so"
    b = subprocess.run([gcc, "-std=c11", "-O1", "-g", "-fno-omit-frame-pointer",
                        "-fsanitize=address,undefined", "-fPIC", "-shared",
                        "-D_POSIX_C_SOURCE=200809L", os.path.join(ROOT, "oracle", "pkv_oracle.c"),
                        "-o", str(lib), "-lm", "-lpthread"], capture_output=True, text=True)
    assert b.returncode == 0, b.stderr[-3000:]
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib), LD_PRELOAD=":".join(rt),
               ASAN_OPTIONS="detect_leaks=0:protect_shadow_gap=0",   # the interpreter's own
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    # -s: a sanitizer aborts the process, so its report must not sit in pytest's capture
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-s", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    report = r.stdout[-3000:] + r.stderr[-3000:]
    assert r.returncode == 0, report
    assert "runtime error" not in report and "AddressSanitizer" not in report, report


@pytest.mark.slow
def test_gpu_entry_points_host_checks_are_clean_under_ubsan(tmp_path):
    """The library built with UndefinedBehaviorSanitizer on its host code; the
    GPU entry points' argument checks get sizes at and past their limits
    (tests/sanitize/abi_extremes.py) with no CUDA device visible."""
    import sys
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a CUDA device is visible: this probe runs on machines without one")
    except ImportError:
        pass
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    ubsan = subprocess.run([gcc, "-print-file-name=libubsan.so"], capture_output=True,
                           text=True).stdout.strip()
    if not os.path.isabs(ubsan):
        pytest.skip("no libubsan for this compiler")
    from paged_kv_cache_311_gb300 import build as libbuild
    lib = libbuild.build(extra_flags=["-Xcompiler", "-fsanitize=undefined",
                                      "-Xcompiler", "-fno-sanitize-recover=undefined"],
                         out_path=str(tmp_path / "libpkv_ubsan.so"))
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", LD_PRELOAD=ubsan,
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "sanitize", "abi_extremes.py"), lib],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    report = r.stdout[-3000:] + r.stderr[-3000:]
    assert r.returncode == 0, report
    assert "runtime error" not in report and r.stdout.startswith("calls "), report
