"""Builds the oracle's C library (test infrastructure only).

Plain gcc, portable C11 (no intrinsics, no -march), so it gives the same
results on x86_64 and aarch64 hosts."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")


def library_path() -> str:
    return os.path.join(HERE, "_lib", "libpkv_oracle.so")


def build_oracle(extra_flags=(), out_path: str | None = None) -> str:
    out = out_path or library_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"   # parallel test workers may build at once
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-D_POSIX_C_SOURCE=200809L", *extra_flags, SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle())
