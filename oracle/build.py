"""Compile the CPU oracle (``fp8_oracle.c``) into a shared library.

Test infrastructure: the oracle is built next to its source, under
``oracle/_build/``, with flags that keep IEEE semantics (no FMA contraction,
no fast-math) so the same source gives the same bits on x86-64 and aarch64.
"""
import os
import platform
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
          "-Wall", "-Wextra", "-Wno-unused-parameter"]


def lib_path() -> str:
    return os.path.join(BUILD_DIR, f"liboracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    out = lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
