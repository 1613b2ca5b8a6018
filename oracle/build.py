"""Compile the C oracle into ``oracle/libep_oracle.so`` with gcc.

Test infrastructure: building the checker is part of ``build()``, using it is
reserved to the tests, the smoke check and the CPU-baseline leg of the
benchmark.  Plain C99, no target-specific flags, so the same source builds on
x86_64 and aarch64 hosts.  Floating-point contraction is switched off so that
every sum is the plain binary32 addition the oracle writes down.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def oracle_library_path() -> str:
    return os.path.join(HERE, "libep_oracle.so")


def build_oracle(force: bool = False) -> str:
    src = os.path.join(HERE, "ep_oracle.c")
    out = oracle_library_path()
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(force=True))
