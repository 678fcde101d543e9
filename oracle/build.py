"""Builds the fp64 oracle (plain C, gcc) into oracle/_lib/ -- test infrastructure."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "_lib", "libccq_oracle.so")


def build(force: bool = False) -> str:
    out = library_path()
    src = os.path.join(_HERE, "ccq_oracle.c")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps every multiply and add a separately rounded
    # fp64 operation, so results are identical on x86-64 and aarch64.
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-std=c11",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
