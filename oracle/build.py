"""Compile the plain-C oracle into oracle/liboracle.so (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg use
the result. Flags: no fast-math, and no implicit FMA contraction, so that every
rounding the oracle performs is the one written in oracle.c.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, src: str = SRC, out: str = LIB, defines=()) -> str:
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", *[f"-D{d}" for d in defines], src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
