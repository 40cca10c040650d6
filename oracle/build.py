"""Compile the C oracle into oracle/libpa_oracle.so with the host gcc.

Test infrastructure only: the library this builds is loaded by the test
suite, the smoke check and the benchmark's CPU-baseline leg, never by the
product path.  Flags keep IEEE semantics: no fast-math and no contraction of
a*b+c into a fused multiply-add, so float division in the fp8 quantiser is
the correctly rounded IEEE operation on every host (x86-64 and aarch64).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
LIB = os.path.join(HERE, "libpa_oracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-std=c99", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
