"""Build ``liboracle.so`` from ``dg_oracle.c`` with the host C compiler.

Part of the oracle (test infrastructure).  Plain C11 + pthreads, no
architecture-specific flags, so the same source builds on x86_64 and aarch64.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dg_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc, "-std=c11", "-O2", "-fPIC", "-shared", "-D_GNU_SOURCE", SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
