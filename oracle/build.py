"""Build the CPU oracle shared library (test infrastructure only).

Compiles ``kvq_oracle.c`` with gcc into ``oracle/_build/libkvq_oracle.so``.
``-ffp-contract=off`` keeps every multiply and add separately rounded, so the
fp32 codec path follows its documented expression order on x86-64 and on
aarch64 alike.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvq_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkvq_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
