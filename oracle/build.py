"""Compile the C oracle (test infrastructure only) with gcc.

The oracle is built in strict IEEE mode: no fast-math, no FMA contraction,
so that x86 and Arm hosts produce the same doubles.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lora_oracle.c")
LIB = os.path.join(HERE, "liblora_oracle.so")


def build(force: bool = False) -> str:
    """Compile liblora_oracle.so next to its source; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
