"""Compile the C oracle (test infrastructure only) with gcc.

The oracle is built in strict IEEE mode: no fast-math, no FMA contraction,
so that x86 and Arm hosts produce the same doubles.  Two builds of the one
source: ``liblora_oracle.so`` (single-threaded) and, where the compiler has
OpenMP, ``liblora_oracle_omp.so`` (the listed rows shared out among
threads; each row is still computed by one thread in the same order, so the
results are bit-identical).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lora_oracle.c")
LIB = os.path.join(HERE, "liblora_oracle.so")
LIB_OMP = os.path.join(HERE, "liblora_oracle_omp.so")
FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def _compile(out: str, extra) -> None:
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *FLAGS, *extra, SRC, "-o", tmp], check=True, capture_output=True)
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile liblora_oracle.so (and the OpenMP build) next to the source;
    return the single-threaded library's path."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        _compile(LIB, [])
    if force or not os.path.exists(LIB_OMP) or os.path.getmtime(LIB_OMP) < os.path.getmtime(SRC):
        try:
            _compile(LIB_OMP, ["-fopenmp"])
        except (subprocess.CalledProcessError, OSError):
            pass  # no OpenMP here: callers fall back to the single-threaded build
    return LIB


def omp_path():
    """Path of the OpenMP build, or None where it could not be built."""
    build()
    return LIB_OMP if os.path.exists(LIB_OMP) else None


if __name__ == "__main__":
    print(build(force=True))
    print(omp_path())
