"""Compile the CPU oracle (plain C) into shared libraries.

Test infrastructure: the oracle is built so that the tests, the smoke check
and the benchmark's CPU baseline can call it; the product path never does.

Two libraries:
  liboracle_fadam.so        the parity build: -O2 -ffp-contract=off, so that
                            every float operation is separately rounded (GCC
                            fuses multiply-adds by default on some targets,
                            Arm among them); the tests use only this one.
  liboracle_fadam_timed.so  the timed-only build of the same source plus an
                            OpenMP driver (oracle_omp.c): -O3 -fopenmp with
                            vectorisation, -ffp-contract=off kept and errno
                            left out of sqrtf so that the loop can vectorise;
                            no -march=native, so that it builds and computes
                            the same on every host.  Only the benchmark's CPU
                            baseline and reference arm time it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fadam_oracle.c")
OMP_SRC = os.path.join(HERE, "oracle_omp.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle_fadam.so")
TIMED_LIB = os.path.join(OUT_DIR, "liboracle_fadam_timed.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra"]
TIMED_CFLAGS = ["-O3", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                "-fno-math-errno", "-Wall", "-Wextra"]


def _compile(out: str, flags, sources, force: bool) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(out)
            and all(os.path.getmtime(out) >= os.path.getmtime(s) for s in sources)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *flags, *sources, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the parity library if it is missing or older than its source."""
    return _compile(LIB, CFLAGS, [SRC], force)


def build_timed(force: bool = False) -> str:
    """Build the timed-only OpenMP library (the CPU baseline's)."""
    return _compile(TIMED_LIB, TIMED_CFLAGS, [SRC, OMP_SRC], force)


if __name__ == "__main__":
    print(build(force=True))
    print(build_timed(force=True))
