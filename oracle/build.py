"""Build the CPU oracle shared library (plain C, gcc, OpenMP over heads/queries).

Test infrastructure only: the oracle is compiled so the tests, the smoke check
and the benchmark's CPU-baseline leg can call it.  The product path never
loads it.
"""
import os
import platform
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vcattn_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libvcattn_oracle.so")
# A library compiled elsewhere from a modified copy of the source (the tests
# that plant mistakes in the oracle point the loader at it with this).
ENV_LIB = "VCATTN_ORACLE_LIB"


def compile_oracle(src: str, out: str) -> None:
    """gcc the oracle source `src` into the shared library `out`."""
    flags = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared"]
    if platform.machine() in ("x86_64", "AMD64"):
        # Lets fmaf() compile to the FMA instruction instead of a libm call;
        # results are the same either way (fmaf is correctly rounded).
        flags.append("-mfma")
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *flags, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile oracle/vcattn_oracle.c into oracle/_build/libvcattn_oracle.so."""
    if os.environ.get(ENV_LIB):
        return os.environ[ENV_LIB]
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    compile_oracle(SRC, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
