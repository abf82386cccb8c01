"""Build the CPU oracle shared library (test infrastructure only).

    python oracle/build.py        # writes oracle/_build/liboracle.so

Plain gcc, -O2, OpenMP, no fast-math.  Portable C: builds the same on x86_64
and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gemm_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def build_variant(c_source: str, out_dir: str, name: str) -> str:
    """Compile a modified copy of the oracle source (tests use this to plant a
    mistake and check that the pins reject it).  Returns the library path."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, name + ".c")
    lib = os.path.join(out_dir, "lib" + name + ".so")
    with open(src, "w") as f:
        f.write(c_source)
    subprocess.run(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-w",
                    "-o", lib, src, "-lm"], check=True)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
