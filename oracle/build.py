"""Build the CPU oracle shared library (test infrastructure only).

Compiles ``memra_oracle.cpp`` with plain IEEE fp32 semantics: no fast-math and no
floating-point contraction, so every multiply and add is rounded on its own.
OpenMP is used when the compiler supports it (it only splits independent output
rows across threads).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "memra_oracle.cpp")
LIB = os.path.join(HERE, "libmemra_oracle.so")

BASE_FLAGS = ["-O2", "-std=c++17", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]


def _openmp_ok(cxx):
    probe = subprocess.run([cxx, "-fopenmp", "-x", "c++", "-", "-o", os.devnull],
                           input=b"int main(){return 0;}", capture_output=True)
    return probe.returncode == 0


def build(force=False, verbose=False):
    """Compile the oracle if the source is newer than the library; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cxx = os.environ.get("CXX", "g++")
    flags = list(BASE_FLAGS)
    if _openmp_ok(cxx):
        flags.append("-fopenmp")
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [cxx] + flags + [SRC, "-o", tmp]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
