"""Build the CPU oracle (test infrastructure) into ``oracle/liboracle.so``.

Plain C99 compiled with gcc.  No fast-math and no FMA contraction, so that the
fp32 operations the formats fix (divisions by the scales, the fp32 products
of dequantisation) are single IEEE operations on every host.  OpenMP is used
for the row loops when the compiler supports it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ["codecs.c", "layout.c", "write.c", "score.c", "topk.c", "attention.c"]
LIB = os.path.join(HERE, "liboracle.so")


def _newer(target, deps):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force=False, verbose=False):
    deps = [os.path.join(HERE, s) for s in SOURCES] + [os.path.join(HERE, "bsp_oracle.h")]
    if not force and _newer(LIB, deps):
        return LIB
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            "-D_DEFAULT_SOURCE", "-Wall", "-Wno-unknown-pragmas"]
    srcs = [os.path.join(HERE, s) for s in SOURCES]
    tmp = LIB + ".tmp"
    for extra in (["-fopenmp"], []):
        cmd = base + extra + srcs + ["-o", tmp, "-lm"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            return LIB
        last = r.stderr
    raise RuntimeError("oracle build failed:\n" + last)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
