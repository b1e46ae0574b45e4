"""Build the CPU oracle (plain C, gcc) in place as ``liboracle.so``.

``build_oracle(src, out, defines)`` also serves the planted-mutant tests,
which compile an edited copy of ``oracle.c`` into a temporary directory.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build_oracle(src=SRC, out=LIB, include_dir=HERE):
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-Wall", "-Wextra", "-I", include_dir, "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


def build(force=False):
    srcs = [SRC, os.path.join(HERE, "oracle.h")]
    if force or not os.path.exists(LIB) or any(
            os.path.getmtime(s) > os.path.getmtime(LIB) for s in srcs):
        build_oracle()
    return LIB
