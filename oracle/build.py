"""Build step of the CPU oracle (test infrastructure): one gcc call, no optimisation tricks.

`-ffp-contract=off` keeps the binary64 additions of the multi-word combine as
separate IEEE operations (no fused multiply-add contraction).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liborc.so")


def build_oracle(force: bool = False) -> str:
    src = os.path.join(HERE, "orc.c")
    newest = max(os.path.getmtime(src), os.path.getmtime(os.path.join(HERE, "orc.h")))
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                           "-Wall", "-o", tmp, src, "-lm"])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_oracle(force=True))
