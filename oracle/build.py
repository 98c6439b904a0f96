"""Compile the CPU oracle (test infrastructure only) into oracle/_build/.

Plain gcc, no CUDA.  -ffp-contract=off keeps every binary32 multiply and add a
separately rounded IEEE operation (no fused multiply-add), which the quantizer's
bit-exact contract relies on; -fno-fast-math is the default and is restated.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle_nvfp4.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-fvisibility=hidden", "-o", tmp, SRC, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
