"""Compile the C oracle with gcc into oracle/_build/libpkv_oracle.so.

Test infrastructure: building the checker is not using it.  The compile uses
-ffp-contract=off so that no multiply-add is fused behind the code's back (the
E4M3 encoding path relies on one plain fp32 multiply).
"""
import os
import platform
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpkv_oracle.so")


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    stamp = LIB + ".arch"
    if (not force and os.path.exists(LIB) and os.path.exists(stamp)
            and open(stamp).read() == platform.machine()
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(platform.machine())
    return LIB


if __name__ == "__main__":
    print(build(force=True))
