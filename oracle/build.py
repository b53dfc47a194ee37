"""Compile the CPU oracle into oracle/libls_oracle.so with the host C compiler.

Test infrastructure: the product library never links or loads this file's
output.  Portable C11 (no target-specific flags), so it builds the same way on
x86_64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ls_oracle.c")
LIB = os.path.join(HERE, "libls_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Build the shared object if it is missing or older than its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
