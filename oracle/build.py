"""Build the fp64 CPU oracle (plain C, OpenMP) into a shared library.

The oracle is test infrastructure: building it is part of ``build()`` so the
checker exists on every machine, but nothing on the product path loads it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pkv_oracle.c")

# No fast-math and no FMA contraction: the oracle must round exactly as the
# C source reads, identically on x86-64 and aarch64.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
          "-fno-fast-math", "-ffp-contract=off", "-Wall"]


def library_path() -> str:
    return os.path.join(HERE, "libpkv_oracle.so")


def build_oracle(source: str = SOURCE, output: str | None = None,
                 extra_flags: list[str] | None = None) -> str:
    """Compile ``source`` with gcc; returns the path of the shared library."""
    out = output or library_path()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, *CFLAGS, *(extra_flags or []), source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(*sys.argv[1:2]))
