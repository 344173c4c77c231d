"""Build step for the oracle's C library (test infrastructure only).

Compiles ``linattn_oracle.c`` with gcc into ``liboracle.so`` beside it (or,
for a planted-mistake variant, into a caller-given directory).  Plain C11,
OpenMP when the compiler has it, no architecture-specific flags, so the same
source builds on x86_64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "linattn_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")


def _compile(out_path: str, defines: tuple[str, ...] = ()) -> None:
    base = ["gcc", "-std=c11", "-O2", "-shared", "-fPIC", "-Wall"]
    base += [f"-D{d}" for d in defines]
    cmd = base + ["-fopenmp", "-o", out_path, SOURCE, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # a compiler without OpenMP still builds the (single-threaded) oracle
        subprocess.run(base + ["-o", out_path, SOURCE, "-lm"], check=True,
                       capture_output=True, text=True)


def build(force: bool = False) -> str:
    """Compile liboracle.so if it is missing or older than its source."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    try:
        _compile(tmp)
        os.replace(tmp, LIBRARY)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return LIBRARY


def build_mutant(mutant: int, out_dir: str) -> str:
    """Compile the oracle with planted mistake number ``mutant`` into out_dir."""
    out = os.path.join(out_dir, f"liboracle_mutant{mutant}.so")
    _compile(out, (f"ORACLE_MUTANT={mutant}",))
    return out


if __name__ == "__main__":
    print(build(force=True))
