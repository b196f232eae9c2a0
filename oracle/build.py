"""Builds the oracle's shared library with the host C compiler (no CUDA).

Test infrastructure: see the package docstring of `oracle`.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pka_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_OUT = os.path.join(_OUT_DIR, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    """Compile pka_oracle.c into oracle/_build/liboracle.so if it is stale."""
    if (not force and os.path.exists(_OUT)
            and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC)):
        return _OUT
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = f"{_OUT}.{os.getpid()}.tmp"
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


if __name__ == "__main__":
    print(build_oracle(force=True))
