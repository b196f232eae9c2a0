"""Paged-KV attention forward for GB300 (sm_103a).

The compute path lives in the CUDA library `libpka.so` (sources under
`csrc/`, C ABI in `include/pka.h`); `pka` is its ctypes binding and
`workloads` builds seeded synthetic batches. Importing the package does not
load the CUDA library; the first call through `pka` does, and fails loudly if
it is missing.
"""
__all__ = ["pka", "workloads"]
