"""The C-ABI library builds, loads and exports what include/pka.h declares, and
its host-side validation rejects bad arguments before touching the device.
Runs without a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

from paged_kv_attention_07_gb300 import build as B
from paged_kv_attention_07_gb300 import pka

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pka.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pka.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKA_API\s+[\w\s\*]+?\b(pka_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_symbols() == sorted(pka.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert pka.pka_status_string(0) == "ok"
    assert pka.pka_status_string(3) == "workspace too small"
    assert pka.pka_status_string(99) == "unknown status"


P = ctypes.c_void_p
FAKE = P(0x10000)  # never dereferenced: every case below fails validation first


def test_cache_write_rejects_bad_arguments(lib):
    st = lib.pka_cache_write(None, None, FAKE, 4, 2, 64, 64, FAKE, None, 8, 16, None, None)
    assert st == 1  # null k
    st = lib.pka_cache_write(FAKE, None, FAKE, -1, 2, 64, 64, FAKE, None, 8, 16, None, None)
    assert st == 1  # negative token count
    st = lib.pka_cache_write(FAKE, FAKE, FAKE, 4, 2, 64, 64, FAKE, None, 8, 16, None, None)
    assert st == 1  # v given without v_cache
    st = lib.pka_cache_write(FAKE, None, FAKE, 4, 2, 60, 64, FAKE, None, 8, 16, None, None)
    assert st == 2  # head_dim not a multiple of 8
    st = lib.pka_cache_write(P(0x10002), None, FAKE, 4, 2, 64, 64, FAKE, None, 8, 16, None, None)
    assert st == 1  # misaligned k
    assert lib.pka_cache_write(None, None, None, 0, 2, 64, 64, None, None, 8, 16, None, None) == 0


def _fwd(lib, **kw):
    a = dict(q=FAKE, k_new=FAKE, v_new=FAKE, k_cache=FAKE, v_cache=FAKE, bt=FAKE, maxb=8, qsl=FAKE,
             sl=FAKE, nd=2, ne=1, np=1, T=66, Hq=4, Hkv=2, d=64, dv=64, nb=64, bs=16, scale=0.125,
             chunk=32, maxq=48, maxs=101, out=FAKE, lse=None, ws=P(0x100000), wsb=1 << 20)
    a.update(kw)
    return lib.pka_paged_attn_forward(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["bt"],
                                      a["maxb"], a["qsl"], a["sl"], a["nd"], a["ne"], a["np"], a["T"],
                                      a["Hq"], a["Hkv"], a["d"], a["dv"], a["nb"], a["bs"], a["scale"],
                                      a["chunk"], a["maxq"], a["maxs"], a["out"], a["lse"], a["ws"],
                                      a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1),
    (dict(out=None), 1),
    (dict(ws=None), 1),
    (dict(k_new=None), 1),                 # prefill/extend need the new K/V
    (dict(d=96, dv=96), 2),                # head size without a kernel
    (dict(d=128, dv=64), 2),
    (dict(Hq=6, Hkv=4), 1),                # Hq not a multiple of Hkv
    (dict(Hq=64, Hkv=2), 2),               # group of 32 heads
    (dict(bs=24), 2),                      # block size not a power of two
    (dict(bs=256), 2),
    (dict(chunk=8), 1),
    (dict(maxs=10), 1),                    # max_seq_len < max_query_len
    (dict(T=3), 1),                        # fewer tokens than the batch needs
    (dict(maxb=2), 1),                     # table narrower than max_seq_len needs
    (dict(scale=float("inf")), 1),
    (dict(scale=0.0), 1),                  # the row max and the masking assume scale > 0
    (dict(scale=-0.125), 1),
    (dict(ws=P(0x100010)), 1),             # workspace not 256-byte aligned
    (dict(v_cache=None), 2),               # latent cache with d = 64
    (dict(v_cache=None, d=576, dv=512, Hq=128, Hkv=1), 2),  # latent cache: decode only
    (dict(nd=5000, ne=0, np=0, T=5000), 2),  # more requests than the planner holds
])
def test_forward_rejects_bad_arguments(lib, kw, status):
    assert _fwd(lib, **kw) == status


def test_merge_and_get_error_reject_bad_arguments(lib):
    assert lib.pka_merge_attn_states(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 64, 2, None) == 1
    assert lib.pka_merge_attn_states(FAKE, None, None, FAKE, FAKE, FAKE, 4, 64, 0, None) == 1
    assert lib.pka_merge_attn_states(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 6, 1, None) == 2
    assert lib.pka_merge_attn_states(None, None, None, None, None, None, 0, 64, 0, None) == 0
    assert lib.pka_get_error(None, None, None) == 1


def test_workspace_size_rejects_unsupported_shapes(lib):
    assert lib.pka_workspace_size(1, 0, 0, 1, 4, 2, 96, 96, 1, 10, 32) == 0
    assert lib.pka_workspace_size(1, 0, 0, 1, 6, 4, 64, 64, 1, 10, 32) == 0


@pytest.mark.parametrize("limit_us,with_code", [(0, True), (2000001, True), (1000, False)])
def test_selftest_wait_rejects_bad_arguments(lib, limit_us, with_code):
    code = ctypes.c_int32(0)
    st = lib.pka_selftest_wait(0, limit_us, ctypes.byref(code) if with_code else None, None)
    assert st == 1  # PKA_ERR_INVALID_ARG, before any CUDA call


def test_fp8_entry_points_reject_bad_arguments(lib):
    # cache write: bad scales, missing V, head_dim not a multiple of 8
    cw = lambda **kw: lib.pka_cache_write_fp8(
        kw.get("k", FAKE), kw.get("v", FAKE), FAKE, 4, 2, kw.get("d", 128), 128, FAKE, kw.get("vc", FAKE), 8, 16,
        ctypes.c_float(kw.get("ks", 0.5)), ctypes.c_float(kw.get("vs", 0.5)), None, None)
    assert cw(ks=0.0) == 1 and cw(vs=float("nan")) == 1 and cw(ks=-1.0) == 1
    assert cw(v=None) == 1 and cw(vc=None) == 1
    assert cw(d=60) == 2

    def fwd(**kw):
        a = dict(nd=2, ne=0, np=0, T=2, d=128, dv=128, ks=0.5, vs=0.5, vc=FAKE)
        a.update(kw)
        return lib.pka_paged_attn_forward_fp8(
            FAKE, FAKE, FAKE, FAKE, a["vc"], FAKE, 8, FAKE, FAKE, a["nd"], a["ne"], a["np"], a["T"], 8, 2, a["d"],
            a["dv"], 64, 16, ctypes.c_float(0.125), ctypes.c_float(a["ks"]), ctypes.c_float(a["vs"]), 32, 4, 100,
            FAKE, None, P(0x100000), 1 << 20, None)
    assert fwd(d=64, dv=64) == 2        # head dim 64
    assert fwd(ne=1, T=6, d=64, dv=64) == 2
    assert fwd(vc=None, d=576, dv=512) == 2  # a latent (MLA) cache has no 8-bit kernel
    # the 8-bit workspace query refuses what the 8-bit forward refuses, before any device query
    assert lib.pka_workspace_size_fp8(1, 1, 1, 8, 8, 2, 64, 64, 6, 100, 32) == 0
    assert lib.pka_workspace_size_fp8(1, 1, 1, 8, 8, 2, 192, 128, 6, 100, 32) == 0
    assert fwd(ks=0.0) == 1 and fwd(vs=float("inf")) == 1


def test_step_entry_points_reject_bad_arguments(lib):
    # no slot mapping: the step's cache write has nothing to write with
    for fn, extra in ((lib.pka_paged_attn_step, ()), (lib.pka_paged_attn_step_fp8,
                                                       (ctypes.c_float(0.5), ctypes.c_float(0.5)))):
        args = [FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 8, FAKE, FAKE, 2, 0, 0, 2, 8, 2, 128, 128, 64, 16,
                ctypes.c_float(0.125), *extra, 32, 1, 100, FAKE, None, None, P(0x100000), 1 << 20, None]
        assert fn(*args) == 1
