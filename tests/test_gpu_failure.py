"""Failure detection on the GPU without a fault: every pipeline wait of the
kernels is bounded, gives up with PKA_DEVERR_TIMEOUT in the device error word
and lets the kernel exit, so the context stays usable. pka_selftest_wait runs
that same wait on its own against an mbarrier nothing arrives on."""
import time

import pytest

from paged_kv_attention_07_gb300 import pka
from paged_kv_attention_07_gb300 import workloads as W
from tests.gpu_util import check_batch

pytestmark = pytest.mark.gpu

TIMEOUT = pka.DEVERR["TIMEOUT"]


def test_wait_returns_when_the_phase_completes():
    assert pka.pka_selftest_wait(True, 1000) == 0


def test_wait_runs_out_and_reports_timeout():
    t0 = time.perf_counter()
    code = pka.pka_selftest_wait(False, 20000)  # 20 ms limit
    dt = time.perf_counter() - t0
    assert code == TIMEOUT
    assert 0.015 < dt < 1.5, dt


def test_context_usable_after_a_timeout():
    assert pka.pka_selftest_wait(False, 5000) == TIMEOUT
    # a full forward pass afterwards still matches the oracle
    check_batch(W.make_batch(W.spec_tiny()))
    assert pka.pka_selftest_wait(True, 1000) == 0
