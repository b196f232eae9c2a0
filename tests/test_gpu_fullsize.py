"""Parity at the full workload sizes, in the launch configuration the
benchmark times: every row where the oracle can afford it (decode configs),
otherwise every decode row plus a seeded sample of >= 4096 (token, head) rows
that includes the first and last token of every request."""
import numpy as np
import pytest

from paged_kv_attention_07_gb300 import workloads as W
from tests.gpu_util import compare, run_gpu, sample_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _run(spec, rows_fn=None):
    batch = W.make_batch(spec)
    out, lse, err, db = run_gpu(batch)
    assert err == 0, f"device error word 0x{err:x}"
    del db
    rows = rows_fn(batch) if rows_fn else None
    return compare(batch, out, lse, rows=rows)


def test_decode_gqa_full():
    _run(W.spec_decode_gqa())


def test_prefill_varlen_full():
    _run(W.spec_prefill(), lambda b: sample_rows(b, 4096, seed=2))


def test_mixed_full():
    _run(W.spec_mixed(), lambda b: sample_rows(b, 4096, seed=3))


def test_mla_decode_full_bs64():
    _run(W.spec_mla_decode())


def test_mla_decode_full_bs1():
    spec = W.spec_mla_decode(block_size=1)
    # all requests, a quarter of the heads of each (oracle time)
    def rows(b):
        Hq = spec.num_q_heads
        return np.array([t * Hq + h for t in range(spec.num_tokens) for h in range(0, Hq, 4)], np.int64)
    _run(spec, rows)
