"""pka_batch_order (host-only): the [decode : extend : prefill] ordering of a
batch, checked against a direct stable partition and against the permutation
invariants of its token maps. No GPU."""
import ctypes

import numpy as np
import pytest

from paged_kv_attention_07_gb300 import build as B
from paged_kv_attention_07_gb300 import pka


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pka.load()


def reference_order(q, c):
    """Stable partition by class: one new token = decode, else cached context =
    extend, else prefill (the decode threshold is 1)."""
    cls = [0 if qi == 1 else (1 if ci > 0 else 2) for qi, ci in zip(q, c)]
    order = [r for k in range(3) for r in range(len(q)) if cls[r] == k]
    return np.array(order, np.int32), np.array([cls.count(k) for k in range(3)], np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_order_matches_a_stable_partition(lib, seed):
    rng = np.random.default_rng(seed)
    B_ = int(rng.integers(1, 40))
    q = np.where(rng.random(B_) < 0.5, 1, rng.integers(2, 50, B_)).astype(np.int32)
    c = np.where(rng.random(B_) < 0.4, 0, rng.integers(1, 5000, B_)).astype(np.int32)
    order, qsl, src, dst, counts = pka.pka_batch_order(q, c)
    ref_order, ref_counts = reference_order(q, c)
    assert np.array_equal(order, ref_order)
    assert np.array_equal(counts, ref_counts)
    assert np.array_equal(qsl, np.concatenate([[0], np.cumsum(q[order])]).astype(np.int32))
    T = int(q.sum())
    # token maps are inverse permutations, and token j of ordered request i is
    # token k of original request order[i]
    assert np.array_equal(np.sort(src), np.arange(T)) and np.array_equal(dst[src], np.arange(T))
    qsl_orig = np.concatenate([[0], np.cumsum(q)])
    for i, r in enumerate(order):
        assert np.array_equal(src[qsl[i]:qsl[i + 1]], np.arange(qsl_orig[r], qsl_orig[r + 1]))


def test_single_token_without_context_is_a_decode(lib):
    order, qsl, src, dst, counts = pka.pka_batch_order([5, 1, 3, 1], [0, 0, 7, 9])
    assert counts.tolist() == [2, 1, 1]
    assert order.tolist() == [1, 3, 2, 0]


def test_already_ordered_batch_is_the_identity(lib):
    q, c = [1, 1, 4, 9, 16], [30, 2, 5, 0, 0]
    order, qsl, src, dst, counts = pka.pka_batch_order(q, c)
    assert order.tolist() == list(range(5)) and counts.tolist() == [2, 1, 2]
    assert np.array_equal(src, np.arange(sum(q))) and np.array_equal(dst, np.arange(sum(q)))


@pytest.mark.parametrize("q,c", [([0, 2], [0, 0]), ([3, 2], [0, -1]), ([], [])])
def test_rejects_bad_batches(lib, q, c):
    n = len(q)
    qa = np.array(q + [0], np.int32)
    ca = np.array(c + [0], np.int32)
    out = np.zeros(64, np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = lib.pka_batch_order(n, p(qa), p(ca), p(out), p(out), None, None, p(out))
    assert st == 1  # PKA_ERR_INVALID_ARG


def test_gather_rows_rejects_bad_arguments(lib):
    buf = (ctypes.c_int32 * 4)()
    assert lib.pka_gather_rows(None, buf, buf, 1, 1, 4, None, None) == 1
    assert lib.pka_gather_rows(buf, buf, buf, -1, 1, 4, None, None) == 1
    assert lib.pka_gather_rows(buf, buf, buf, 1, 1, 0, None, None) == 1
    assert lib.pka_gather_rows(buf, buf, buf, 1 << 62, 1, 16, None, None) == 1  # byte size overflows
