"""pka_paged_decode_noalloc: the split-KV decode for callers that cannot
give the library scratch memory (its scratch is a fixed device array inside
the library). Called through the C ABI, it must match pka_paged_attn_forward
on the same decode batch, on two calls in a row (the second call reuses the
array the first one left behind).

This file sorts last so that a run stopping at the first failure has already
run every other test."""
import ctypes

import numpy as np
import pytest

from paged_kv_attention_07_gb300 import workloads as W
from tests.gpu_util import LSE_ATOL, OUT_ATOL

pytestmark = pytest.mark.gpu


def _noalloc(lib, db, out, lse, err, nd=None):
    import torch
    s = db.spec
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.pka_paged_decode_noalloc(
        p(db.q), p(db.k_cache), p(db.v_cache), p(db.block_table), db.block_table.shape[1], p(db.qsl),
        p(db.seq_lens), s.num_decodes if nd is None else nd, s.num_q_heads, s.num_kv_heads, s.head_dim,
        db.k_cache.shape[0], s.block_size, float(s.scale), db.max_seq_len, p(out), p(lse), p(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_forward_twice():
    import torch
    from paged_kv_attention_07_gb300 import pka
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    spec = W.spec_decode_gqa(seed=11, num_reqs=96, lo=1, hi=6000)
    db = DeviceBatch(W.make_batch(spec))
    db.step()  # existing entry point (caller workspace)
    assert db.error_word() == 0
    ref_out = db.out.float().cpu().numpy()
    ref_lse = db.lse.cpu().numpy()
    lib = pka.load()
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(db.out, float("nan"))
        lse = torch.full_like(db.lse, float("nan"))
        st = _noalloc(lib, db, out, lse, err)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error word 0x{int(err.item()):x}"
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(l).all()
        assert np.abs(o - ref_out).max() <= OUT_ATOL
        assert np.abs(l - ref_lse).max() <= LSE_ATOL


def test_noalloc_rejects_batches_beyond_the_scratch():
    import torch
    from paged_kv_attention_07_gb300 import pka
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    spec = W.spec_decode_gqa(seed=12, num_reqs=8, lo=1, hi=100)
    db = DeviceBatch(W.make_batch(spec))
    lib = pka.load()
    out = torch.empty_like(db.out)
    # 4000 requests of 32 heads x 128 dims need more partial storage than the
    # fixed array holds: rejected on the host, nothing launched or read
    assert _noalloc(lib, db, out, None, None, nd=4000) == 3
