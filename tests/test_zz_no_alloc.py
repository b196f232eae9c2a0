"""pka_paged_decode_noalloc: the split-KV decode for callers that cannot
give the library scratch memory (its scratch is a fixed device array inside
the library). Called through the C ABI, it must match the float64 oracle and
pka_paged_attn_forward on the same decode batch, on two calls in a row (the
second call reuses the array the first one left behind).

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


@pytest.mark.parametrize("d,bs", [(128, 16), (64, 4)])  # TMA tile loads; 16-byte copies below block size 8
def test_noalloc_decode_matches_forward_twice(d, bs):
    """Against the float64 oracle (the tolerance of every parity test) and,
    bit for bit, against pka_paged_attn_forward: both run the same kernels
    with the same split plan, so any difference is a scratch-layout slip."""
    import torch
    import oracle
    from paged_kv_attention_07_gb300 import pka
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    spec = W.spec_custom(f"noalloc_d{d}", ctx=np.random.default_rng(d).integers(0, 6000, 96).tolist(),
                         qlen=[1] * 96, num_decodes=96, num_extends=0, num_prefills=0, Hq=32, Hkv=4, d=d,
                         dv=d, bs=bs, seed=11 + d)
    batch = W.make_batch(spec)
    db = DeviceBatch(batch)
    db.step()  # existing entry point (caller workspace)
    assert db.error_word() == 0
    ref_o, ref_l = oracle.batch_reference(batch)
    lib = pka.load()
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(db.out, float("nan"))
        lse = torch.full_like(db.lse, float("nan"))
        st = _noalloc(lib, db, out, lse, err)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error word 0x{int(err.item()):x}"
        o = out.float().cpu().numpy().reshape(-1, d)
        l = lse.cpu().numpy().reshape(-1)
        assert np.isfinite(o).all() and np.isfinite(l).all()
        assert np.abs(o - ref_o).max() <= OUT_ATOL, f"call {call}"
        assert np.abs(l - ref_l).max() <= LSE_ATOL, f"call {call}"
        assert torch.equal(out.view(torch.int16), db.out.view(torch.int16)), f"call {call}"
        assert torch.equal(lse, db.lse), f"call {call}"


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
