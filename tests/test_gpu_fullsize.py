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


def test_mla_prefill_extend_full():
    """The non-absorbed MLA prefill/extend workload exactly as the benchmark
    runs it (128 heads, values drawn on the device from the same seeded
    generator): two heads' K, V and q come back to the host, and the oracle
    checks their rows for a seeded sample of >= 4096 (token, head) rows plus
    the first and last token of every request."""
    import torch
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    spec = W.spec_mla_prefill()
    batch = W.make_batch(spec, values=False)
    db = DeviceBatch(batch, values_on_device_seed=1234)
    db.step()
    torch.cuda.synchronize()
    assert db.error_word() == 0 and db.canaries_intact()
    heads = [0, 77]
    T = spec.num_tokens
    # the same batch restricted to two heads (heads are independent: MHA)
    sub = W.spec_custom("mla_prefill_2h", ctx=spec.ctx, qlen=spec.qlen, num_decodes=0,
                        num_extends=spec.num_extends, num_prefills=spec.num_prefills, Hq=2, Hkv=2, d=192, dv=128,
                        bs=spec.block_size, scale=spec.scale, chunk=spec.context_chunk)
    to_bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    q = to_bits(db.q[:, heads])
    kc = to_bits(db.k_cache[:, heads])
    vc = to_bits(db.v_cache[:, heads])
    out = db.out[:, heads].float().cpu().numpy().reshape(-1, 128)
    lse = db.lse[:, heads].cpu().numpy().reshape(-1)
    del db
    torch.cuda.empty_cache()
    import oracle
    qsl = batch.query_start_loc
    toks = set(np.random.default_rng(5).choice(T, 2048, replace=False).tolist())
    for r in range(spec.num_reqs):
        toks.update((int(qsl[r]), int(qsl[r + 1]) - 1))
    rows = np.array(sorted(t * 2 + h for t in toks for h in range(2)), np.int64)
    ref_o, ref_l = oracle.attention(q, kc, vc, batch.block_table, batch.query_start_loc, batch.seq_lens,
                                    sub.scale, sub.block_size, head_dim_v=128, rows=rows)
    assert np.isfinite(out[rows]).all() and np.isfinite(lse[rows]).all()
    eo = np.abs(out[rows] - ref_o).max()
    el = np.abs(lse[rows] - ref_l).max()
    assert rows.size >= 4096 and eo <= 2e-2 and el <= 1e-3, (rows.size, eo, el)
