"""A batch that arrives in any request order: pka_batch_order orders it as
[decode : extend : prefill], pka_gather_rows moves the token and request rows
into that order and the outputs back, and the result matches the oracle of the
same requests. Also: the whole step replays from a CUDA graph bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_07_gb300 import pka
from paged_kv_attention_07_gb300 import workloads as W
from paged_kv_attention_07_gb300.device_batch import DeviceBatch, UnorderedBatch
from tests.gpu_util import LSE_ATOL, OUT_ATOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", [0, 1])
def test_shuffled_batch_through_order_and_gather(seed):
    # the workload builder makes an ordered batch; the user's batch is a shuffle of it
    spec = W.spec_custom("ordered", ctx=[3, 700, 77, 40, 1500, 0, 0], qlen=[1, 1, 1, 33, 70, 100, 7],
                         num_decodes=3, num_extends=2, num_prefills=2, Hq=16, Hkv=2, d=128, dv=128, bs=16,
                         chunk=512, seed=40 + seed)
    batch = W.make_batch(spec)
    db = DeviceBatch(batch)
    perm = np.random.default_rng(seed).permutation(spec.num_reqs)
    ub = UnorderedBatch(db, perm)
    assert ub.counts == [3, 2, 2]
    ub.step()
    torch.cuda.synchronize()
    assert ub.error_word() == 0
    ref_o, ref_l = oracle.batch_reference(batch)
    Hq, dv = spec.num_q_heads, spec.head_dim_v
    rows = (ub.tok_u[:, None] * Hq + np.arange(Hq)[None, :]).reshape(-1)
    eo = np.abs(ub.out_u.float().cpu().numpy().reshape(-1, dv) - ref_o[rows]).max()
    el = np.abs(ub.lse_u.cpu().numpy().reshape(-1) - ref_l[rows]).max()
    assert eo <= OUT_ATOL and el <= LSE_ATOL, (eo, el)


@pytest.mark.parametrize("width", [4, 1024])  # 16-byte rows and 4 KB rows, both through the flat (row, copy) loop
def test_gather_rows_bad_index_zero_fills_and_flags(width):
    src = torch.arange(10 * width, dtype=torch.float32, device="cuda").view(10, width)
    idx = torch.tensor([3, -1, 9, 10], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dst = torch.full((4, width), 7.0, device="cuda")
    pka.pka_gather_rows(dst, src, idx, error_word=err)
    torch.cuda.synchronize()
    assert torch.equal(dst[0], src[3]) and torch.equal(dst[2], src[9])
    assert torch.all(dst[1] == 0) and torch.all(dst[3] == 0)
    assert int(err.item()) == pka.DEVERR["INDEX"]


@pytest.mark.parametrize("row_bytes", [1, 6, 12, 16, 8192])
def test_gather_rows_widths(row_bytes):
    g = torch.Generator(device="cuda").manual_seed(row_bytes)
    src = torch.randint(0, 255, (33, row_bytes), dtype=torch.uint8, device="cuda", generator=g)
    idx = torch.randint(0, 33, (50,), dtype=torch.int32, device="cuda", generator=g)
    dst = torch.empty((50, row_bytes), dtype=torch.uint8, device="cuda")
    pka.pka_gather_rows(dst, src, idx)
    torch.cuda.synchronize()
    assert torch.equal(dst, src[idx.long()])


def _graph_of_step(db):
    """Capture db.step() (cache write + forward) in a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        db.step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        db.step()
    return graph


def test_step_replays_from_a_cuda_graph():
    spec = W.spec_custom("graph", ctx=[3, 700, 40, 1500, 0, 0], qlen=[1, 1, 33, 70, 100, 7], num_decodes=2,
                         num_extends=2, num_prefills=2, Hq=16, Hkv=2, d=128, dv=128, bs=16, chunk=512, seed=7)
    db = DeviceBatch(W.make_batch(spec))
    db.step()
    torch.cuda.synchronize()
    ref_out, ref_lse = db.out.clone(), db.lse.clone()
    graph = _graph_of_step(db)
    db.out.zero_()
    db.lse.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert db.error_word() == 0
    assert torch.equal(db.out, ref_out) and torch.equal(db.lse, ref_lse)


def test_graph_replays_new_metadata():
    """What a serving loop does with a captured step: each replay gets a new
    batch written into the same buffers (other lengths, block table, slots, Q
    and K/V; same request counts and token count, lengths within the host
    hints the graph was captured with). Every replay must match the oracle of
    the batch it was given."""
    common = dict(num_decodes=2, num_extends=2, num_prefills=2, Hq=16, Hkv=2, d=128, dv=128, bs=16, chunk=512)
    first = W.spec_custom("graph_a", ctx=[3, 700, 40, 1500, 0, 0], qlen=[1, 1, 33, 70, 100, 7], seed=8, **common)
    db = DeviceBatch(W.make_batch(first))
    graph = _graph_of_step(db)
    nb = db.k_cache.shape[0]
    later = [  # 212 new tokens each, like the captured batch
        W.spec_custom("graph_b", ctx=[650, 12, 1400, 90, 0, 0], qlen=[1, 1, 50, 53, 60, 47], seed=9,
                      num_blocks=nb, **common),
        W.spec_custom("graph_c", ctx=[1, 1, 1, 1, 0, 0], qlen=[1, 1, 2, 98, 99, 11], seed=10, num_blocks=nb,
                      **common),
    ]
    for spec in [first] + later:
        batch = W.make_batch(spec)
        if spec is not first:
            db.refill(batch)
        db.out.fill_(float("nan"))
        db.lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert db.error_word() == 0, spec.name
        assert db.canaries_intact(), spec.name
        ref_o, ref_l = oracle.batch_reference(batch)
        o = db.out.float().cpu().numpy().reshape(-1, spec.head_dim_v)
        l = db.lse.cpu().numpy().reshape(-1)
        assert np.isfinite(o).all() and np.isfinite(l).all(), spec.name
        eo, el = np.abs(o - ref_o).max(), np.abs(l - ref_l).max()
        assert eo <= OUT_ATOL and el <= LSE_ATOL, (spec.name, eo, el)


def test_packed_staging_buffers_give_the_same_step():
    """The inputs moved into one device arena and out / lse into one buffer
    (the layout the end-to-end benchmark copies with one transfer each way):
    the step from host-staged inputs matches the oracle and the unpacked step
    bit for bit, and nothing is written past the outputs."""
    spec = W.spec_custom("packed", ctx=[40, 300, 70, 0], qlen=[1, 1, 30, 50], num_decodes=2, num_extends=1,
                         num_prefills=1, Hq=8, Hkv=2, d=128, dv=128, bs=16, chunk=64, seed=77)
    batch = W.make_batch(spec)
    db = DeviceBatch(batch)
    db.step()
    out0, lse0 = db.out.clone(), db.lse.clone()
    arena, outs = db.pack_io()
    host_in = arena.cpu().pin_memory()
    arena.zero_()
    arena.copy_(host_in, non_blocking=True)
    db.step()
    host_out = outs.cpu()
    torch.cuda.synchronize()
    assert db.error_word() == 0 and db.canaries_intact()
    assert torch.equal(db.out, out0) and torch.equal(db.lse, lse0)
    T, Hq, dv = spec.num_tokens, spec.num_q_heads, spec.head_dim_v
    out = host_out[:T * Hq * dv * 2].view(torch.bfloat16).float().numpy().reshape(-1, dv)
    lse_off = (T * Hq * dv * 2 + 255) // 256 * 256
    lse = host_out[lse_off:lse_off + T * Hq * 4].view(torch.float32).numpy().reshape(-1)
    ref_o, ref_l = oracle.batch_reference(batch)
    assert np.abs(out - ref_o).max() <= OUT_ATOL and np.abs(lse - ref_l).max() <= LSE_ATOL


@pytest.mark.parametrize("kind", ["bf16", "fp8", "mla"])
def test_one_call_step_equals_two_calls(kind):
    """pka_paged_attn_step (cache write and forward in one call, the planner
    overlapping the write) gives the cache, out and lse of pka_cache_write
    followed by the forward call, bit for bit."""
    if kind == "mla":
        spec = W.spec_custom("step_mla", ctx=[100, 900, 64], qlen=[1, 1, 1], num_decodes=3, num_extends=0,
                             num_prefills=0, Hq=128, Hkv=1, d=576, dv=512, bs=64, scale=1 / np.sqrt(192),
                             mla=True, seed=81)
    else:
        spec = W.spec_custom("step_" + kind, ctx=[40, 300, 70, 0], qlen=[1, 1, 30, 50], num_decodes=2,
                             num_extends=1, num_prefills=1, Hq=8, Hkv=2, d=128, dv=128, bs=16, chunk=64, seed=82)
    batch = W.make_batch(spec)
    scales = (0.0125, 0.02) if kind == "fp8" else None
    a, b = DeviceBatch(batch, kv_scales=scales), DeviceBatch(batch, kv_scales=scales)
    a.step()
    b.step_separate()
    torch.cuda.synchronize()
    assert a.error_word() == 0 and b.error_word() == 0 and a.canaries_intact()
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t  # unwritten slots hold NaN
    assert torch.equal(bits(a.k_cache), bits(b.k_cache))
    if a.v_cache is not None:
        assert torch.equal(bits(a.v_cache), bits(b.v_cache))
    assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)


def test_one_call_step_reports_a_bad_slot():
    spec = W.spec_custom("step_bad", ctx=[40, 70], qlen=[1, 30], num_decodes=1, num_extends=1, num_prefills=0,
                         Hq=8, Hkv=2, d=128, dv=128, bs=16, chunk=64, seed=83)
    db = DeviceBatch(W.make_batch(spec))
    db.slot_mapping[3] = db.k_cache.shape[0] * spec.block_size + 5  # past the cache
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = spec
    pka.pka_paged_attn_step(db.q, db.k_new, db.v_new, db.slot_mapping, db.k_cache, db.v_cache, db.block_table,
                            db.qsl, db.seq_lens, *db.counts, s.scale, s.context_chunk, db.max_query_len,
                            db.max_seq_len, db.out, db.lse, db.workspace, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pka.DEVERR["SLOT"]
    assert db.canaries_intact()
