"""GPU parity: every path of the CUDA library against the float64 oracle, on
seeded inputs that span several tiles, ragged tails and the degenerate cases
(context 0, a single key, block size 1, one query head per kv head)."""
import numpy as np
import pytest

import oracle
from paged_kv_attention_07_gb300 import workloads as W
from tests.gpu_util import LSE_ATOL, OUT_ATOL, check_batch, compare, run_gpu

pytestmark = pytest.mark.gpu


def _dec(name, ctx, Hq, Hkv, d, bs, seed, mla=False, dv=None):
    return W.spec_custom(name, ctx=ctx, qlen=[1] * len(ctx), num_decodes=len(ctx), num_extends=0,
                         num_prefills=0, Hq=Hq, Hkv=Hkv, d=d, dv=dv or d, bs=bs, mla=mla, seed=seed,
                         scale=None if not mla else 1 / np.sqrt(192))


DEC_CTX = [0, 1, 15, 16, 17, 255, 256, 257, 600, 1500, 4100]


def test_tiny_mixed_config():
    check_batch(W.make_batch(W.spec_tiny()))


@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32, 64, 128])
def test_decode_gqa_block_sizes(bs):
    check_batch(W.make_batch(_dec(f"dec_bs{bs}", DEC_CTX, 32, 4, 128, bs, seed=bs)))


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (32, 4), (32, 2), (6, 3)])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_gqa_groups(Hq, Hkv, d):
    check_batch(W.make_batch(_dec(f"dec_g{Hq // Hkv}", DEC_CTX, Hq, Hkv, d, 16, seed=Hq + d)))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 8])
def test_prefill_varlen(d, G):
    lens = [1, 2, 63, 64, 65, 130, 300]
    spec = W.spec_custom("pre", ctx=[0] * len(lens), qlen=lens, num_decodes=0, num_extends=0,
                         num_prefills=len(lens), Hq=2 * G, Hkv=2, d=d, dv=d, bs=16, seed=d + G)
    check_batch(W.make_batch(spec))


@pytest.mark.parametrize("chunk", [16, 48, 1000])
@pytest.mark.parametrize("bs", [1, 16, 64])
def test_extend_chunks(chunk, bs):
    spec = W.spec_custom("ext", ctx=[1, 5, 100, 300], qlen=[2, 17, 64, 129], num_decodes=0,
                         num_extends=4, num_prefills=0, Hq=8, Hkv=2, d=128, dv=128, bs=bs, chunk=chunk,
                         seed=chunk + bs)
    check_batch(W.make_batch(spec))


@pytest.mark.parametrize("d", [64, 128])
def test_mixed_three_paths(d):
    spec = W.spec_custom("mixed_small", ctx=[3, 700, 40, 2000, 0, 0], qlen=[1, 1, 33, 70, 100, 7],
                         num_decodes=2, num_extends=2, num_prefills=2, Hq=16, Hkv=2, d=d, dv=d, bs=16,
                         chunk=512, seed=d)
    check_batch(W.make_batch(spec))


@pytest.mark.parametrize("Hq", [16, 32, 64, 128])
@pytest.mark.parametrize("bs", [1, 4, 16, 64])
def test_decode_mla(Hq, bs):
    ctx = [0, 1, 17, 200, 1500, 3000] if Hq == 128 else [0, 17, 1500]
    spec = _dec("mla", ctx, Hq, 1, 576, bs, seed=Hq + bs, mla=True, dv=512)
    check_batch(W.make_batch(spec))


def test_decode_mla_two_head_groups():
    """256 heads: two groups of 128 heads per split on the tensor-core kernel."""
    spec = _dec("mla_256", [0, 63, 64, 65, 1100], 256, 1, 576, 16, seed=256, mla=True, dv=512)
    check_batch(W.make_batch(spec))


def _amplify_keys(batch, r, lo, hi, factor, dims=slice(None)):
    """Scale dims `dims` of keys [lo, hi) of request r (bf16 round trip) so that,
    for some rows and not others, the running max jumps by more than 2^8
    mid-sequence: the lazy O rescale then runs for part of a warp's rows only."""
    rows = batch.seq_start[r] + np.arange(lo, hi)
    f = W.bf16_bits_to_f32(batch.k_seq[rows])
    f[..., dims] *= np.float32(factor)
    batch.k_seq[rows] = W.to_bf16_bits(f)


def test_decode_mla_rescale_some_heads():
    # split 1 of request 0 (keys 1024..2047) meets a band at 1500 whose last 64
    # latent dims (scores only; the value is dims 0..511, left as drawn, so
    # |O| stays O(1)) are amplified: 43 of 128 heads, in all four warps, must
    # rescale O
    spec = W.spec_custom("mla_rs", ctx=[2999, 1999], qlen=[1, 1], num_decodes=2, num_extends=0,
                         num_prefills=0, Hq=128, Hkv=1, d=576, dv=512, bs=64, scale=1 / np.sqrt(192),
                         mla=True, seed=5)
    batch = W.make_batch(spec)
    _amplify_keys(batch, 0, 1500, 1564, 7.0, dims=slice(512, 576))
    check_batch(batch)


def test_prefill_rescale_some_rows():
    # keys 600..639 amplified: about a third of the rows that see them, in
    # every warp, must rescale O mid-sequence
    spec = W.spec_custom("fa_rs", ctx=[0], qlen=[1000], num_decodes=0, num_extends=0, num_prefills=1,
                         Hq=16, Hkv=2, d=128, dv=128, bs=16, seed=6)
    batch = W.make_batch(spec)
    _amplify_keys(batch, 0, 600, 640, 3.5)
    check_batch(batch)


def test_decode_mla_many_units():
    """More (request, split, half) units than SMs, several splits per request."""
    rng = np.random.default_rng(17)
    ctx = rng.integers(1, 2500, 192).tolist()
    spec = _dec("mla_many", ctx, 128, 1, 576, 64, seed=17, mla=True, dv=512)
    check_batch(W.make_batch(spec))


def _repeat_bitwise(batch, steps, kv_scales=None):
    """Run the same step `steps` times; every output must equal the first bit
    for bit. Work units are taken dynamically, so the CTA that runs a unit,
    and what ran on that CTA before it, changes from step to step: a race
    between a unit and its predecessor on the same CTA shows up here even
    when it stays inside the tolerance of a single comparison. The bf16 cases
    also check the first output against the oracle (the 8-bit paths have
    their own oracle tests)."""
    import torch
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    db = DeviceBatch(batch, kv_scales=kv_scales)
    db.step()
    torch.cuda.synchronize()
    first_o, first_l = db.out.clone(), db.lse.clone()
    for _ in range(steps):
        db.step()
        torch.cuda.synchronize()
        assert torch.equal(db.out, first_o) and torch.equal(db.lse, first_l), "a repeated step changed the output"
    assert db.error_word() == 0
    if kv_scales is None:
        out = first_o.float().cpu().numpy().reshape(-1, batch.spec.head_dim_v)
        compare(batch, out, first_l.cpu().numpy().reshape(-1))


@pytest.mark.parametrize("bs", [64, 4])
def test_decode_mla_repeated_steps_bitwise(bs):
    # consecutive units of one CTA alternate value halves, whose latent
    # chunks split into score-only and value parts differently; block size
    # 4 loads every tile by row gathers
    rng = np.random.default_rng(17)
    ctx = rng.integers(1, 2500, 192).tolist()
    _repeat_bitwise(W.make_batch(_dec("mla_rep", ctx, 128, 1, 576, bs, seed=17, mla=True, dv=512)), 24)


@pytest.mark.parametrize("kind", ["gqa", "mixed", "gqa_fp8", "mixed_fp8"])
def test_repeated_steps_bitwise(kind):
    rng = np.random.default_rng(23)
    if kind.startswith("gqa"):
        ctx = rng.integers(1, 5000, 256).tolist()
        batch = W.make_batch(_dec("gqa_rep", ctx, 32, 8, 128, 16, seed=23))
    else:
        spec = W.spec_custom("mixed_rep", ctx=[900, 3000, 40, 2000, 0, 0], qlen=[1, 1, 300, 77, 500, 129],
                             num_decodes=2, num_extends=2, num_prefills=2, Hq=16, Hkv=2, d=128, dv=128, bs=16,
                             chunk=1024, seed=23)
        batch = W.make_batch(spec)
    _repeat_bitwise(batch, 12, kv_scales=(0.0125, 0.02) if kind.endswith("fp8") else None)


def test_constant_v_gives_constant_output():
    spec = W.spec_custom("const", ctx=[0, 90, 30, 0], qlen=[1, 1, 20, 50], num_decodes=2,
                         num_extends=1, num_prefills=1, Hq=8, Hkv=2, d=128, dv=128, bs=16, chunk=32)
    batch = W.make_batch(spec)
    batch.v_seq[:] = W.to_bf16_bits(np.array([0.375], np.float32))[0]
    out, lse, err, _ = run_gpu(batch)
    assert err == 0
    assert np.all(out == 0.375)


def test_cache_write_bit_exact():
    import torch
    from paged_kv_attention_07_gb300 import pka
    from paged_kv_attention_07_gb300.device_batch import bf16_tensor
    spec = W.spec_custom("cw", ctx=[37, 100, 64, 0], qlen=[1, 1, 16, 48], num_decodes=2, num_extends=1,
                         num_prefills=1, Hq=4, Hkv=2, d=64, dv=64, bs=16, num_blocks=64, seed=9)
    batch = W.make_batch(spec)
    kc_ref, vc_ref = oracle.populate_cache(batch, "context")
    slots = batch.slot_mapping.copy()
    slots[5] = -1  # padding token
    oracle.cache_write(batch.k_new, batch.v_new, slots, kc_ref, vc_ref, spec.block_size)
    kc = bf16_tensor(oracle.populate_cache(batch, "context")[0], "cuda")
    vc = bf16_tensor(oracle.populate_cache(batch, "context")[1], "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pka.pka_cache_write(bf16_tensor(batch.k_new, "cuda"), bf16_tensor(batch.v_new, "cuda"),
                        torch.from_numpy(slots).cuda(), kc, vc, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(kc.view(torch.int16).cpu().numpy().view(np.uint16), kc_ref)
    assert np.array_equal(vc.view(torch.int16).cpu().numpy().view(np.uint16), vc_ref)


def test_cache_write_latent_and_bad_slot():
    import torch
    from paged_kv_attention_07_gb300 import pka
    from paged_kv_attention_07_gb300.device_batch import bf16_tensor
    spec = _dec("cwl", [5, 70], 16, 1, 576, 4, seed=3, mla=True, dv=512)
    batch = W.make_batch(spec)
    kc_ref, _ = oracle.populate_cache(batch, "context")
    slots = batch.slot_mapping.copy()
    oracle.cache_write(batch.k_new, None, slots, kc_ref, None, spec.block_size)
    kc = bf16_tensor(oracle.populate_cache(batch, "context")[0], "cuda")
    bad = slots.copy()
    bad[0] = kc_ref.shape[0] * spec.block_size + 3  # beyond the cache: skipped + flagged
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pka.pka_cache_write(bf16_tensor(batch.k_new, "cuda"), None, torch.from_numpy(bad).cuda(), kc, None,
                        error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pka.DEVERR["SLOT"]
    got = kc.view(torch.int16).cpu().numpy().view(np.uint16)
    # the good token landed, the bad one was dropped
    blk, off = divmod(int(slots[1]), spec.block_size)
    assert np.array_equal(got[blk, 0, off], kc_ref[blk, 0, off])
    blk0, off0 = divmod(int(slots[0]), spec.block_size)
    assert np.all(got[blk0, 0, off0] == 0x7FC0)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_merge_attn_states(io):
    import torch
    from paged_kv_attention_07_gb300 import pka
    rng = np.random.default_rng(1)
    n, dv = 777, 128
    a = rng.standard_normal((n, dv)).astype(np.float32)
    b = rng.standard_normal((n, dv)).astype(np.float32)
    la = (rng.standard_normal(n) * 3).astype(np.float32)
    lb = (rng.standard_normal(n) * 3).astype(np.float32)
    la[:5] = -np.inf  # empty prefix
    lb[5:10] = -np.inf  # empty suffix
    la[10:12] = lb[10:12] = -np.inf  # both empty
    if io == "bf16":
        a = W.bf16_bits_to_f32(W.to_bf16_bits(a))
        b = W.bf16_bits_to_f32(W.to_bf16_bits(b))
    ref_o, ref_l = oracle.merge_attn_states(a, la, b, lb)
    dt = torch.float32 if io == "f32" else torch.bfloat16
    ta, tb = torch.from_numpy(a).cuda().to(dt), torch.from_numpy(b).cuda().to(dt)
    out = torch.empty_like(ta)
    out_lse = torch.empty(n, dtype=torch.float32, device="cuda")
    pka.pka_merge_attn_states(out, out_lse, ta, torch.from_numpy(la).cuda(), tb, torch.from_numpy(lb).cuda())
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    l = out_lse.cpu().numpy()
    tol = 1e-5 if io == "f32" else OUT_ATOL
    np.testing.assert_allclose(o, ref_o, atol=tol, rtol=0)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin)
    np.testing.assert_allclose(l[fin], ref_l[fin], atol=1e-5, rtol=0)


def test_repeat_is_bitwise_deterministic():
    import torch
    spec = W.spec_custom("det", ctx=[3, 700, 40, 2000, 0], qlen=[1, 1, 33, 70, 100], num_decodes=2,
                         num_extends=2, num_prefills=1, Hq=16, Hkv=2, d=128, dv=128, bs=16, chunk=512,
                         seed=4)
    out, lse, err, db = run_gpu(W.make_batch(spec))
    first = db.out.clone()
    db.forward()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), db.out.view(torch.int16))


# ---------------------------------------------------------------- error paths
def _with_metadata(batch, **changes):
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    db = DeviceBatch(batch)
    for k, v in changes.items():
        getattr(db, k).copy_(v)
    return db


def test_device_error_order():
    """A prefill placed in the decode slice: ORDER bit, nothing computed."""
    import torch
    from paged_kv_attention_07_gb300 import pka
    spec = W.spec_custom("ord", ctx=[10, 0], qlen=[1, 5], num_decodes=1, num_extends=0, num_prefills=1,
                         Hq=4, Hkv=2, d=64, dv=64, bs=16)
    db = _with_metadata(W.make_batch(spec))
    db.spec = W.spec_custom("ord", ctx=[10, 0], qlen=[1, 5], num_decodes=2, num_extends=0,
                            num_prefills=0, Hq=4, Hkv=2, d=64, dv=64, bs=16)
    db.counts = (2, 0, 0)
    db.workspace = torch.zeros(db.workspace.numel() + (4 << 20), dtype=torch.uint8, device="cuda")
    db.out.fill_(7.0)
    db.forward()
    err = db.error_word()
    assert err & pka.DEVERR["ORDER"]
    assert torch.all(db.out == 7.0)  # no work was done


def test_device_error_bad_block_id():
    """A block id past the cache is flagged and never dereferenced."""
    import torch
    from paged_kv_attention_07_gb300 import pka
    spec = W.spec_custom("blk", ctx=[40, 33], qlen=[1, 9], num_decodes=1, num_extends=1,
                         num_prefills=0, Hq=4, Hkv=2, d=128, dv=128, bs=16, chunk=16)
    batch = W.make_batch(spec)
    db = _with_metadata(batch)
    bt = db.block_table.clone()
    bt[0, 1] = batch.num_blocks + 5
    bt[1, 0] = -3
    db.block_table.copy_(bt)
    db.forward()
    err = db.error_word()
    assert err & pka.DEVERR["BLOCK_ID"]
    assert err & ~(pka.DEVERR["BLOCK_ID"]) == 0


def test_device_error_seq_len_hint():
    """seq_len above the max_seq_len hint: SEQ_LEN bit, plan left empty."""
    from paged_kv_attention_07_gb300 import pka
    spec = W.spec_custom("sl", ctx=[40, 100], qlen=[1, 1], num_decodes=2, num_extends=0,
                         num_prefills=0, Hq=4, Hkv=2, d=64, dv=64, bs=16)
    db = _with_metadata(W.make_batch(spec))
    db.max_seq_len = 50
    db.forward()
    assert db.error_word() & pka.DEVERR["SEQ_LEN"]


def test_workspace_too_small_is_rejected():
    import torch
    from paged_kv_attention_07_gb300 import pka
    spec = W.spec_tiny()
    db = _with_metadata(W.make_batch(spec))
    small = db.workspace[:1024]
    with pytest.raises(pka.PkaError) as ei:
        s = db.spec
        pka.pka_paged_attn_forward(db.q, db.k_new, db.v_new, db.k_cache, db.v_cache, db.block_table,
                                   db.qsl, db.seq_lens, s.num_decodes, s.num_extends, s.num_prefills,
                                   s.scale, s.context_chunk, db.max_query_len, db.max_seq_len, db.out,
                                   db.lse, small)
    assert ei.value.status == 3


def test_output_only_16_byte_aligned():
    """out 16- but not 32-byte aligned: the prefill/extend epilogue falls back
    from 32-byte to 16-byte stores, with the same results."""
    import torch
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    spec = W.spec_custom("al16", ctx=[40, 0, 0], qlen=[33, 70, 200], num_decodes=0, num_extends=1,
                         num_prefills=2, Hq=8, Hkv=2, d=128, dv=128, bs=16, chunk=32, seed=16)
    batch = W.make_batch(spec)
    db = DeviceBatch(batch)
    db.cache_write()
    T, Hq, dv = spec.num_tokens, spec.num_q_heads, spec.head_dim_v
    buf = torch.zeros(T * Hq * dv + 8, dtype=torch.bfloat16, device=db.device)
    out = buf[8:].view(T, Hq, dv)
    assert out.data_ptr() % 32 == 16
    db.forward(out=out)
    torch.cuda.synchronize()
    assert db.error_word() == 0
    compare(batch, out.float().cpu().numpy().reshape(-1, dv), db.lse.cpu().numpy().reshape(-1))


@pytest.mark.parametrize("bs", [1, 16])
def test_decodes_routed_through_the_extend_path(bs):
    """The single-path routing: decodes placed in the extend slice (num_decodes
    0) run through the prefill/extend kernel and its chunk merge, same results."""
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    spec = W.spec_custom("unified", ctx=[3, 700, 1, 40, 2000, 0, 0], qlen=[1, 1, 1, 33, 70, 100, 7],
                         num_decodes=3, num_extends=2, num_prefills=2, Hq=16, Hkv=2, d=128, dv=128, bs=bs,
                         chunk=512, seed=11 + bs)
    batch = W.make_batch(spec)
    db = DeviceBatch(batch, unified=True)
    assert db.counts == (0, 5, 2)
    db.step()
    import torch
    torch.cuda.synchronize()
    assert db.error_word() == 0
    compare(batch, db.out.float().cpu().numpy().reshape(-1, spec.head_dim_v), db.lse.cpu().numpy().reshape(-1))


def test_unified_routing_mostly_one_token_requests():
    """Single-path routing of a decode-heavy batch: 64 one-token requests and
    one 4-token extend all in the extend slice, so the extend slice holds
    fewer than two new tokens per request."""
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    rng = np.random.default_rng(21)
    ctx = rng.integers(1, 3000, 64).tolist()
    spec = W.spec_custom("unified_dec", ctx=ctx + [500], qlen=[1] * 64 + [4], num_decodes=64, num_extends=1,
                         num_prefills=0, Hq=32, Hkv=4, d=128, dv=128, bs=16, chunk=1024, seed=21)
    batch = W.make_batch(spec)
    db = DeviceBatch(batch, unified=True)
    assert db.counts == (0, 65, 0)
    db.step()
    import torch
    torch.cuda.synchronize()
    assert db.error_word() == 0
    assert db.canaries_intact()
    compare(batch, db.out.float().cpu().numpy().reshape(-1, spec.head_dim_v), db.lse.cpu().numpy().reshape(-1))


# ---------------------------------------------------------------- MLA non-absorbed prefill / extend
# The pages' non-absorbed recipe for MLA prefill and extend runs ordinary
# attention over the decompressed K (192 dims: 128 + 64 rope) and V (128).

@pytest.mark.parametrize("G", [1, 4])
def test_nonabsorbed_prefill(G):
    lens = [1, 2, 63, 64, 65, 130, 300]
    spec = W.spec_custom("na_pre", ctx=[0] * len(lens), qlen=lens, num_decodes=0, num_extends=0,
                         num_prefills=len(lens), Hq=2 * G, Hkv=2, d=192, dv=128, bs=16, seed=300 + G)
    check_batch(W.make_batch(spec))


@pytest.mark.parametrize("chunk", [16, 48, 1000])
@pytest.mark.parametrize("bs", [1, 16, 64])
def test_nonabsorbed_extend_chunks(chunk, bs):
    spec = W.spec_custom("na_ext", ctx=[1, 5, 100, 300], qlen=[2, 17, 64, 129], num_decodes=0, num_extends=4,
                         num_prefills=0, Hq=4, Hkv=4, d=192, dv=128, bs=bs, chunk=chunk, seed=310 + chunk + bs)
    check_batch(W.make_batch(spec))


def test_nonabsorbed_mixed():
    """Extends (one-token ones included: decodes routed through the extend
    path) and prefills in one batch."""
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    spec = W.spec_custom("na_mixed", ctx=[700, 3, 40, 2000, 0, 0], qlen=[1, 1, 33, 300, 100, 7], num_decodes=2,
                         num_extends=2, num_prefills=2, Hq=8, Hkv=8, d=192, dv=128, bs=16, chunk=512, seed=320)
    batch = W.make_batch(spec)
    db = DeviceBatch(batch, unified=True)
    db.step()
    import torch
    torch.cuda.synchronize()
    assert db.error_word() == 0 and db.canaries_intact()
    compare(batch, db.out.float().cpu().numpy().reshape(-1, 128), db.lse.cpu().numpy().reshape(-1))


def test_nonabsorbed_rejects_the_decode_slice():
    from paged_kv_attention_07_gb300 import pka
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    spec = W.spec_custom("na_dec", ctx=[70, 0], qlen=[1, 5], num_decodes=1, num_extends=0, num_prefills=1,
                         Hq=4, Hkv=4, d=192, dv=128, bs=16, seed=3)
    with pytest.raises(RuntimeError):  # the workspace query rejects the shape (no split-KV kernel at d 192)
        DeviceBatch(W.make_batch(spec))
    assert pka.pka_workspace_size(1, 0, 1, 6, 4, 4, 192, 128, 5, 71, 32) == 0
