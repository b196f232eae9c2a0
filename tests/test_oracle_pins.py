"""Pins for the float64 oracle, against things other than itself.

* a library routine: torch's scaled_dot_product_attention (float64, CPU,
  explicit bottom-right causal mask, GQA by repeating KV heads) on the dense
  per-request K/V, i.e. without the block table;
* closed forms: constant V, a single key, q = 0, two keys;
* invariants the pages rely on: chunked context + LSE merge equals unchunked
  attention ("Beyond porting", extend path: chunks combined by an LSE merge),
  split-KV + merge equals no split, block-size and block-permutation
  invariance, GQA equals MHA with repeated KV heads;
* the cache write as an exact round trip that leaves other slots untouched.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_07_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _f64(bits):
    return torch.from_numpy(W.bf16_bits_to_f32(bits).astype(np.float64))


def sdpa_reference(batch):
    """Dense per-request attention with torch SDPA (float64)."""
    spec = batch.spec
    G = spec.num_q_heads // spec.num_kv_heads
    outs = []
    for r in range(spec.num_reqs):
        s0, s1 = int(batch.seq_start[r]), int(batch.seq_start[r + 1])
        t0, t1 = int(batch.query_start_loc[r]), int(batch.query_start_loc[r + 1])
        ctx = spec.ctx[r]
        q = _f64(batch.q[t0:t1]).permute(1, 0, 2)  # [Hq, qlen, d]
        k = _f64(batch.k_seq[s0:s1]).permute(1, 0, 2)  # [Hkv, S, d]
        if batch.v_seq is None:
            v = k[..., : spec.head_dim_v]
        else:
            v = _f64(batch.v_seq[s0:s1]).permute(1, 0, 2)
        k = k.repeat_interleave(G, dim=0)
        v = v.repeat_interleave(G, dim=0)
        i = torch.arange(t1 - t0)[:, None]
        j = torch.arange(s1 - s0)[None, :]
        mask = j <= ctx + i  # bottom-right aligned causal mask
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                             scale=spec.scale)
        outs.append(o.permute(1, 0, 2).reshape(-1, spec.head_dim_v))
    return torch.cat(outs).numpy()


def _full_cache_attention(batch, **kw):
    spec = batch.spec
    kc, vc = oracle.populate_cache(batch, "all")
    return oracle.attention(batch.q, kc, vc, batch.block_table, batch.query_start_loc,
                            batch.seq_lens, spec.scale, spec.block_size,
                            head_dim_v=spec.head_dim_v, **kw)


SMALL_SPECS = [
    W.spec_tiny(),
    W.spec_custom("gqa8_bs1", ctx=[0, 5, 30, 0], qlen=[1, 1, 9, 13], num_decodes=2, num_extends=1,
                  num_prefills=1, Hq=16, Hkv=2, d=32, dv=32, bs=1, seed=5),
    W.spec_custom("mha_bs64", ctx=[70, 3], qlen=[1, 40], num_decodes=1, num_extends=1,
                  num_prefills=0, Hq=3, Hkv=3, d=16, dv=16, bs=64, seed=6),
    W.spec_custom("mla_like", ctx=[17, 40], qlen=[1, 1], num_decodes=2, num_extends=0,
                  num_prefills=0, Hq=8, Hkv=1, d=48, dv=32, bs=4, mla=True, seed=7),
    # separate K and V caches with d != dv: the shape of the non-absorbed MLA
    # prefill/extend (192 / 128) scaled down (next row f2)
    W.spec_custom("mha_d24_dv16", ctx=[9, 33, 0], qlen=[1, 12, 5], num_decodes=1, num_extends=1,
                  num_prefills=1, Hq=4, Hkv=2, d=24, dv=16, bs=8, seed=8),
]


@pytest.mark.parametrize("spec", SMALL_SPECS, ids=lambda s: s.name)
def test_oracle_matches_sdpa(spec):
    batch = W.make_batch(spec)
    out, _ = oracle.batch_reference(batch)
    ref = sdpa_reference(batch)
    assert out.shape == ref.shape
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_decode_sees_its_own_key():
    """A decode query at position ctx attends to ctx + 1 keys (its own included):
    with q = 0 every visible key has the same score, so lse = ln(ctx + 1)."""
    spec = W.spec_custom("dec", ctx=[0, 1, 37, 100], qlen=[1, 1, 1, 1], num_decodes=4,
                         num_extends=0, num_prefills=0, Hq=2, Hkv=1, d=8, dv=8, bs=16, seed=1)
    batch = W.make_batch(spec)
    batch.q[:] = 0
    out, lse = oracle.batch_reference(batch)
    for r, c in enumerate(spec.ctx):
        s0, s1 = int(batch.seq_start[r]), int(batch.seq_start[r + 1])
        mean_v = W.bf16_bits_to_f32(batch.v_seq[s0:s1, 0]).astype(np.float64).mean(axis=0)
        for h in range(2):
            assert lse[r * 2 + h] == pytest.approx(math.log(c + 1), abs=1e-13)
            np.testing.assert_allclose(out[r * 2 + h], mean_v, atol=1e-13)


def test_constant_v_returns_constant():
    spec = W.spec_tiny()
    batch = W.make_batch(spec)
    batch.v_seq[:] = W.to_bf16_bits(np.array([0.375], np.float32))[0]
    out, _ = oracle.batch_reference(batch)
    np.testing.assert_allclose(out, 0.375, rtol=1e-15, atol=0)


def test_single_key_closed_form():
    """One visible key: o = v0 and lse = scale * q . k0."""
    spec = W.spec_custom("one", ctx=[0, 0], qlen=[1, 1], num_decodes=0, num_extends=0,
                         num_prefills=2, Hq=4, Hkv=2, d=16, dv=16, bs=16, scale=0.3, seed=3)
    batch = W.make_batch(spec)
    out, lse = oracle.batch_reference(batch)
    for r in range(2):
        for h in range(4):
            q = W.bf16_bits_to_f32(batch.q[r, h]).astype(np.float64)
            k0 = W.bf16_bits_to_f32(batch.k_seq[r, h // 2]).astype(np.float64)
            v0 = W.bf16_bits_to_f32(batch.v_seq[r, h // 2]).astype(np.float64)
            assert lse[r * 4 + h] == pytest.approx(0.3 * float(q @ k0), abs=1e-12)
            np.testing.assert_allclose(out[r * 4 + h], v0, atol=1e-15)


def test_two_key_closed_form():
    """Two keys: o = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1, lse = log(e^s0 + e^s1)."""
    spec = W.spec_custom("two", ctx=[1], qlen=[1], num_decodes=1, num_extends=0, num_prefills=0,
                         Hq=1, Hkv=1, d=2, dv=2, bs=16, scale=1.0, seed=3)
    batch = W.make_batch(spec)
    bf = lambda a: W.to_bf16_bits(np.asarray(a, np.float32))
    batch.q[0, 0] = bf([1.0, 0.0])
    batch.k_seq[0, 0] = bf([1.0, 0.0])  # s0 = 1
    batch.k_seq[1, 0] = bf([0.0, 1.0])  # s1 = 0
    batch.v_seq[0, 0] = bf([1.0, 2.0])
    batch.v_seq[1, 0] = bf([3.0, 4.0])
    out, lse = oracle.batch_reference(batch)
    p0 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(out[0], [p0 * 1 + (1 - p0) * 3, p0 * 2 + (1 - p0) * 4], atol=1e-15)
    assert lse[0] == pytest.approx(math.log(math.e + 1.0), abs=1e-15)


@pytest.mark.parametrize("chunk", [1, 7, 32, 10 ** 6])
def test_chunked_context_merge_equals_plain(chunk):
    spec = W.spec_custom("ext", ctx=[37, 100, 64, 5, 0], qlen=[1, 1, 16, 9, 48], num_decodes=2,
                         num_extends=2, num_prefills=1, Hq=4, Hkv=2, d=32, dv=32, bs=16, seed=11)
    batch = W.make_batch(spec)
    kc, vc = oracle.populate_cache(batch, "all")
    args = (batch.q, kc, vc, batch.block_table, batch.query_start_loc, batch.seq_lens, spec.scale,
            spec.block_size)
    plain_out, plain_lse = oracle.attention(*args)
    out, lse = oracle.extend_forward(*args, chunk=chunk)
    np.testing.assert_allclose(out, plain_out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, plain_lse, atol=1e-12, rtol=0)


@pytest.mark.parametrize("split", [1, 5, 16, 1000])
def test_split_kv_merge_equals_plain(split):
    batch = W.make_batch(W.spec_tiny())
    spec = batch.spec
    kc, vc = oracle.populate_cache(batch, "all")
    args = (batch.q, kc, vc, batch.block_table, batch.query_start_loc, batch.seq_lens, spec.scale,
            spec.block_size)
    plain_out, plain_lse = oracle.attention(*args)
    out, lse = oracle.split_kv_forward(*args, split=split)
    np.testing.assert_allclose(out, plain_out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, plain_lse, atol=1e-12, rtol=0)


def _with_block_size(spec, bs, seed_perm=None):
    s = W.spec_custom(spec.name, spec.ctx, spec.qlen, spec.num_decodes, spec.num_extends,
                      spec.num_prefills, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                      spec.head_dim_v, bs, scale=spec.scale, mla=spec.mla, seed=spec.seed)
    return s


def test_block_size_and_permutation_invariance():
    base = W.spec_tiny()
    results = []
    for bs in (1, 16, 64):
        spec = _with_block_size(base, bs)
        rng = np.random.default_rng(123)
        batch = W.make_batch(spec, rng=rng)
        results.append(_full_cache_attention(batch))
    # same values, other block order
    spec = _with_block_size(base, 16)
    b1 = W.make_batch(spec, rng=np.random.default_rng(123))
    nb = b1.num_blocks
    perm = np.random.default_rng(999).permutation(nb).astype(np.int32)
    b2 = W.make_batch(spec, rng=np.random.default_rng(123), block_perm=perm)
    assert not np.array_equal(b1.block_table, b2.block_table)
    results.append(_full_cache_attention(b2))
    for o, l in results[1:]:
        np.testing.assert_array_equal(o, results[0][0])
        np.testing.assert_array_equal(l, results[0][1])


def test_gqa_equals_mha_with_repeated_kv_heads():
    spec = W.spec_custom("gqa", ctx=[20, 0], qlen=[1, 12], num_decodes=1, num_extends=0,
                         num_prefills=1, Hq=6, Hkv=2, d=16, dv=16, bs=8, seed=21)
    b = W.make_batch(spec, rng=np.random.default_rng(5))
    out_gqa, lse_gqa = _full_cache_attention(b)
    spec_mha = W.spec_custom("mha", spec.ctx, spec.qlen, 1, 0, 1, Hq=6, Hkv=6, d=16, dv=16, bs=8,
                             seed=21)
    b2 = W.make_batch(spec_mha, rng=np.random.default_rng(5))
    b2.q[:] = b.q
    b2.k_seq = np.repeat(b.k_seq, 3, axis=1)
    b2.v_seq = np.repeat(b.v_seq, 3, axis=1)
    b2.block_table[:] = b.block_table
    b2.slot_all[:] = b.slot_all
    out_mha, lse_mha = _full_cache_attention(b2)
    np.testing.assert_array_equal(out_gqa, out_mha)
    np.testing.assert_array_equal(lse_gqa, lse_mha)


def test_merge_closed_forms():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((5, 8))
    l = rng.standard_normal(5)
    # merging a result with itself keeps o and adds ln 2
    mo, ml = oracle.merge_attn_states(o, l, o, l)
    np.testing.assert_allclose(mo, o, atol=1e-15)
    np.testing.assert_allclose(ml, l + math.log(2.0), atol=1e-15)
    # an empty side (lse = -inf) contributes nothing, from either side
    empty_o, empty_l = np.zeros_like(o), np.full_like(l, -np.inf)
    for args in ((o, l, empty_o, empty_l), (empty_o, empty_l, o, l)):
        mo, ml = oracle.merge_attn_states(*args)
        np.testing.assert_array_equal(mo, o)
        np.testing.assert_array_equal(ml, l)
    mo, ml = oracle.merge_attn_states(empty_o, empty_l, empty_o, empty_l)
    assert np.all(mo == 0) and np.all(ml == -np.inf)
    # two single-key results merge to the two-key closed form
    v0, v1 = np.array([[1.0, 2.0]]), np.array([[3.0, 4.0]])
    mo, ml = oracle.merge_attn_states(v0, np.array([1.0]), v1, np.array([0.0]))
    p0 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(mo[0], p0 * v0[0] + (1 - p0) * v1[0], atol=1e-15)
    assert ml[0] == pytest.approx(math.log(math.e + 1.0), abs=1e-15)


def test_cache_write_round_trip_and_untouched_slots():
    spec = W.spec_tiny()
    batch = W.make_batch(spec)
    kc, vc = oracle.populate_cache(batch, "context")
    before_k, before_v = kc.copy(), vc.copy()
    slots = batch.slot_mapping.copy()
    slots[3] = -1  # a padding token: must not be written
    oracle.cache_write(batch.k_new, batch.v_new, slots, kc, vc, spec.block_size)
    bs = spec.block_size
    written = np.zeros(kc.shape[0] * bs, dtype=bool)
    for i, s in enumerate(batch.slot_all):
        blk, off = divmod(int(s), bs)
        is_new = i in set(batch.new_index.tolist())
        if is_new and slots[list(batch.new_index).index(i)] < 0:
            np.testing.assert_array_equal(kc[blk, :, off], before_k[blk, :, off])
            continue
        written[s] = True
        np.testing.assert_array_equal(kc[blk, :, off], batch.k_seq[i])
        np.testing.assert_array_equal(vc[blk, :, off], batch.v_seq[i])
    # every slot the batch does not own still holds the NaN poison
    kflat = kc.transpose(0, 2, 1, 3).reshape(-1, spec.num_kv_heads * spec.head_dim)
    assert np.all(kflat[~written] == 0x7FC0)
    assert np.array_equal(before_k.transpose(0, 2, 1, 3).reshape(kflat.shape)[~written], kflat[~written])


def test_golden_tiny_rows():
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_mixed_oracle.json")
    with open(path) as f:
        g = json.load(f)
    batch = W.make_batch(W.spec_tiny(g["seed"]))
    rows = np.array(g["rows"], dtype=np.int64)
    out, lse = oracle.batch_reference(batch, rows=rows)
    np.testing.assert_allclose(out[:, : len(g["out"][0])], np.array(g["out"]), atol=1e-12)
    np.testing.assert_allclose(lse, np.array(g["lse"]), atol=1e-12)
