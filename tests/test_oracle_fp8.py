"""Pins of the oracle's FP8 E4M3 codec (CPU): the decoded value of every code
against torch's float8_e4m3fn conversion (a library routine), the format's
printed constants, round-to-nearest-even against torch on random values, the
exact round trip of every finite code, saturation and the sign of zero."""
import numpy as np
import pytest
import torch

from oracle import fp8


def test_every_code_decodes_like_torch():
    ours = fp8.decode(np.arange(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))


def test_format_constants():
    v = fp8.decode([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0x80, 0xB8, 0xFE])
    assert v.tolist() == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 448.0, -0.0, -1.0, -448.0]
    assert np.isnan(fp8.decode([0x7F, 0xFF])).all()
    assert np.isnan(fp8.decode(np.arange(256))).sum() == 2


def test_finite_codes_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(fp8.encode(fp8.decode(codes)), codes)


@pytest.mark.parametrize("seed", range(3))
def test_rounding_matches_torch_in_range(seed):
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.normal(0, s, 4000) for s in (1e-3, 1e-1, 1.0, 30.0)]).astype(np.float32)
    x = x[np.abs(x) <= fp8.MAX_FINITE]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(x), ref)


def test_ties_go_to_the_even_code():
    # exact midpoints: between 1.0 (0x38) and 1.125 (0x39); between the two
    # smallest subnormals; between 0 and the smallest subnormal
    assert fp8.encode([1.0625, 3 * 2.0 ** -10, 2.0 ** -10, 1.1875]).tolist() == [0x38, 0x02, 0x00, 0x3A]


def test_saturation_nan_and_signed_zero():
    assert fp8.encode([500.0, -1e9, 448.0, 464.0]).tolist() == [0x7E, 0xFE, 0x7E, 0x7E]
    assert fp8.encode([np.nan]).tolist() == [0x7F]
    assert fp8.encode([0.0, -0.0]).tolist() == [0x00, 0x80]


def test_scaled_round_trip_error_bound():
    # relative error of a normal-range value is at most half an ulp: 2^-4
    rng = np.random.default_rng(7)
    x = rng.normal(0, 1, 10000)
    scale = 0.05
    y = fp8.dequantize(fp8.quantize(x, scale), scale)
    normal = np.abs(x / scale) >= 2.0 ** -6
    rel = np.abs(y[normal] - x[normal]) / np.abs(x[normal])
    assert rel.max() <= 2.0 ** -4 + 1e-12


def test_codes_have_exact_bf16_values():
    from paged_kv_attention_07_gb300 import workloads as W
    codes = np.arange(256)
    v = W.bf16_bits_to_f32(fp8.codes_to_bf16_bits(codes)).astype(np.float64)
    ref = fp8.decode(codes)
    assert np.array_equal(np.isnan(v), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(v[fin], ref[fin])


def test_fp8_cache_attention_matches_dense_float64():
    """An 8-bit cache (codes of the batch's K/V with per-tensor scales) through
    the oracle against torch SDPA on the dequantized dense K/V."""
    import oracle
    from paged_kv_attention_07_gb300 import workloads as W
    spec = W.spec_custom("fp8", ctx=[9, 40, 0], qlen=[1, 6, 5], num_decodes=1, num_extends=1,
                         num_prefills=1, Hq=4, Hkv=2, d=16, dv=16, bs=8, seed=12)
    batch = W.make_batch(spec)
    kc, vc = oracle.populate_cache(batch, "all")
    k_scale, v_scale = 0.0137, 0.0211  # arbitrary, not powers of two
    fin = lambda bits: W.bf16_bits_to_f32(bits).astype(np.float64)
    k_codes = fp8.quantize(np.nan_to_num(fin(kc)), k_scale)
    v_codes = fp8.quantize(np.nan_to_num(fin(vc)), v_scale)
    out, lse = fp8.attention_fp8(batch.q, k_codes, v_codes, k_scale, v_scale, batch.block_table,
                                 batch.query_start_loc, batch.seq_lens, spec.scale, spec.block_size)
    # dense reference on the dequantized values, request by request
    G = spec.num_q_heads // spec.num_kv_heads
    kd, vd = fp8.dequantize(k_codes, k_scale), fp8.dequantize(v_codes, v_scale)
    rows = []
    for r in range(spec.num_reqs):
        t0, t1 = int(batch.query_start_loc[r]), int(batch.query_start_loc[r + 1])
        S, ctx = int(batch.seq_lens[r]), spec.ctx[r]
        blocks = batch.block_table[r]
        K = np.stack([kd[blocks[j // spec.block_size], :, j % spec.block_size] for j in range(S)], 1)
        V = np.stack([vd[blocks[j // spec.block_size], :, j % spec.block_size] for j in range(S)], 1)
        q = torch.from_numpy(W.bf16_bits_to_f32(batch.q[t0:t1]).astype(np.float64)).permute(1, 0, 2)
        Kt = torch.from_numpy(K).repeat_interleave(G, 0)
        Vt = torch.from_numpy(V).repeat_interleave(G, 0)
        mask = torch.arange(S)[None, :] <= ctx + torch.arange(t1 - t0)[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(q, Kt, Vt, attn_mask=mask, scale=spec.scale)
        rows.append(o.permute(1, 0, 2).reshape(-1, spec.head_dim_v).numpy())
    np.testing.assert_allclose(out, np.concatenate(rows), rtol=0, atol=1e-12)
    assert np.isfinite(lse).all()


@pytest.mark.parametrize("scale", [0.0125, 0.02, 1.0 / 3.0, 7.0])
def test_float32_quotient_codes_match_torch(scale):
    # torch divides two float32 tensors in float32 and casts the quotient to
    # float8_e4m3fn (round to nearest even): in range, the same codes
    rng = np.random.default_rng(int(scale * 1000))
    x = (rng.standard_normal(20000) * 3.0).astype(np.float32)
    q = torch.from_numpy(x) / torch.tensor(scale, dtype=torch.float32)
    keep = (q.abs() <= fp8.MAX_FINITE).numpy()
    ref = q[torch.from_numpy(keep)].to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.quantize_f32(x, scale)[keep], ref)


def test_float32_quotient_differs_from_exact_only_at_double_rounding():
    # the float32 quotient can land exactly on a midpoint the exact quotient
    # misses; away from such cases the two encodings agree
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(50000)).astype(np.float32)
    s = 0.0123
    a, b = fp8.quantize_f32(x, s), fp8.quantize(x.astype(np.float64), np.float64(np.float32(s)))
    assert (a != b).sum() <= 5
    assert np.all(np.abs(fp8.decode(a) - fp8.decode(b))[a != b] <= 2.0 ** -3 * np.abs(fp8.decode(b))[a != b] + 2 ** -9)


def _snap_batch(batch, s):
    """The batch with its context rows and its decodes' new rows moved onto
    the grid of E4M3 values x s (s a power of two: those values are bf16
    values, so a cache of their codes holds them exactly); the extends' and
    prefills' new rows stay arbitrary bf16."""
    from paged_kv_attention_07_gb300 import workloads as W
    spec = batch.spec
    snap_rows = [batch.ctx_index]
    for r in range(spec.num_decodes):
        snap_rows.append(batch.seq_start[r] + np.arange(spec.ctx[r], spec.ctx[r] + spec.qlen[r]))
    idx = np.concatenate(snap_rows)
    for name in ("k_seq", "v_seq"):
        a = getattr(batch, name).copy()
        x = W.bf16_bits_to_f32(a[idx]).astype(np.float64)
        a[idx] = W.to_bf16_bits(fp8.dequantize(fp8.quantize(x, s), s).astype(np.float32))
        setattr(batch, name, a)
    return batch


def _codes_cache(batch, s):
    """Codes of every position (what the 8-bit cache write leaves), NaN code elsewhere."""
    from paged_kv_attention_07_gb300 import workloads as W
    spec = batch.spec
    shape = (batch.num_blocks, spec.num_kv_heads, spec.block_size)
    kc = np.full(shape + (spec.head_dim,), 0x7F, np.uint8)
    vc = np.full(shape + (spec.head_dim_v,), 0x7F, np.uint8)
    blk, off = batch.slot_all // spec.block_size, batch.slot_all % spec.block_size
    for cache, seq in ((kc, batch.k_seq), (vc, batch.v_seq)):
        codes = fp8.quantize_f32(W.bf16_bits_to_f32(seq), s)
        for hk in range(spec.num_kv_heads):
            cache[blk, hk, off] = codes[:, hk]
    return kc, vc


@pytest.mark.parametrize("bs,seed", [(8, 21), (1, 22), (16, 23)])
def test_step_reference_fp8_equals_plain_attention_on_exact_codes(bs, seed):
    """When every cached value is exactly a code's value, the 8-bit step
    reference must equal the plain definition (the C oracle) on a bf16 cache
    holding the same values, with the extends' and prefills' new tokens taken
    at full bf16 precision (they are not on the E4M3 grid here, so reading
    them from the cache instead would fail this)."""
    import oracle
    from paged_kv_attention_07_gb300 import workloads as W
    s = 2.0 ** -3
    spec = W.spec_custom("f8step", ctx=[5, 33, 20, 47, 0, 0], qlen=[1, 1, 7, 18, 9, 3], num_decodes=2,
                         num_extends=2, num_prefills=2, Hq=6, Hkv=2, d=16, dv=8, bs=bs, seed=seed)
    batch = _snap_batch(W.make_batch(spec), s)
    new_ext = batch.k_seq[batch.new_index][2:]  # the extends' and prefills' new rows
    x = W.bf16_bits_to_f32(new_ext).astype(np.float64)
    assert np.any(fp8.dequantize(fp8.quantize(x, s), s) != x)  # off the grid
    kc, vc = _codes_cache(batch, s)
    out, lse = fp8.step_reference_fp8(batch.q, kc, vc, batch.k_new, batch.v_new, s, s, batch.block_table,
                                      batch.query_start_loc, batch.seq_lens, spec.num_decodes, spec.scale,
                                      spec.block_size)
    kb, vb = oracle.populate_cache(batch, "all")
    ref_o, ref_l = oracle.attention(batch.q, kb, vb, batch.block_table, batch.query_start_loc, batch.seq_lens,
                                    spec.scale, spec.block_size, head_dim_v=spec.head_dim_v)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_step_reference_fp8_decodes_read_their_own_token_from_the_cache():
    """A decode-only step: every position, the new one included, comes from
    the codes, so the reference equals the oracle's attention over the 8-bit
    cache with arbitrary (not power-of-two) scales."""
    from paged_kv_attention_07_gb300 import workloads as W
    spec = W.spec_custom("f8dec", ctx=[3, 40, 17], qlen=[1, 1, 1], num_decodes=3, num_extends=0,
                         num_prefills=0, Hq=4, Hkv=1, d=16, dv=16, bs=4, seed=31)
    batch = W.make_batch(spec)
    ks, vs = 0.0137, 0.0211
    kc = _codes_cache(batch, ks)[0]
    vc = _codes_cache(batch, vs)[1]
    out, lse = fp8.step_reference_fp8(batch.q, kc, vc, batch.k_new, batch.v_new, ks, vs, batch.block_table,
                                      batch.query_start_loc, batch.seq_lens, 3, spec.scale, spec.block_size)
    ref_o, ref_l = fp8.attention_fp8(batch.q, kc, vc, ks, vs, batch.block_table, batch.query_start_loc,
                                     batch.seq_lens, spec.scale, spec.block_size)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)
