"""GPU parity of the 8-bit (FP8 E4M3) KV cache: the quantising cache write
bit for bit against the oracle's codes (float32 quotient, nearest code, ties
to even, saturation), and the forward over the codes against the oracle's
8-bit step: decodes read every position from the codes, extends their
cached positions (gathered into the workspace) with their new tokens from
k_new / v_new, prefills only k_new / v_new."""
import numpy as np
import pytest

from oracle import fp8
from paged_kv_attention_07_gb300 import workloads as W
from tests.gpu_util import LSE_ATOL, OUT_ATOL

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 0.0125, 0.02


_CODE_TABLES = {}


def _codes_of(bits, scale):
    """Codes of bf16 values: the oracle's float32-quotient quantiser applied
    once to every bf16 bit pattern, then looked up."""
    if scale not in _CODE_TABLES:
        every = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        with np.errstate(invalid="ignore"):  # the NaN patterns encode to the NaN code
            _CODE_TABLES[scale] = fp8.quantize_f32(W.bf16_bits_to_f32(every), scale)
    return _CODE_TABLES[scale][np.asarray(bits, dtype=np.uint16)]


def oracle_fp8_cache(batch, k_scale, v_scale):
    """The oracle's 8-bit caches after the step's cache write: every position
    (context and new tokens) quantised, every other slot the NaN code.
    Quantised request by request (bounded host memory at full size)."""
    spec = batch.spec
    shape = (batch.num_blocks, spec.num_kv_heads, spec.block_size)
    kc = np.full(shape + (spec.head_dim,), 0x7F, np.uint8)
    vc = np.full(shape + (spec.head_dim_v,), 0x7F, np.uint8)
    for r in range(spec.num_reqs):
        a, b = int(batch.seq_start[r]), int(batch.seq_start[r + 1])
        blk, off = batch.slot_all[a:b] // spec.block_size, batch.slot_all[a:b] % spec.block_size
        k, v = _codes_of(batch.k_seq[a:b], k_scale), _codes_of(batch.v_seq[a:b], v_scale)
        for hk in range(spec.num_kv_heads):
            kc[blk, hk, off] = k[:, hk]
            vc[blk, hk, off] = v[:, hk]
    return kc, vc


def run_fp8(batch, k_scale=K_SCALE, v_scale=V_SCALE):
    import torch
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    db = DeviceBatch(batch, kv_scales=(k_scale, v_scale))
    db.step()
    torch.cuda.synchronize()
    assert db.canaries_intact()
    return db


def check_fp8(batch, k_scale=K_SCALE, v_scale=V_SCALE, rows=None):
    db = run_fp8(batch, k_scale, v_scale)
    assert db.error_word() == 0
    spec = batch.spec
    out = db.out.float().cpu().numpy().reshape(-1, spec.head_dim_v)
    lse = db.lse.cpu().numpy().reshape(-1)
    k_dev, v_dev = db.k_cache.cpu().numpy(), db.v_cache.cpu().numpy()
    del db
    kc, vc = oracle_fp8_cache(batch, k_scale, v_scale)
    # the cache the kernel read is exactly the oracle's codes
    assert np.array_equal(k_dev, kc)
    assert np.array_equal(v_dev, vc)
    del k_dev, v_dev
    ref_o, ref_l = fp8.step_reference_fp8(batch.q, kc, vc, batch.k_new, batch.v_new, k_scale, v_scale,
                                          batch.block_table, batch.query_start_loc, batch.seq_lens,
                                          spec.num_decodes, spec.scale, spec.block_size, rows=rows)
    if rows is not None:
        out, lse = out[rows], lse[rows]
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    eo, el = np.abs(out - ref_o).max(), np.abs(lse - ref_l).max()
    assert eo <= OUT_ATOL and el <= LSE_ATOL, (eo, el)
    return eo, el


DEC_CTX = [0, 1, 15, 16, 17, 255, 256, 257, 600, 1500, 4100]


@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 64, 128])
def test_fp8_decode_block_sizes(bs):
    spec = W.spec_custom(f"f8_bs{bs}", ctx=DEC_CTX, qlen=[1] * len(DEC_CTX), num_decodes=len(DEC_CTX),
                         num_extends=0, num_prefills=0, Hq=32, Hkv=4, d=128, dv=128, bs=bs, seed=100 + bs)
    check_fp8(W.make_batch(spec))


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (32, 4), (32, 2), (6, 3)])
def test_fp8_decode_groups(Hq, Hkv):
    spec = W.spec_custom(f"f8_g{Hq // Hkv}", ctx=DEC_CTX, qlen=[1] * len(DEC_CTX), num_decodes=len(DEC_CTX),
                         num_extends=0, num_prefills=0, Hq=Hq, Hkv=Hkv, d=128, dv=128, bs=16, seed=200 + Hq)
    check_fp8(W.make_batch(spec))


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.004, 0.05)])
def test_fp8_decode_scales(k_scale, v_scale):
    # scale 1: N(0,1) values use few codes; 0.004: many values saturate at 448
    spec = W.spec_custom("f8_sc", ctx=[30, 700, 2500], qlen=[1, 1, 1], num_decodes=3, num_extends=0,
                         num_prefills=0, Hq=16, Hkv=2, d=128, dv=128, bs=16, seed=7)
    check_fp8(W.make_batch(spec), k_scale, v_scale)


def test_fp8_decode_config_shape():
    """Every row of the decode-only GQA workload (256 requests, context
    U[1024, 8192], 32 query / 4 KV heads, head dim 128, block 16)."""
    check_fp8(W.make_batch(W.spec_decode_gqa()))


def test_fp8_cache_write_rounding_cases():
    """Hand-placed values: exact ties (to the even code), saturation, values
    below half the smallest subnormal, signed zero, a skipped (negative) slot
    and an out-of-range slot (flagged, skipped)."""
    import torch
    from paged_kv_attention_07_gb300 import pka
    s = 0.5  # a power of two: x / s is exact, so the ties below are real ties
    vals = np.array([1.0625, 1.1875, -1.0625, 500.0, -2.0 ** 20, 2.0 ** -10, 3 * 2.0 ** -10, 0.0, -0.0, 448.0,
                     464.0, 2.0 ** -11, 1.0, -2.5, 0.375, 7.0], np.float32) * np.float32(s)
    T, Hkv, d = 4, 1, 16
    x = np.tile(vals, (T, Hkv, 1)).astype(np.float32)
    x[1] *= -1
    bits = W.to_bf16_bits(x)
    assert np.array_equal(W.bf16_bits_to_f32(bits), x)  # every value is a bf16 value
    nb, bs = 4, 2
    slots = np.array([0, 5, -1, nb * bs + 1], np.int64)
    kc = torch.full((nb, Hkv, bs, d), 0x7F, dtype=torch.uint8, device="cuda")
    vc = torch.full((nb, Hkv, bs, d), 0x7F, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kt = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    pka.pka_cache_write_fp8(kt, kt, torch.from_numpy(slots).cuda(), kc, vc, s, 2 * s, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pka.DEVERR["SLOT"]
    ref_k = np.full((nb, Hkv, bs, d), 0x7F, np.uint8)
    ref_v = ref_k.copy()
    for t in range(2):
        blk, off = divmod(int(slots[t]), bs)
        ref_k[blk, 0, off] = fp8.quantize_f32(x[t, 0], s)
        ref_v[blk, 0, off] = fp8.quantize_f32(x[t, 0], 2 * s)
    assert np.array_equal(kc.cpu().numpy(), ref_k)
    assert np.array_equal(vc.cpu().numpy(), ref_v)
    # the first row's codes, spelled out: ties to even, saturation, subnormal ties, signed zero
    assert ref_k[0, 0, 0, :12].tolist() == [0x38, 0x3A, 0xB8, 0x7E, 0xFE, 0x00, 0x02, 0x00, 0x80, 0x7E, 0x7E, 0x00]


@pytest.mark.slow
def test_fp8_mixed_full():
    """The mixed workload (128 decodes, 8 extends with up to 100K context in
    32K chunks, 4 prefills) over an 8-bit cache, in the benchmark's launch
    configuration: the whole cache bit for bit, every decode row, the first
    and last token of every request and a seeded sample of other rows."""
    from tests.gpu_util import sample_rows
    batch = W.make_batch(W.spec_mixed())
    check_fp8(batch, rows=sample_rows(batch, 4096, seed=4))


@pytest.mark.parametrize("bs,chunk", [(16, 64), (1, 48), (64, 1000), (128, 128), (8, 32768)])
def test_fp8_mixed_step(bs, chunk):
    """Decodes, extends (context over several chunks, ragged tails) and
    prefills in one step over an 8-bit cache."""
    spec = W.spec_custom(f"f8_mix{bs}_{chunk}", ctx=[7, 300, 1100, 129, 700, 255, 0, 0],
                         qlen=[1, 1, 1, 40, 130, 3, 200, 17], num_decodes=3, num_extends=3, num_prefills=2,
                         Hq=16, Hkv=2, d=128, dv=128, bs=bs, chunk=chunk, seed=400 + bs)
    check_fp8(W.make_batch(spec))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 4), (12, 4)])
def test_fp8_extend_only(Hq, Hkv):
    spec = W.spec_custom(f"f8_ext{Hq}", ctx=[1, 64, 500, 2000], qlen=[5, 256, 70, 129], num_decodes=0,
                         num_extends=4, num_prefills=0, Hq=Hq, Hkv=Hkv, d=128, dv=128, bs=16, chunk=512,
                         seed=410 + Hq)
    check_fp8(W.make_batch(spec))


def test_fp8_prefill_only():
    spec = W.spec_custom("f8_pre", ctx=[0, 0, 0], qlen=[1, 300, 129], num_decodes=0, num_extends=0,
                         num_prefills=3, Hq=8, Hkv=2, d=128, dv=128, bs=16, seed=420)
    check_fp8(W.make_batch(spec))


def test_fp8_one_token_extends():
    """Requests with one new token routed through the extend slice read
    their context from the gathered cache and their own token from k_new."""
    spec = W.spec_custom("f8_uni", ctx=[10, 900, 33], qlen=[1, 1, 1], num_decodes=0, num_extends=3,
                         num_prefills=0, Hq=8, Hkv=2, d=128, dv=128, bs=16, chunk=256, seed=430)
    check_fp8(W.make_batch(spec))


def test_fp8_unsupported_shapes_are_refused():
    """Shapes the 8-bit path has no kernel for are refused before any launch."""
    from paged_kv_attention_07_gb300 import pka
    assert pka.pka_workspace_size_fp8(1, 1, 1, 8, 8, 2, 64, 64, 6, 100, 32) == 0
    assert pka.pka_workspace_size_fp8(1, 1, 1, 8, 8, 2, 192, 128, 6, 100, 32) == 0
    assert pka.pka_workspace_size_fp8(1, 1, 1, 8, 8, 2, 128, 128, 6, 100, 32) > 0
