"""FP8 E4M3 codes for a KV cache stored in 8 bits with a per-tensor scale
(TEST INFRASTRUCTURE, like the rest of `oracle/`; next row f3 of the build:
the cache the pages' `gather_and_maybe_dequant_cache` step dequantises).

Written from the format's definition (the "fn" variant: no infinities):
bit 7 sign, bits 6..3 exponent with bias 7, bits 2..0 mantissa. Exponent
field 0 holds the subnormals m * 2^-9; otherwise the value is
(1 + m/8) * 2^(e - 7). The all-ones pattern S.1111.111 is NaN, so the largest
finite magnitude is 1.75 * 2^8 = 448. Encoding rounds to the nearest code,
ties to the even code, and saturates finite values beyond 448 to +-448.
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0


def _decode_definition(c: np.ndarray) -> np.ndarray:
    """The format's definition, applied to int64 codes."""
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


_VALUE = _decode_definition(np.arange(256, dtype=np.int64))  # value of every code


def decode(codes) -> np.ndarray:
    """float64 value of each 8-bit code (NaN for the two NaN codes)."""
    return _VALUE[np.asarray(codes, dtype=np.uint8)]


_POS = decode(np.arange(0x7F))  # the 127 non-negative finite values, ascending with the code


def encode(x) -> np.ndarray:
    """Nearest code (ties to the even code), finite values beyond 448
    saturated to +-448, NaN to 0x7F; the sign of zero is kept."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), MAX_FINITE)
    hi = np.clip(np.searchsorted(_POS, a, side="left"), 0, len(_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - _POS[lo], _POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize(x, scale: float) -> np.ndarray:
    """Codes of x / scale (scale > 0)."""
    return encode(np.asarray(x, dtype=np.float64) / scale)


def quantize_f32(x, scale: float) -> np.ndarray:
    """Codes of the float32 quotient x / scale: x and scale are float32 values,
    the division is IEEE float32 (round to nearest even), and that quotient is
    encoded. This is where the code is decided for the 8-bit cache write, so
    both the kernel and this reference take the decision in float32 (the
    pages fix no precision for the scale division)."""
    xf = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore"):
        qf = xf / np.float32(scale)
    return encode(qf.astype(np.float64))


def dequantize(codes, scale: float) -> np.ndarray:
    """code value * scale, float64."""
    return decode(codes) * scale


def codes_to_bf16_bits(codes) -> np.ndarray:
    """bf16 bit patterns of the codes' values. Exact: every E4M3 value (3
    mantissa bits, exponents 2^-9 .. 2^8) is a bf16 value; NaN stays NaN."""
    v = decode(codes).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def attention_fp8(q, k_codes, v_codes, k_scale, v_scale, block_table, query_start_loc, seq_lens, scale,
                  block_size, **kw):
    """Attention over an 8-bit cache with per-tensor scales: K = k_scale x code,
    V = v_scale x code. The scales come out of the sums (the score scale
    becomes scale x k_scale, the output is multiplied by v_scale, the LSE
    does not change), so the plain definition in `pka_oracle.c` runs on the
    codes' exact bf16 values. Returns (out, lse) like `oracle.attention`."""
    from . import attention
    out, lse = attention(q, codes_to_bf16_bits(k_codes), codes_to_bf16_bits(v_codes), block_table,
                         query_start_loc, seq_lens, scale * k_scale, block_size, **kw)
    return out * v_scale, lse


def _bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def step_reference_fp8(q, k_codes, v_codes, k_new, v_new, k_scale, v_scale, block_table, query_start_loc,
                       seq_lens, num_decodes, scale, block_size, rows=None):
    """One step over an 8-bit cache, float64, written out per request and head.

    Which values a query sees (the pages' prefill listing: the new tokens'
    attention runs on the step's own K/V, the context chunks on the cache
    gathered and dequantised, `gather_and_maybe_dequant_cache`):
      * a decode request (the first `num_decodes`) reads every position from
        the cache, its own new token included (the cache write stored it):
        K_j = k_scale * code_j, V_j = v_scale * code_j;
      * an extend or prefill request reads its ctx cached positions from the
        cache the same way and its new tokens' K/V from k_new / v_new (bf16).
    Query i of a request with ctx cached tokens sits at position ctx + i and
    sees keys 0 .. ctx + i (bottom-right causal); s_j = scale * <q, K_j>,
    lse = log sum_j e^{s_j}, out = sum_j e^{s_j - lse} V_j.

    q, k_new, v_new: bf16 bits [T, H, d]; k_codes / v_codes: uint8
    [blocks, Hkv, bs, d]. Returns (out, lse) for `rows` (flattened t * Hq + h,
    default every row in order)."""
    q = np.asarray(q)
    T, Hq, d = q.shape
    Hkv, dv = k_codes.shape[1], v_codes.shape[3]
    G = Hq // Hkv
    rows = np.arange(T * Hq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, dv))
    lse = np.zeros(rows.size)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    row_t, row_h = rows // Hq, rows % Hq
    row_r = np.searchsorted(qsl, row_t, side="right") - 1  # request of each row
    for r in np.unique(row_r):
        t0, t1 = int(qsl[r]), int(qsl[r + 1])
        n, s = t1 - t0, int(seq_lens[r])
        ctx = s - n
        cached = s if r < num_decodes else ctx  # positions read from the cache
        pos = np.arange(cached)
        blk = np.asarray(block_table[r], dtype=np.int64)[pos // block_size]
        for hk in range(Hkv):
            mine = np.nonzero((row_r == r) & (row_h // G == hk))[0]
            if mine.size == 0:
                continue
            K = dequantize(k_codes[blk, hk, pos % block_size], k_scale)
            V = dequantize(v_codes[blk, hk, pos % block_size], v_scale)
            if cached < s:
                K = np.concatenate([K, _bf16_bits_to_f64(k_new[t0:t1, hk])])
                V = np.concatenate([V, _bf16_bits_to_f64(v_new[t0:t1, hk])])
            for i in mine:
                t, h = int(row_t[i]), int(row_h[i])
                vis = ctx + (t - t0) + 1  # keys 0 .. ctx + (t - t0)
                sc = scale * (K[:vis] @ _bf16_bits_to_f64(q[t, h]))
                m = sc.max()
                e = np.exp(sc - m)
                den = e.sum()
                out[i] = (e @ V[:vis]) / den
                lse[i] = m + np.log(den)
    return out, lse
