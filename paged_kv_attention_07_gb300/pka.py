"""ctypes binding of libpka.so (include/pka.h). Argument marshalling only.

Every function has the C entry point's name and meaning; tensors are torch
CUDA tensors whose shapes give the sizes, streams default to torch's current
stream. A non-OK status raises PkaError. Nothing here computes attention:
if libpka.so is missing the first call raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpka.so")

PKA_OK = 0
STATUS_NAMES = {0: "PKA_OK", 1: "PKA_ERR_INVALID_ARG", 2: "PKA_ERR_UNSUPPORTED",
                3: "PKA_ERR_WORKSPACE_TOO_SMALL", 4: "PKA_ERR_CUDA", 5: "PKA_ERR_DEVICE_METADATA"}
DEVERR = {"QUERY_START_LOC": 0x01, "SEQ_LEN": 0x02, "ORDER": 0x04, "QUERY_LEN": 0x08,
          "BLOCK_TABLE": 0x10, "BLOCK_ID": 0x20, "SLOT": 0x40, "CAPACITY": 0x80, "TIMEOUT": 0x100,
          "INDEX": 0x200}
EXPORTED = ("pka_cache_write", "pka_cache_write_fp8", "pka_workspace_size", "pka_workspace_size_fp8",
            "pka_paged_attn_forward",
            "pka_paged_attn_forward_fp8", "pka_paged_attn_step", "pka_paged_attn_step_fp8",
            "pka_merge_attn_states", "pka_get_error", "pka_paged_decode_noalloc", "pka_kernel_timer",
            "pka_kernel_timer_read", "pka_batch_order", "pka_gather_rows", "pka_selftest_wait",
            "pka_status_string")
KERNELS = {"cache_write": 0, "planner": 1, "decode": 2, "decode_reduce": 3, "prefill_extend": 4,
           "extend_reduce": 5, "merge": 6, "gather": 7, "ctx_dequant": 8}


class PkaError(RuntimeError):
    def __init__(self, status: int, where: str, code: int | None = None):
        self.status = status
        self.code = code
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        if code is not None:
            msg += f" (device error word 0x{code:x})"
        super().__init__(msg)


_lib = None


def load(path: str | None = None):
    """Load libpka.so (built by __graft_entry__.build()). Raises if missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libpka.so not found at {p}: the CUDA library must be built "
                           f"(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    lib.pka_cache_write.restype = i32
    lib.pka_cache_write.argtypes = [P, P, P, i64, i32, i32, i32, P, P, i64, i32, P, P]
    lib.pka_cache_write_fp8.restype = i32
    lib.pka_cache_write_fp8.argtypes = [P, P, P, i64, i32, i32, i32, P, P, i64, i32, f32, f32, P, P]
    lib.pka_paged_attn_forward_fp8.restype = i32
    lib.pka_paged_attn_forward_fp8.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                               i32, i32, i64, i32, f32, f32, f32, i32, i32, i32, P, P, P, sz, P]
    # q, k_new, v_new, slot_mapping, k_cache, v_cache, block_table, max_blocks, qsl, seq_lens, nd, ne, np, T,
    # Hq, Hkv, d, dv, num_blocks, bs, scale, [k_scale, v_scale,] chunk, max_q, max_s, out, lse, cw_err, ws,
    # ws_bytes, stream
    lib.pka_paged_attn_step.restype = i32
    lib.pka_paged_attn_step.argtypes = [P, P, P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                        i64, i32, f32, i32, i32, i32, P, P, P, P, sz, P]
    lib.pka_paged_attn_step_fp8.restype = i32
    lib.pka_paged_attn_step_fp8.argtypes = [P, P, P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                            i64, i32, f32, f32, f32, i32, i32, i32, P, P, P, P, sz, P]
    lib.pka_workspace_size.restype = sz
    lib.pka_workspace_size.argtypes = [i32] * 11
    lib.pka_workspace_size_fp8.restype = sz
    lib.pka_workspace_size_fp8.argtypes = [i32] * 11
    lib.pka_paged_attn_forward.restype = i32
    lib.pka_paged_attn_forward.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                           i32, i32, i64, i32, f32, i32, i32, i32, P, P, P, sz, P]
    lib.pka_merge_attn_states.restype = i32
    lib.pka_merge_attn_states.argtypes = [P, P, P, P, P, P, i64, i32, i32, P]
    lib.pka_get_error.restype = i32
    lib.pka_get_error.argtypes = [P, ctypes.POINTER(ctypes.c_int32), P]
    lib.pka_paged_decode_noalloc.restype = i32
    lib.pka_paged_decode_noalloc.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32, i64, i32, f32, i32,
                                             P, P, P, P]
    lib.pka_kernel_timer.restype = i32
    lib.pka_kernel_timer.argtypes = [i32, i32]
    lib.pka_kernel_timer_read.restype = i32
    lib.pka_kernel_timer_read.argtypes = [i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(ctypes.c_int)]
    lib.pka_status_string.restype = ctypes.c_char_p
    lib.pka_batch_order.restype = i32
    lib.pka_batch_order.argtypes = [i32, P, P, P, P, P, P, P]
    lib.pka_gather_rows.restype = i32
    lib.pka_gather_rows.argtypes = [P, P, P, i64, i64, i64, P, P]
    lib.pka_selftest_wait.argtypes = [i32, ctypes.c_uint32, ctypes.POINTER(ctypes.c_int32), P]
    lib.pka_selftest_wait.restype = i32
    lib.pka_status_string.argtypes = [i32]
    if path is None:
        _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, where: str):
    if st != PKA_OK:
        raise PkaError(st, where)


def pka_cache_write(k, v, slot_mapping, k_cache, v_cache, error_word=None, stream=None):
    """k [T, Hkv, d], v [T, Hkv, dv] or None, slot_mapping [T] int64,
    k_cache [nb, Hkv, bs, d], v_cache [nb, Hkv, bs, dv] or None."""
    T, Hkv, d = k.shape
    dv = 0 if v is None else v.shape[2]
    nb, _, bs, _ = k_cache.shape
    st = load().pka_cache_write(_ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, d, dv, _ptr(k_cache),
                                _ptr(v_cache), nb, bs, _ptr(error_word), _stream(stream))
    _check(st, "pka_cache_write")


def pka_cache_write_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, error_word=None, stream=None):
    """k [T, Hkv, d], v [T, Hkv, dv] bf16; caches [nb, Hkv, bs, d(v)] uint8 E4M3 codes."""
    T, Hkv, d = k.shape
    dv = v.shape[2]
    nb, _, bs, _ = k_cache.shape
    st = load().pka_cache_write_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, d, dv, _ptr(k_cache),
                                    _ptr(v_cache), nb, bs, float(k_scale), float(v_scale), _ptr(error_word),
                                    _stream(stream))
    _check(st, "pka_cache_write_fp8")


def pka_workspace_size(num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads,
                       head_dim, head_dim_v, max_query_len, max_seq_len, context_chunk_tokens) -> int:
    return int(load().pka_workspace_size(num_decodes, num_extends, num_prefills, num_tokens, num_q_heads,
                                         num_kv_heads, head_dim, head_dim_v, max_query_len, max_seq_len,
                                         context_chunk_tokens))


def pka_workspace_size_fp8(num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads,
                           head_dim, head_dim_v, max_query_len, max_seq_len, context_chunk_tokens) -> int:
    return int(load().pka_workspace_size_fp8(num_decodes, num_extends, num_prefills, num_tokens, num_q_heads,
                                             num_kv_heads, head_dim, head_dim_v, max_query_len, max_seq_len,
                                             context_chunk_tokens))


def pka_paged_attn_forward(q, k_new, v_new, k_cache, v_cache, block_table, query_start_loc, seq_lens,
                           num_decodes, num_extends, num_prefills, scale, context_chunk_tokens,
                           max_query_len, max_seq_len, out, lse, workspace, head_dim_v=None,
                           stream=None):
    """q [T, Hq, d]; k_new/v_new [T, Hkv, d] or None; caches as in pka_cache_write
    (v_cache None = latent cache); out [T, Hq, dv]; lse [T, Hq] float32 or None;
    workspace a uint8 CUDA tensor of >= pka_workspace_size(...) bytes."""
    T, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    dv = out.shape[2] if head_dim_v is None else head_dim_v
    st = load().pka_paged_attn_forward(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(query_start_loc), _ptr(seq_lens), num_decodes, num_extends,
        num_prefills, T, Hq, Hkv, d, dv, nb, bs, float(scale), context_chunk_tokens, max_query_len,
        max_seq_len, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(st, "pka_paged_attn_forward")


def pka_paged_attn_forward_fp8(q, k_new, v_new, k_cache, v_cache, block_table, query_start_loc, seq_lens,
                               num_decodes, num_extends, num_prefills, scale, k_scale, v_scale,
                               context_chunk_tokens, max_query_len, max_seq_len, out, lse, workspace, stream=None):
    """pka_paged_attn_forward over uint8 E4M3 caches with per-tensor scales."""
    T, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    dv = out.shape[2]
    st = load().pka_paged_attn_forward_fp8(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(query_start_loc), _ptr(seq_lens), num_decodes, num_extends,
        num_prefills, T, Hq, Hkv, d, dv, nb, bs, float(scale), float(k_scale), float(v_scale),
        context_chunk_tokens, max_query_len, max_seq_len, _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pka_paged_attn_forward_fp8")


def pka_paged_attn_step(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_table, query_start_loc, seq_lens,
                        num_decodes, num_extends, num_prefills, scale, context_chunk_tokens, max_query_len,
                        max_seq_len, out, lse, workspace, error_word=None, kv_scales=None, stream=None):
    """Cache write of the new tokens + forward pass in one call (bf16 cache, or
    an 8-bit cache with kv_scales=(k_scale, v_scale))."""
    T, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    dv = out.shape[2]
    common = (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
              block_table.shape[1], _ptr(query_start_loc), _ptr(seq_lens), num_decodes, num_extends, num_prefills,
              T, Hq, Hkv, d, dv, nb, bs, float(scale))
    tail = (context_chunk_tokens, max_query_len, max_seq_len, _ptr(out), _ptr(lse), _ptr(error_word),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if kv_scales is None:
        st = load().pka_paged_attn_step(*common, *tail)
    else:
        st = load().pka_paged_attn_step_fp8(*common, float(kv_scales[0]), float(kv_scales[1]), *tail)
    _check(st, "pka_paged_attn_step")


def pka_merge_attn_states(out, out_lse, prefix_out, prefix_lse, suffix_out, suffix_lse, stream=None):
    """out/prefix/suffix [rows..., head_dim] float32 or bf16 (same dtype), lse float32."""
    import torch
    io = {torch.float32: 0, torch.bfloat16: 1}[prefix_out.dtype]
    head_dim = prefix_out.shape[-1]
    rows = prefix_out.numel() // head_dim
    st = load().pka_merge_attn_states(_ptr(out), _ptr(out_lse), _ptr(prefix_out), _ptr(prefix_lse),
                                      _ptr(suffix_out), _ptr(suffix_lse), rows, head_dim, io,
                                      _stream(stream))
    _check(st, "pka_merge_attn_states")


def pka_get_error(workspace, stream=None) -> int:
    """Synchronise the stream and return the device error word (0 = clean)."""
    code = ctypes.c_int32(0)
    st = load().pka_get_error(_ptr(workspace), ctypes.byref(code), _stream(stream))
    if st not in (PKA_OK, 5):
        raise PkaError(st, "pka_get_error")
    return int(code.value)


def pka_kernel_timer(kernel: str, enable: bool = True):
    """Turn per-launch event timing of a kernel family on (resetting it) or off."""
    _check(load().pka_kernel_timer(KERNELS[kernel], 1 if enable else 0), "pka_kernel_timer")


def pka_kernel_timer_read(kernel: str):
    """(total device ms, launches, timed launches) of a kernel family since enabled."""
    ms, n, t = ctypes.c_double(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(load().pka_kernel_timer_read(KERNELS[kernel], ctypes.byref(ms), ctypes.byref(n),
                                        ctypes.byref(t)), "pka_kernel_timer_read")
    return float(ms.value), int(n.value), int(t.value)


def pka_batch_order(query_lens, ctx_lens):
    """Order a batch as [decode : extend : prefill] (host arrays, see include/pka.h).
    Returns (req_order[B], qsl_ordered[B+1], token_src[T], token_dst[T], counts[3]) as
    int32 numpy arrays."""
    import numpy as np
    q = np.ascontiguousarray(query_lens, dtype=np.int32)
    c = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    B, T = int(q.shape[0]), int(q.sum()) if q.size else 0
    order = np.zeros(B, np.int32)
    qsl = np.zeros(B + 1, np.int32)
    src = np.zeros(max(T, 1), np.int32)
    dst = np.zeros(max(T, 1), np.int32)
    counts = np.zeros(3, np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(load().pka_batch_order(B, p(q), p(c), p(order), p(qsl), p(src), p(dst), p(counts)), "pka_batch_order")
    return order, qsl, src[:T], dst[:T], counts


def pka_gather_rows(dst, src, index, error_word=None, stream=None):
    """dst[i] = src[index[i]] over the first dimension (packed rows); index is a
    CUDA int32 tensor of len(dst) entries."""
    if dst.shape[0] == 0:
        return
    if not (dst.is_contiguous() and src.is_contiguous() and index.is_contiguous()):
        raise ValueError("pka_gather_rows: dst, src and index must be contiguous (packed rows)")
    import torch
    if dst.dtype != src.dtype or dst[0].numel() != src[0].numel():
        raise ValueError("pka_gather_rows: dst and src rows must match")
    if index.dtype != torch.int32:
        raise ValueError("pka_gather_rows: index must be int32")
    if not (dst.is_cuda and src.is_cuda and index.is_cuda) or len({dst.device, src.device, index.device}) != 1:
        raise ValueError("pka_gather_rows: dst, src and index must be CUDA tensors on one device")
    if index.numel() < dst.shape[0]:
        raise ValueError("pka_gather_rows: index shorter than dst")
    row_bytes = dst[0].numel() * dst.element_size()
    _check(load().pka_gather_rows(_ptr(dst), _ptr(src), _ptr(index), int(dst.shape[0]), int(src.shape[0]),
                                  int(row_bytes), _ptr(error_word), _stream(stream)), "pka_gather_rows")


def pka_selftest_wait(arrive: bool, limit_us: int, stream=None) -> int:
    """Run the library's bounded mbarrier wait alone (see include/pka.h); returns
    the run's device error word (0, or PKA_DEVERR_TIMEOUT when nothing arrived)."""
    code = ctypes.c_int32(0)
    _check(load().pka_selftest_wait(1 if arrive else 0, int(limit_us), ctypes.byref(code),
                                    _stream(stream)), "pka_selftest_wait")
    return int(code.value)


def pka_status_string(status: int) -> str:
    return load().pka_status_string(status).decode()
