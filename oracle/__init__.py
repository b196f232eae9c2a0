"""Float64 CPU oracle for paged-KV attention (test infrastructure).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT: only `tests/`, the package's
`__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg may import it. It
shares no code with the CUDA library and never imports it.

`pka_oracle.c` holds the plain definition (see its header); this module loads
it with ctypes and adds, in numpy, the pages' own decomposition of a step so
the tests can check that the decomposition reaches the plain definition:

* `extend_forward` follows "Beyond porting" (page 2), section "Three-path
  processing explained", extend path: stage 1 attends the new tokens to
  themselves (causal), stage 2 loops over fixed-size context chunks, each
  giving an output and an LSE that are merged, stage 3 merges with stage 1.
* `split_kv_forward` is the same merge applied to contiguous key splits (the
  split-KV decode reduction).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None


def bind(path):
    """Load an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_cache_write.restype = i32
    lib.oracle_cache_write.argtypes = [P, P, P, i64, i32, i32, i32, P, P, i64, i32]
    lib.oracle_attention.restype = i32
    lib.oracle_attention.argtypes = [P, P, P, P, i32, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                     i64, dbl, P, i64, P, P, i32]
    lib.oracle_merge_attn_states.restype = None
    lib.oracle_merge_attn_states.argtypes = [i64, i32, P, P, P, P, P, P]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(build_oracle())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def cache_write(k, v, slot_mapping, k_cache, v_cache, block_size):
    """In-place scatter of new K/V rows (uint16 bf16 bits) into the caches."""
    lib = _load()
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = None if v is None else np.ascontiguousarray(v, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_cache.flags.c_contiguous and (v_cache is None or v_cache.flags.c_contiguous)
    T, Hkv, d = k.shape
    dv = 0 if v is None else v.shape[2]
    st = lib.oracle_cache_write(_ptr(k), _ptr(v), _ptr(slots), T, Hkv, d, dv, _ptr(k_cache),
                                _ptr(v_cache), k_cache.shape[0], block_size)
    if st != 0:
        raise ValueError(f"oracle_cache_write failed with status {st}")


def attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale, block_size,
              head_dim_v=None, rows=None, key_begin=None, key_end=None, nthreads=None):
    """Plain softmax attention through the block table, float64.

    Returns (out [n, dv] float64, lse [n] float64) for `rows` (flattened
    t * Hq + h, default all rows in order). `key_begin` / `key_end` (per
    request) restrict the key range on top of the causal bound.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    T, Hq, d = q.shape
    nb, Hkv = k_cache.shape[0], k_cache.shape[1]
    dv = head_dim_v if head_dim_v is not None else (v_cache.shape[3] if v_cache is not None else d)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    kb = None if key_begin is None else np.ascontiguousarray(key_begin, dtype=np.int32)
    ke = None if key_end is None else np.ascontiguousarray(key_end, dtype=np.int32)
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = T * Hq if rows_a is None else rows_a.shape[0]
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    if n == 0:
        return out, lse
    st = lib.oracle_attention(_ptr(q), _ptr(np.ascontiguousarray(k_cache)),
                              _ptr(None if v_cache is None else np.ascontiguousarray(v_cache)),
                              _ptr(bt), bt.shape[1], _ptr(qsl), _ptr(sl), sl.shape[0], _ptr(kb),
                              _ptr(ke), Hq, Hkv, d, dv, block_size, nb, float(scale), _ptr(rows_a), n,
                              _ptr(out), _ptr(lse), nthreads or default_threads())
    if st != 0:
        raise ValueError(f"oracle_attention failed with status {st}")
    return out, lse


def merge_attn_states(a_out, a_lse, b_out, b_lse):
    """LSE merge of two partial results (float64)."""
    lib = _load()
    a_out = np.ascontiguousarray(a_out, dtype=np.float64)
    b_out = np.ascontiguousarray(b_out, dtype=np.float64)
    a_lse = np.ascontiguousarray(a_lse, dtype=np.float64)
    b_lse = np.ascontiguousarray(b_lse, dtype=np.float64)
    n = a_lse.shape[0]
    dv = a_out.shape[-1]
    out = np.empty((n, dv), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    lib.oracle_merge_attn_states(n, dv, _ptr(a_out.reshape(n, dv)), _ptr(a_lse),
                                 _ptr(b_out.reshape(n, dv)), _ptr(b_lse), _ptr(out), _ptr(lse))
    return out, lse


def _rows_request_ranges(query_start_loc, seq_lens):
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    sl = np.asarray(seq_lens, dtype=np.int64)
    qlen = qsl[1:] - qsl[:-1]
    ctx = sl - qlen
    return qlen, ctx


def extend_forward(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale, block_size,
                   chunk, head_dim_v=None, nthreads=None):
    """The pages' extend path for every row of the batch, in the pages' order:

    1. attention of the new tokens over the new tokens' own keys (causal);
    2. for each context chunk c: attention over context keys
       [c*chunk, min((c+1)*chunk, ctx)), merged into a running context result;
    3. a final merge of the context result with stage 1.
    Requests without context (prefill, decode with ctx 0) get stage 1 only.
    """
    qlen, ctx = _rows_request_ranges(query_start_loc, seq_lens)
    sl = np.asarray(seq_lens, dtype=np.int64)
    common = dict(head_dim_v=head_dim_v, nthreads=nthreads)
    new_out, new_lse = attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale,
                                 block_size, key_begin=ctx, key_end=sl, **common)
    n_chunks = int(((ctx + chunk - 1) // chunk).max()) if len(ctx) else 0
    acc_out = np.zeros_like(new_out)
    acc_lse = np.full_like(new_lse, -np.inf)
    for c in range(n_chunks):
        kb = np.minimum(c * chunk, ctx)
        ke = np.minimum((c + 1) * chunk, ctx)
        o_c, l_c = attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale,
                             block_size, key_begin=kb, key_end=ke, **common)
        acc_out, acc_lse = merge_attn_states(acc_out, acc_lse, o_c, l_c)
    return merge_attn_states(acc_out, acc_lse, new_out, new_lse)


def split_kv_forward(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale, block_size,
                     split, head_dim_v=None, nthreads=None):
    """Every row's keys cut into contiguous splits of `split` positions from 0,
    each split attended separately and the partials LSE-merged in order."""
    sl = np.asarray(seq_lens, dtype=np.int64)
    n_splits = int(((sl + split - 1) // split).max())
    acc_out = acc_lse = None
    for s in range(n_splits):
        kb = np.minimum(s * split, sl)
        ke = np.minimum((s + 1) * split, sl)
        o_s, l_s = attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, scale,
                             block_size, key_begin=kb, key_end=ke, head_dim_v=head_dim_v,
                             nthreads=nthreads)
        if acc_out is None:
            acc_out, acc_lse = o_s, l_s
        else:
            acc_out, acc_lse = merge_attn_states(acc_out, acc_lse, o_s, l_s)
    return acc_out, acc_lse


def populate_cache(batch, positions="context"):
    """Host caches for a workloads.Batch, NaN-poisoned, with context rows (or
    all rows, positions="all") written by this oracle's cache_write."""
    spec = batch.spec
    nb, Hkv, bs = batch.num_blocks, spec.num_kv_heads, spec.block_size
    k_cache = np.full((nb, Hkv, bs, spec.head_dim), 0x7FC0, dtype=np.uint16)
    v_cache = None if spec.mla else np.full((nb, Hkv, bs, spec.head_dim_v), 0x7FC0, dtype=np.uint16)
    idx = batch.ctx_index if positions == "context" else np.arange(batch.k_seq.shape[0])
    if idx.size:
        cache_write(batch.k_seq[idx], None if batch.v_seq is None else batch.v_seq[idx],
                    batch.slot_all[idx], k_cache, v_cache, bs)
    return k_cache, v_cache


def batch_reference(batch, rows=None, nthreads=None):
    """Oracle output of a whole step for a workloads.Batch: cache_write of the
    new tokens into a context-populated cache, then plain attention."""
    spec = batch.spec
    k_cache, v_cache = populate_cache(batch, "context")
    cache_write(batch.k_new, batch.v_new, batch.slot_mapping, k_cache, v_cache, spec.block_size)
    return attention(batch.q, k_cache, v_cache, batch.block_table, batch.query_start_loc,
                     batch.seq_lens, spec.scale, spec.block_size, head_dim_v=spec.head_dim_v,
                     rows=rows, nthreads=nthreads)
