"""Seeded synthetic batches shaped like the serving workloads of the ROCm
attention-backend pages ("Beyond porting: how vLLM orchestrates high-performance
inference on AMD ROCm", section "Benchmark"; ISL 10K / OSL 1K random prompts,
max-num-batched-tokens 16384).

This module is the one piece shared by the CUDA path's harness and by the
oracle's tests. It draws random numbers, request lengths and a block-table
permutation, and derives each position's cache slot (the `slot_mapping` a
serving runtime hands to `reshape_and_cache`). It holds none of the attention
arithmetic: no scores, no softmax, no merge, no cache layout.

Conventions
-----------
* A request r has `ctx[r]` tokens already in the cache and `qlen[r]` new
  tokens; `seq_len[r] = ctx[r] + qlen[r]`. Requests are ordered
  [decode : extend : prefill].
* Values are float32 N(0, 1) draws rounded to bf16 (round-to-nearest-even);
  arrays hold the raw bf16 bit patterns as uint16.
* `k_seq` / `v_seq` hold the keys/values of EVERY position of every request,
  request-major (`seq_start[r] .. seq_start[r+1]`), before any cache layout.
  `slot_all[i]` is the cache slot of row i: block_table[r][pos // bs] * bs
  + pos % bs. The context rows are `ctx_index`, the new rows `new_index`
  (in batch token order), so `k_new = k_seq[new_index]`.
* Blocks: a random permutation of `num_blocks` ids, handed out in batch
  order, ceil(seq_len / bs) per request. Unused table entries hold 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BF16_QNAN = np.uint16(0x7FC0)
_CHUNK = 1 << 24  # elements drawn per RNG call (fixed, so the stream is reproducible)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round-to-nearest-even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


@dataclass
class BatchSpec:
    """Shape of one continuous batch (lengths already drawn)."""

    name: str
    seed: int
    ctx: list
    qlen: list
    num_decodes: int
    num_extends: int
    num_prefills: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    head_dim_v: int
    block_size: int
    scale: float
    context_chunk: int = 32768
    num_blocks: int = 0  # 0 -> exactly the blocks the batch needs
    mla: bool = False  # single latent cache, V = first head_dim_v dims of K

    @property
    def num_reqs(self) -> int:
        return len(self.ctx)

    @property
    def seq_lens(self) -> list:
        return [c + q for c, q in zip(self.ctx, self.qlen)]

    @property
    def num_tokens(self) -> int:
        return int(sum(self.qlen))

    def blocks_needed(self) -> int:
        bs = self.block_size
        return int(sum((s + bs - 1) // bs for s in self.seq_lens))


@dataclass
class Batch:
    spec: BatchSpec
    query_start_loc: np.ndarray  # int32 [B+1]
    seq_lens: np.ndarray  # int32 [B]
    block_table: np.ndarray  # int32 [B, max_blocks]
    q: np.ndarray  # uint16 [T, Hq, d]
    k_seq: np.ndarray  # uint16 [S_total, Hkv, d]
    v_seq: np.ndarray | None  # uint16 [S_total, Hkv, dv] (None for the latent cache)
    seq_start: np.ndarray  # int64 [B+1]
    slot_all: np.ndarray  # int64 [S_total]
    ctx_index: np.ndarray  # int64 rows of k_seq that are context
    new_index: np.ndarray  # int64 [T] rows of k_seq that are new tokens
    num_blocks: int
    extra: dict = field(default_factory=dict)

    @property
    def k_new(self) -> np.ndarray:
        return None if self.k_seq is None else self.k_seq[self.new_index]

    @property
    def v_new(self) -> np.ndarray | None:
        return None if self.v_seq is None else self.v_seq[self.new_index]

    @property
    def slot_mapping(self) -> np.ndarray:
        return self.slot_all[self.new_index]

    @property
    def max_blocks_per_req(self) -> int:
        return int(self.block_table.shape[1])


def make_batch(spec: BatchSpec, rng: np.random.Generator | None = None,
               block_perm: np.ndarray | None = None, values: bool = True) -> Batch:
    """Materialise a spec: Q, K, V draws, then the block permutation (in that
    order, so the values do not depend on the block size). With
    values=False only the metadata is built (q/k_seq/v_seq are None) and the
    permutation comes from default_rng(seed + 2000)."""
    if rng is None:
        rng = np.random.default_rng(spec.seed + 1000)
    B = spec.num_reqs
    bs = spec.block_size
    seq = np.asarray(spec.seq_lens, dtype=np.int64)
    ql = np.asarray(spec.qlen, dtype=np.int64)
    ctx = np.asarray(spec.ctx, dtype=np.int64)
    assert B == spec.num_decodes + spec.num_extends + spec.num_prefills
    T = int(ql.sum())
    S = int(seq.sum())
    Hq, Hkv, d, dv = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.head_dim_v
    if values:
        q = _normal_bf16(rng, (T, Hq, d))
        k_seq = _normal_bf16(rng, (S, Hkv, d))
        v_seq = None if spec.mla else _normal_bf16(rng, (S, Hkv, dv))
    else:
        q = k_seq = v_seq = None
        rng = np.random.default_rng(spec.seed + 2000)

    nblk = (seq + bs - 1) // bs
    need = int(nblk.sum())
    nb = spec.num_blocks or need
    assert nb >= need, "not enough cache blocks"
    perm = rng.permutation(nb).astype(np.int32) if block_perm is None else block_perm
    maxb = max(1, int(nblk.max()))
    bt = np.zeros((B, maxb), dtype=np.int32)
    off = 0
    for r in range(B):
        bt[r, : nblk[r]] = perm[off: off + nblk[r]]
        off += int(nblk[r])

    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(ql)
    seq_start = np.zeros(B + 1, dtype=np.int64)
    seq_start[1:] = np.cumsum(seq)
    slot_all = np.empty(S, dtype=np.int64)
    ctx_index, new_index = [], []
    for r in range(B):
        pos = np.arange(seq[r], dtype=np.int64)
        slot_all[seq_start[r]: seq_start[r + 1]] = bt[r, pos // bs].astype(np.int64) * bs + pos % bs
        ctx_index.append(seq_start[r] + np.arange(ctx[r], dtype=np.int64))
        new_index.append(seq_start[r] + ctx[r] + np.arange(ql[r], dtype=np.int64))
    ctx_index = np.concatenate(ctx_index) if ctx_index else np.zeros(0, np.int64)
    new_index = np.concatenate(new_index) if new_index else np.zeros(0, np.int64)
    return Batch(spec=spec, query_start_loc=qsl, seq_lens=seq.astype(np.int32), block_table=bt,
                 q=q, k_seq=k_seq, v_seq=v_seq, seq_start=seq_start, slot_all=slot_all,
                 ctx_index=ctx_index, new_index=new_index, num_blocks=nb)


# ---------------------------------------------------------------------------
# The five workloads (lengths drawn with numpy default_rng(seed)).
# ---------------------------------------------------------------------------

def spec_tiny(seed: int = 0) -> BatchSpec:
    """2 decodes (ctx 37, 100), 1 extend (ctx 64 + 16 new), 1 prefill (48),
    4 q heads / 2 kv heads, d 64, block 16 of a 64-block cache, scale 1/8,
    32-token context chunks."""
    return BatchSpec(name="tiny_mixed", seed=seed, ctx=[37, 100, 64, 0], qlen=[1, 1, 16, 48],
                     num_decodes=2, num_extends=1, num_prefills=1, num_q_heads=4, num_kv_heads=2,
                     head_dim=64, head_dim_v=64, block_size=16, scale=1.0 / 8.0,
                     context_chunk=32, num_blocks=64)


def spec_decode_gqa(seed: int = 1, num_reqs: int = 256, lo: int = 1024, hi: int = 8192,
                    block_size: int = 16) -> BatchSpec:
    """Decode-only GQA: ctx U[lo, hi], 32 q / 4 kv heads, d 128, block 16."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi, num_reqs, endpoint=True).tolist()
    return BatchSpec(name="decode_gqa", seed=seed, ctx=ctx, qlen=[1] * num_reqs,
                     num_decodes=num_reqs, num_extends=0, num_prefills=0, num_q_heads=32,
                     num_kv_heads=4, head_dim=128, head_dim_v=128, block_size=block_size,
                     scale=1.0 / math.sqrt(128))


def spec_prefill(seed: int = 2, num_seqs: int = 8, lo: int = 1024, hi: int = 4096,
                 max_total: int = 16384) -> BatchSpec:
    """Varlen causal prefill: lengths U[lo, hi], redrawn until the sum fits max_total."""
    rng = np.random.default_rng(seed)
    while True:
        lens = rng.integers(lo, hi, num_seqs, endpoint=True)
        if lens.sum() <= max_total:
            break
    return BatchSpec(name="prefill_varlen", seed=seed, ctx=[0] * num_seqs, qlen=lens.tolist(),
                     num_decodes=0, num_extends=0, num_prefills=num_seqs, num_q_heads=32,
                     num_kv_heads=4, head_dim=128, head_dim_v=128, block_size=16,
                     scale=1.0 / math.sqrt(128))


def spec_mixed(seed: int = 3, n_dec: int = 128, n_ext: int = 8, n_pre: int = 4,
               dec_lo: int = 2048, dec_hi: int = 16384, ext_lo: int = 32768, ext_hi: int = 102400,
               ext_new: int = 512, pre_len: int = 2048, chunk: int = 32768) -> BatchSpec:
    """[decode:extend:prefill]: 128 decodes (ctx 2K-16K), 8 extends (ctx 32K-100K,
    512 new), 4 prefills of 2048; 32/4 heads, d 128, block 16, 32K chunks."""
    rng = np.random.default_rng(seed)
    dctx = rng.integers(dec_lo, dec_hi, n_dec, endpoint=True).tolist()
    ectx = rng.integers(ext_lo, ext_hi, n_ext, endpoint=True).tolist()
    return BatchSpec(name="mixed", seed=seed, ctx=dctx + ectx + [0] * n_pre,
                     qlen=[1] * n_dec + [ext_new] * n_ext + [pre_len] * n_pre,
                     num_decodes=n_dec, num_extends=n_ext, num_prefills=n_pre, num_q_heads=32,
                     num_kv_heads=4, head_dim=128, head_dim_v=128, block_size=16,
                     scale=1.0 / math.sqrt(128), context_chunk=chunk)


def spec_mla_decode(seed: int = 4, num_reqs: int = 64, lo: int = 1024, hi: int = 32768,
                    block_size: int = 64, heads: int = 128) -> BatchSpec:
    """Absorbed MLA decode: 128 heads over one 576-dim latent (V = first 512)."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi, num_reqs, endpoint=True).tolist()
    return BatchSpec(name="mla_decode", seed=seed, ctx=ctx, qlen=[1] * num_reqs,
                     num_decodes=num_reqs, num_extends=0, num_prefills=0, num_q_heads=heads,
                     num_kv_heads=1, head_dim=576, head_dim_v=512, block_size=block_size,
                     scale=1.0 / math.sqrt(192), mla=True)


def spec_mla_prefill(seed: int = 5, n_ext: int = 8, n_pre: int = 4, ext_lo: int = 32768, ext_hi: int = 102400,
                     ext_new: int = 512, pre_len: int = 2048, heads: int = 128, chunk: int = 32768,
                     block_size: int = 16) -> BatchSpec:
    """MLA's non-absorbed prefill/extend (the decompressed form): 8 extends
    (ctx 32K-100K, 512 new) and 4 prefills of 2048 like the mixed workload,
    128 heads each with its own K (192 = 128 + 64 rope dims) and V (128),
    32K-token context chunks, scale 1/sqrt(192)."""
    rng = np.random.default_rng(seed)
    ectx = rng.integers(ext_lo, ext_hi, n_ext, endpoint=True).tolist()
    return BatchSpec(name="mla_prefill_extend", seed=seed, ctx=ectx + [0] * n_pre,
                     qlen=[ext_new] * n_ext + [pre_len] * n_pre, num_decodes=0, num_extends=n_ext,
                     num_prefills=n_pre, num_q_heads=heads, num_kv_heads=heads, head_dim=192, head_dim_v=128,
                     block_size=block_size, scale=1.0 / math.sqrt(192), context_chunk=chunk)


def spec_custom(name, ctx, qlen, num_decodes, num_extends, num_prefills, Hq, Hkv, d, dv, bs,
                scale=None, chunk=32768, num_blocks=0, mla=False, seed=0) -> BatchSpec:
    return BatchSpec(name=name, seed=seed, ctx=list(ctx), qlen=list(qlen), num_decodes=num_decodes,
                     num_extends=num_extends, num_prefills=num_prefills, num_q_heads=Hq,
                     num_kv_heads=Hkv, head_dim=d, head_dim_v=dv, block_size=bs,
                     scale=(1.0 / math.sqrt(d)) if scale is None else scale, context_chunk=chunk,
                     num_blocks=num_blocks, mla=mla)


def subset(spec: BatchSpec, requests) -> BatchSpec:
    """Same workload restricted to some requests (keeps the [dec:ext:pre] order)."""
    requests = sorted(requests)
    nd = sum(1 for r in requests if r < spec.num_decodes)
    ne = sum(1 for r in requests if spec.num_decodes <= r < spec.num_decodes + spec.num_extends)
    npf = len(requests) - nd - ne
    return BatchSpec(name=spec.name + "_subset", seed=spec.seed, ctx=[spec.ctx[r] for r in requests],
                     qlen=[spec.qlen[r] for r in requests], num_decodes=nd, num_extends=ne,
                     num_prefills=npf, num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                     head_dim=spec.head_dim, head_dim_v=spec.head_dim_v, block_size=spec.block_size,
                     scale=spec.scale, context_chunk=spec.context_chunk, num_blocks=0, mla=spec.mla)


ALL_SPECS = {
    "tiny_mixed": spec_tiny,
    "decode_gqa": spec_decode_gqa,
    "prefill_varlen": spec_prefill,
    "mixed": spec_mixed,
    "mla_decode": spec_mla_decode,
    "mla_prefill_extend": spec_mla_prefill,
}
