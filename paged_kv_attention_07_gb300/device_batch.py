"""A synthetic batch resident on the GPU, driven through the C ABI.

Holds the device copies of a `workloads.Batch` (metadata, Q, the new
tokens' K/V, the paged caches, outputs and the workspace) and runs one step:
`pka_cache_write` of the new tokens, then `pka_paged_attn_forward`. The
caches start NaN-poisoned and receive the context rows through
`pka_cache_write`, so every slot the batch does not own stays NaN.
"""
from __future__ import annotations

import numpy as np
import torch

from . import pka
from . import workloads as W


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


GUARD_BYTES = 4096  # canary bytes before and after each output and the workspace
CANARY = 0xA5


def guarded_empty(nbytes: int, device) -> tuple[torch.Tensor, torch.Tensor]:
    """A zeroed uint8 buffer of nbytes with GUARD_BYTES of CANARY on both sides
    (the offset keeps the start 256-byte aligned). Returns (whole, inner)."""
    buf = torch.full((GUARD_BYTES + nbytes + GUARD_BYTES,), CANARY, dtype=torch.uint8, device=device)
    inner = buf[GUARD_BYTES:GUARD_BYTES + nbytes]
    inner.zero_()
    return buf, inner


def canary_intact(buf: torch.Tensor) -> bool:
    return bool(torch.all(buf[:GUARD_BYTES] == CANARY)) and bool(torch.all(buf[-GUARD_BYTES:] == CANARY))


FP8_NAN = 0x7F  # an E4M3 NaN code: the poison of an 8-bit cache


class DeviceBatch:
    """kv_scales=(k_scale, v_scale) makes the caches 8-bit (E4M3 codes with one
    scale per tensor): written by pka_cache_write_fp8, read by
    pka_paged_attn_forward_fp8."""

    def __init__(self, batch: W.Batch, device="cuda", values_on_device_seed: int | None = None,
                 unified: bool = False, kv_scales: tuple[float, float] | None = None):
        spec = batch.spec
        self.batch, self.spec, self.device = batch, spec, device
        self.kv_scales = kv_scales
        # unified: the decodes go in the extend slice (num_decodes 0), so every
        # request with context runs through the extend path
        nd = 0 if unified else spec.num_decodes
        self.counts = (nd, spec.num_extends + spec.num_decodes - nd, spec.num_prefills)
        Hq, Hkv, d, dv, bs = (spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.head_dim_v,
                              spec.block_size)
        T = spec.num_tokens
        S = int(batch.seq_start[-1])
        self.qsl = torch.from_numpy(batch.query_start_loc).to(device)
        self.seq_lens = torch.from_numpy(batch.seq_lens).to(device)
        self.block_table = torch.from_numpy(batch.block_table).to(device)
        self.slot_mapping = torch.from_numpy(np.ascontiguousarray(batch.slot_mapping)).to(device)
        nb = batch.num_blocks
        if kv_scales is None:
            self.k_cache = torch.full((nb, Hkv, bs, d), float("nan"), dtype=torch.bfloat16, device=device)
            self.v_cache = None if spec.mla else torch.full((nb, Hkv, bs, dv), float("nan"),
                                                            dtype=torch.bfloat16, device=device)
        else:
            assert not spec.mla, "the 8-bit cache holds separate K and V"
            self.k_cache = torch.full((nb, Hkv, bs, d), FP8_NAN, dtype=torch.uint8, device=device)
            self.v_cache = torch.full((nb, Hkv, bs, dv), FP8_NAN, dtype=torch.uint8, device=device)
        if values_on_device_seed is None:
            self.q = bf16_tensor(batch.q, device)
            k_seq = bf16_tensor(batch.k_seq, device)
            v_seq = None if batch.v_seq is None else bf16_tensor(batch.v_seq, device)
        else:  # same shapes, N(0,1) drawn on the device (fast path for large benchmarks)
            g = torch.Generator(device=device)
            g.manual_seed(values_on_device_seed)
            self.q = torch.randn((T, Hq, d), generator=g, device=device).to(torch.bfloat16)
            k_seq = torch.randn((S, Hkv, d), generator=g, device=device).to(torch.bfloat16)
            v_seq = None if spec.mla else torch.randn((S, Hkv, dv), generator=g,
                                                      device=device).to(torch.bfloat16)
        new_idx = torch.from_numpy(batch.new_index).to(device)
        ctx_idx = torch.from_numpy(batch.ctx_index).to(device)
        slot_all = torch.from_numpy(batch.slot_all).to(device)
        self.k_new = k_seq.index_select(0, new_idx).contiguous()
        self.v_new = None if v_seq is None else v_seq.index_select(0, new_idx).contiguous()
        if ctx_idx.numel():
            kc = k_seq.index_select(0, ctx_idx).contiguous()
            vc = None if v_seq is None else v_seq.index_select(0, ctx_idx).contiguous()
            self._write(kc, vc, slot_all.index_select(0, ctx_idx).contiguous())
            del kc, vc
        del k_seq, v_seq
        # out, lse and the workspace sit between canary bytes: a store past
        # either end of them shows up in canaries_intact()
        self._out_buf, inner = guarded_empty(T * Hq * dv * 2, device)
        self.out = inner.view(torch.bfloat16).view(T, Hq, dv)
        self._lse_buf, inner = guarded_empty(T * Hq * 4, device)
        self.lse = inner.view(torch.float32).view(T, Hq)
        self.max_query_len = int(max(spec.qlen))
        self.max_seq_len = int(max(spec.seq_lens))
        size_fn = pka.pka_workspace_size if kv_scales is None else pka.pka_workspace_size_fp8
        ws = size_fn(*self.counts, T, Hq, Hkv, d, dv, self.max_query_len, self.max_seq_len, spec.context_chunk)
        if ws == 0:
            raise RuntimeError("pka_workspace_size rejected the batch shape")
        self._ws_buf, self.workspace = guarded_empty(ws, device)
        torch.cuda.synchronize()

    INPUTS = ("q", "k_new", "v_new", "slot_mapping", "qsl", "seq_lens", "block_table")

    def pack_io(self):
        """Move the step's inputs into one contiguous device arena, and out and
        lse into one guarded buffer (each piece 256-byte aligned), so a host
        loop moves a step's inputs with one copy and its results with another
        (what a server does with persistent staging buffers). Returns
        (input arena, output span): uint8 views covering exactly those bytes."""
        def place(names):
            offs, off = {}, 0
            for n in names:
                t = getattr(self, n)
                if t is None:
                    continue
                offs[n] = off
                off = (off + t.numel() * t.element_size() + 255) // 256 * 256
            return offs, off
        offs, total = place(self.INPUTS)
        arena = torch.empty(total, dtype=torch.uint8, device=self.device)
        for n, o in offs.items():
            t = getattr(self, n)
            nbytes = t.numel() * t.element_size()
            view = arena[o:o + nbytes].view(t.dtype).view(t.shape)
            view.copy_(t)
            setattr(self, n, view)
        self._in_offs = offs
        T, Hq, dv = self.out.shape
        lse_off = (T * Hq * dv * 2 + 255) // 256 * 256
        span = lse_off + T * Hq * 4
        self._out_buf, inner = guarded_empty(span, self.device)
        self._lse_off = lse_off
        self.out = inner[:T * Hq * dv * 2].view(torch.bfloat16).view(T, Hq, dv)
        self.lse = inner[lse_off:span].view(torch.float32).view(T, Hq)
        self._lse_buf = self._out_buf
        torch.cuda.synchronize()
        return arena, inner

    def use_io(self, arena: torch.Tensor, outs: torch.Tensor):
        """Point the step at another input arena and output span laid out as
        pack_io's (double buffering: the next step's inputs arrive while this
        one runs)."""
        for n, o in self._in_offs.items():
            t = getattr(self, n)
            setattr(self, n, arena[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape))
        T, Hq, dv = self.out.shape
        self.out = outs[:T * Hq * dv * 2].view(torch.bfloat16).view(T, Hq, dv)
        self.lse = outs[self._lse_off:self._lse_off + T * Hq * 4].view(torch.float32).view(T, Hq)

    def canaries_intact(self) -> bool:
        """True when no byte next to out, lse or the workspace was written."""
        torch.cuda.synchronize()
        return all(canary_intact(b) for b in (self._out_buf, self._lse_buf, self._ws_buf))

    def refill(self, batch: W.Batch):
        """Write another batch with the same request counts and token count, and
        lengths within this one's hints, into the same device buffers (what a
        server does between replays of a captured step): metadata, Q, the new
        tokens' K/V, and the cache (poisoned again, then the new context rows)."""
        s, spec = self.spec, batch.spec
        assert (spec.num_decodes, spec.num_extends, spec.num_prefills) == (
            s.num_decodes, s.num_extends, s.num_prefills)
        assert spec.num_tokens == s.num_tokens and batch.num_blocks <= self.k_cache.shape[0]
        assert max(spec.qlen) <= self.max_query_len and max(spec.seq_lens) <= self.max_seq_len
        assert batch.block_table.shape[1] <= self.block_table.shape[1]
        dev = self.device
        bt = np.zeros(tuple(self.block_table.shape), dtype=np.int32)
        bt[:, : batch.block_table.shape[1]] = batch.block_table
        self.block_table.copy_(torch.from_numpy(bt))
        self.qsl.copy_(torch.from_numpy(batch.query_start_loc))
        self.seq_lens.copy_(torch.from_numpy(batch.seq_lens))
        self.slot_mapping.copy_(torch.from_numpy(np.ascontiguousarray(batch.slot_mapping)))
        self.q.copy_(bf16_tensor(batch.q, dev))
        self.k_new.copy_(bf16_tensor(batch.k_new, dev))
        if self.v_new is not None:
            self.v_new.copy_(bf16_tensor(batch.v_new, dev))
        poison = float("nan") if self.kv_scales is None else FP8_NAN
        self.k_cache.fill_(poison)
        if self.v_cache is not None:
            self.v_cache.fill_(poison)
        if batch.ctx_index.size:
            ci = batch.ctx_index
            kc = bf16_tensor(batch.k_seq[ci], dev)
            vc = None if batch.v_seq is None else bf16_tensor(batch.v_seq[ci], dev)
            self._write(kc, vc, torch.from_numpy(batch.slot_all[ci]).to(dev))
        self.batch = batch
        torch.cuda.synchronize()

    def _write(self, k, v, slots, stream=None):
        if self.kv_scales is None:
            pka.pka_cache_write(k, v, slots, self.k_cache, self.v_cache, stream=stream)
        else:
            pka.pka_cache_write_fp8(k, v, slots, self.k_cache, self.v_cache, *self.kv_scales, stream=stream)

    def cache_write(self, stream=None):
        self._write(self.k_new, self.v_new, self.slot_mapping, stream=stream)

    def forward(self, stream=None, out=None, lse=None):
        s = self.spec
        if self.kv_scales is not None:
            pka.pka_paged_attn_forward_fp8(
                self.q, self.k_new, self.v_new, self.k_cache, self.v_cache, self.block_table, self.qsl,
                self.seq_lens, *self.counts, s.scale, *self.kv_scales, s.context_chunk, self.max_query_len,
                self.max_seq_len, self.out if out is None else out, self.lse if lse is None else lse,
                self.workspace, stream=stream)
            return
        pka.pka_paged_attn_forward(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                   self.block_table, self.qsl, self.seq_lens, *self.counts, s.scale,
                                   s.context_chunk,
                                   self.max_query_len, self.max_seq_len,
                                   self.out if out is None else out,
                                   self.lse if lse is None else lse, self.workspace,
                                   head_dim_v=s.head_dim_v, stream=stream)

    def step(self, stream=None):
        """The whole step in one call: the new tokens' cache write, then the
        forward pass (pka_paged_attn_step)."""
        s = self.spec
        pka.pka_paged_attn_step(self.q, self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache,
                                self.block_table, self.qsl, self.seq_lens, *self.counts, s.scale, s.context_chunk,
                                self.max_query_len, self.max_seq_len, self.out, self.lse, self.workspace,
                                kv_scales=self.kv_scales, stream=stream)

    def step_separate(self, stream=None):
        """The same step as two calls: pka_cache_write(_fp8), then the forward."""
        self.cache_write(stream)
        self.forward(stream)

    def error_word(self) -> int:
        return pka.pka_get_error(self.workspace)


class UnorderedBatch:
    """A DeviceBatch whose requests arrive in another order: user request i is
    batch request perm[i]. A step does what a server does with such a batch:
    the token and request rows are gathered into [decode : extend : prefill]
    order (pka_batch_order's maps, computed once on the host from the
    lengths), cache write and forward run on the ordered rows, and out / lse
    are gathered back into the user's order (out_u, lse_u)."""

    def __init__(self, db: DeviceBatch, perm):
        b, dev = db.batch, db.device
        qsl0 = np.asarray(b.query_start_loc, dtype=np.int64)
        qlen = np.diff(qsl0).astype(np.int32)
        ctx = (np.asarray(b.seq_lens, dtype=np.int64) - qlen).astype(np.int32)
        perm = np.asarray(perm, dtype=np.int64)
        self.tok_u = np.concatenate([np.arange(qsl0[r], qsl0[r + 1]) for r in perm])
        idx = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
        sel = lambda t, a: None if t is None else t.index_select(0, idx(a).long()).contiguous()
        self.db = db
        # the rows as the user hands them over (set up once, outside the step)
        self.q_u, self.k_u, self.v_u = sel(db.q, self.tok_u), sel(db.k_new, self.tok_u), sel(db.v_new, self.tok_u)
        self.slot_u = sel(db.slot_mapping, self.tok_u)
        self.seq_u, self.bt_u = sel(db.seq_lens, perm), sel(db.block_table, perm)
        order, qsl_o, src, dst, counts = pka.pka_batch_order(qlen[perm], ctx[perm])
        self.counts = [int(c) for c in counts]
        self.src, self.dst, self.order, self.qsl_o = idx(src), idx(dst), idx(order), idx(qsl_o)
        empty = lambda t: None if t is None else torch.empty_like(t)
        self.q_o, self.k_o, self.v_o, self.slot_o = empty(self.q_u), empty(self.k_u), empty(self.v_u), empty(self.slot_u)
        self.seq_o, self.bt_o = empty(self.seq_u), empty(self.bt_u)
        self.out_o, self.lse_o = torch.empty_like(db.out), torch.empty_like(db.lse)
        self.out_u, self.lse_u = torch.empty_like(db.out), torch.empty_like(db.lse)
        rows = lambda t: 0 if t is None else t.numel() * t.element_size()
        # bytes the gathers read and write per step
        self.gather_bytes = 2 * sum(rows(t) for t in (self.q_u, self.k_u, self.v_u, self.slot_u, self.seq_u,
                                                       self.bt_u, self.out_o, self.lse_o))
        torch.cuda.synchronize()

    def step(self, stream=None):
        g = pka.pka_gather_rows
        col = lambda t: t.view(-1, 1)
        g(self.q_o, self.q_u, self.src, stream=stream)
        g(self.k_o, self.k_u, self.src, stream=stream)
        if self.v_u is not None:
            g(self.v_o, self.v_u, self.src, stream=stream)
        g(col(self.slot_o), col(self.slot_u), self.src, stream=stream)
        g(col(self.seq_o), col(self.seq_u), self.order, stream=stream)
        g(self.bt_o, self.bt_u, self.order, stream=stream)
        db, s = self.db, self.db.spec
        pka.pka_cache_write(self.k_o, self.v_o, self.slot_o, db.k_cache, db.v_cache, stream=stream)
        pka.pka_paged_attn_forward(self.q_o, self.k_o, self.v_o, db.k_cache, db.v_cache, self.bt_o, self.qsl_o,
                                   self.seq_o, self.counts[0], self.counts[1], self.counts[2], s.scale,
                                   s.context_chunk, db.max_query_len, db.max_seq_len, self.out_o, self.lse_o,
                                   db.workspace, head_dim_v=s.head_dim_v, stream=stream)
        g(self.out_u, self.out_o, self.dst, stream=stream)
        g(self.lse_u, self.lse_o, self.dst, stream=stream)

    def error_word(self) -> int:
        return self.db.error_word()
