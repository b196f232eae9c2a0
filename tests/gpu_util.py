"""Helpers for the GPU parity tests: run a seeded batch through the C ABI and
compare with the float64 oracle on the same inputs."""
import numpy as np

import oracle
from paged_kv_attention_07_gb300 import workloads as W

# bf16 output after fp32 accumulation; LSE in fp32 (natural log).
OUT_ATOL = 2e-2
LSE_ATOL = 1e-3


def run_gpu(batch, values_on_device_seed=None):
    import torch
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    db = DeviceBatch(batch, values_on_device_seed=values_on_device_seed)
    db.step()
    torch.cuda.synchronize()
    assert db.canaries_intact(), "a kernel wrote past out, lse or the workspace"
    err = db.error_word()
    dv = batch.spec.head_dim_v
    out = db.out.float().cpu().numpy().reshape(-1, dv)
    lse = db.lse.cpu().numpy().reshape(-1)
    return out, lse, err, db


def compare(batch, out, lse, rows=None, nthreads=None):
    ref_o, ref_l = oracle.batch_reference(batch, rows=rows, nthreads=nthreads)
    if rows is not None:
        out, lse = out[rows], lse[rows]
    assert np.isfinite(out).all(), "non-finite output"
    assert np.isfinite(lse).all(), "non-finite lse"
    eo = np.abs(out.astype(np.float64) - ref_o)
    el = np.abs(lse.astype(np.float64) - ref_l)
    worst = np.unravel_index(np.argmax(eo), eo.shape)
    assert eo.max() <= OUT_ATOL, f"out max abs err {eo.max():.3e} at row {worst[0]} (limit {OUT_ATOL})"
    assert el.max() <= LSE_ATOL, f"lse max abs err {el.max():.3e} at row {int(np.argmax(el))} (limit {LSE_ATOL})"
    return float(eo.max()), float(el.max())


def check_batch(batch, rows=None):
    out, lse, err, db = run_gpu(batch)
    assert err == 0, f"device error word 0x{err:x}"
    return compare(batch, out, lse, rows=rows)


def sample_rows(batch, n, seed=0, all_decodes=True):
    """Every decode row, the first and last token of every request (all heads)
    and a seeded sample of other (token, head) rows; flattened t * Hq + h."""
    spec = batch.spec
    Hq = spec.num_q_heads
    T = spec.num_tokens
    qsl = batch.query_start_loc
    toks = set()
    for r in range(spec.num_reqs):
        toks.add(int(qsl[r]))
        toks.add(int(qsl[r + 1]) - 1)
    if all_decodes:
        toks.update(range(spec.num_decodes))
    rows = {t * Hq + h for t in toks for h in range(Hq)}
    rng = np.random.default_rng(seed)
    extra = rng.choice(T * Hq, size=min(n, T * Hq), replace=False)
    rows.update(int(x) for x in extra)
    return np.array(sorted(rows), dtype=np.int64)
