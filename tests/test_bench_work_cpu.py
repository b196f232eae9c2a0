"""The work bench.py divides by (the roofline numerator): bytes and flops of a
step counted from the batch itself, against a brute-force count of the
visible (query, key) pairs and of the keys each decode reads. No GPU."""
import importlib.util
import os

import pytest

from paged_kv_attention_07_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def brute_force_pairs(spec, first, last):
    """(query, key) pairs with key <= ctx + i, requests [first, last)."""
    n = 0
    for r in range(first, last):
        q, c = spec.qlen[r], spec.ctx[r]
        for i in range(q):
            n += sum(1 for j in range(c + q) if j <= c + i)
    return n


@pytest.mark.parametrize("spec", [
    W.spec_tiny(),
    W.spec_custom("w", ctx=[5, 300, 17, 0, 0], qlen=[1, 1, 40, 7, 64], num_decodes=2, num_extends=1,
                  num_prefills=2, Hq=8, Hkv=2, d=64, dv=64, bs=16),
    W.spec_custom("wm", ctx=[100, 7], qlen=[1, 1], num_decodes=2, num_extends=0, num_prefills=0, Hq=128,
                  Hkv=1, d=576, dv=512, bs=64, mla=True),
], ids=lambda s: s.name)
def test_work_matches_brute_force(bench, spec):
    w = bench.algorithmic_work(spec)
    nd, ne = spec.num_decodes, spec.num_extends
    Hq, Hkv, d, dv = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.head_dim_v
    per_pair = Hq * 2 * (d + dv)  # q.k and p.v multiply-adds per query head
    assert w["ext_flops"] == brute_force_pairs(spec, nd, nd + ne) * per_pair
    assert w["pre_flops"] == brute_force_pairs(spec, nd + ne, spec.num_reqs) * per_pair
    dec_keys = brute_force_pairs(spec, 0, nd)  # a decode's one query sees all its keys
    assert dec_keys == sum(spec.seq_lens[:nd])
    key_bytes = d * 2 if spec.mla else Hkv * (d + dv) * 2  # MLA: one latent row per key
    assert w["dec_bytes"] == dec_keys * key_bytes
    assert w["dec_flops"] == dec_keys * per_pair
    assert w["tokens"] == sum(spec.qlen)
