"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, swaps it in, and checks that at least
one pin from test_oracle_pins fails. The committed oracle is never modified.
"""
import os
import shutil
import subprocess

import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pka_oracle.c")

MUTANTS = {
    "gqa_head_modulo": ("int g = h / G;", "int g = h % J->num_kv_heads;"),
    "scale_dropped": ("s *= J->scale;", "s *= 1.0;"),
    "causal_off_by_one": ("int64_t j0 = 0, j1 = p + 1;", "int64_t j0 = 0, j1 = p;"),
    "causal_top_left": ("int64_t p = ctx + (t - J->qsl[r]);", "int64_t p = (t - J->qsl[r]);"),
    "lse_base2": ("J->lse[i] = m + log(l);", "J->lse[i] = m + log2(l);"),
    "lse_without_max": ("J->lse[i] = m + log(l);", "J->lse[i] = log(l);"),
    "merge_weights_swapped": ("o[x] = (wa * oa[x] + wb * ob[x]) / (wa + wb);",
                              "o[x] = (wb * oa[x] + wa * ob[x]) / (wa + wb);"),
    "key_offset_shifted": ("* bs + j % bs) * d;\n            double s", "* bs + (j + 1) % bs) * d;\n            double s"),
    "cache_write_offset": ("int64_t off = slot % block_size;", "int64_t off = (slot + 1) % block_size;"),
}

PIN_CALLS = [
    lambda: [pins.test_oracle_matches_sdpa(s) for s in pins.SMALL_SPECS],
    pins.test_decode_sees_its_own_key,
    pins.test_single_key_closed_form,
    pins.test_two_key_closed_form,
    lambda: [pins.test_chunked_context_merge_equals_plain(c) for c in (7, 32)],
    pins.test_merge_closed_forms,
    pins.test_cache_write_round_trip_and_untouched_slots,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run([os.environ.get("CC", "gcc"), "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    str(mut), "-o", str(so), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.bind(str(so)))
    caught = 0
    for call in PIN_CALLS:
        try:
            call()
        except (AssertionError, ValueError):
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake {name!r}"
