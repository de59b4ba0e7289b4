"""Planted mistakes in a copy of the oracle must fail at least one pin.

Each mutant is a one-line edit of ``oracle/ref_attn.c`` (a dropped term, a
wrong index or sign, a swapped operand, a finite -inf sentinel), compiled into
a temporary library and run through every check in ``tests/pins.py``.  All
edits keep memory accesses in bounds.
"""
import os

import pytest

import oracle
from tests import pins

MUTANTS = {
    "gqa_head_modulo": ("int kvh = h / group;", "int kvh = h % num_kv_heads;"),
    "slot_off_by_one": ("int64_t slot = t % page_size;\n      int64_t k_base",
                        "int64_t slot = (t + 1) % page_size;\n      int64_t k_base"),
    "hnd_instead_of_nhd": (
        "  return ((page * page_size + slot) * num_kv_heads + kvh) * head_dim;",
        "  return ((page * num_kv_heads + kvh) * page_size + slot) * head_dim;"),
    "hnd_head_and_slot_swapped": (
        "    return ((page * num_kv_heads + kvh) * page_size + slot) * head_dim;",
        "    return ((page * page_size + slot) * num_kv_heads + kvh) * head_dim;"),
    "scale_dropped": ("s[t] = sm_scale * dot;", "s[t] = dot;"),
    "lse_without_max": ("lse[i] = m + log(z);", "lse[i] = log(z);"),
    "finite_sentinel": ("double m = -INFINITY;\n    for (int64_t t",
                        "double m = -50000.0;\n    for (int64_t t"),
    "max_as_min": ("if (s[t] > m) m = s[t];", "if (s[t] < m || m == -INFINITY) m = s[t];"),
    "unnormalised": ("for (int d = 0; d < head_dim; ++d) o[d] /= z;", ""),
    "value_from_keys": ("o[d] += w * element(v_pages, dtype, v_base + d);",
                        "o[d] += w * element(k_pages, dtype, v_base + d);"),
    "f16_bias": ("expo - 25", "expo - 24"),
    "bf16_shift": ("(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    "merge_wrong_weight": ("double wb = exp(s_b[i] - m);", "double wb = exp(s_a[i] - m);"),
    "merge_no_normaliser": (
        "v[d] = (wa * v_a[i * head_dim + d] + wb * v_b[i * head_dim + d]) / z;",
        "v[d] = wa * v_a[i * head_dim + d] + wb * v_b[i * head_dim + d];"),
    "merge_lse_sign": ("s_out[i] = m + log(z);", "s_out[i] = m - log(z);"),
    "merge_no_empty_rule": ("if (s_a[i] == -INFINITY && s_b[i] == -INFINITY) {",
                            "if (0) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, "mutation site not unique: %s" % name
    mutant_src = tmp_path / ("mutant_%s.c" % name)
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant_src),
                                str(tmp_path / ("libmutant_%s.so" % name)))
    failed = pins.failing_checks(oracle.Oracle(lib))
    assert failed, "mutant %s passes every pin" % name


def test_committed_oracle_passes_all():
    assert pins.failing_checks(oracle.default()) == []
    assert os.path.exists(oracle.SOURCE)
