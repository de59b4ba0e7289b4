"""Planted mistakes in copies of the page-append restatement: each must fail a pin.

The mistakes are written into the source of oracle/append_ref.py's append_kv
(gather_tokens is left alone), the copy is loaded as a module, and the pins of
tests/test_append_ref.py are run against it.
"""
import inspect
import types

import pytest

import oracle.append_ref as original
from tests import test_append_ref as pins

MUTANTS = {
    "wrong slot": ("k[page, t % page_size] = k_new[i]", "k[page, (t + 1) % page_size] = k_new[i]"),
    "previous request's pages": ("page = int(kv_indices[int(kv_indptr[b]) + t // page_size])",
                                 "page = int(kv_indices[int(kv_indptr[max(b - 1, 0)]) + t // page_size])"),
    "past-the-end token kept": ("t >= lengths[b]", "t > lengths[b]"),
    "V written with K": ("v[page, t % page_size] = v_new[i]", "v[page, t % page_size] = k_new[i]"),
    "page index from the slot": ("+ t // page_size])", "+ t % page_size])"),
    "HND: slot and head swapped": ("k[page, :, t % page_size] = k_new[i]",
                                   "k[page, t % page_size, :] = k_new[i]"),
    "HND: slot from the page index": ("k[page, :, t % page_size] = k_new[i]",
                                      "k[page, :, t // page_size] = k_new[i]"),
    "HND: page size from the head axis": ("page_size = k.shape[2] if layout",
                                          "page_size = k.shape[1] if layout"),
}

PINS = [pins.test_appended_rows_read_back_and_others_are_untouched,
        pins.test_append_order_does_not_matter_and_out_of_range_is_skipped,
        pins.test_appended_token_is_what_its_request_attends_to,
        pins.test_hnd_append_is_the_transpose_of_nhd_append]


def _mutated(old, new):
    src = inspect.getsource(original)
    body = src[src.index("def append_kv("):src.index("def gather_tokens(")]
    assert body.count(old) == 1, old
    src = src.replace(body, body.replace(old, new))
    mod = types.ModuleType("append_ref_mutant")
    exec(compile(src, "append_ref_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_planted_mistake_fails_a_pin(name, monkeypatch):
    monkeypatch.setattr(pins, "append_ref", _mutated(*MUTANTS[name]))
    failed = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failed += 1
    assert failed >= 1, name


def test_the_unmutated_copy_passes_every_pin(monkeypatch):
    monkeypatch.setattr(pins, "append_ref", _mutated("t >= lengths[b]", "t >= lengths[b]"))
    for pin in PINS:
        pin()
