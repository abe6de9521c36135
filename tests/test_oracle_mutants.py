"""The oracle's pins are sensitive: each plausible mistake planted in a copy of
the oracle (on the CPU, in a scratch directory) makes at least one pin fail.

The real oracle source is never modified; each mutant is a textual edit of a
copy, compiled with the oracle's own build step into a temporary library.
"""
from __future__ import annotations

import shutil

import pytest

import oracle as oracle_pkg
from oracle import build as oracle_build

import test_oracle_pins as pins

# (name, old text, new text, replace every occurrence)
MUTANTS = [
    ("nibble order swapped", "(4 * (i % 2))", "(4 * (1 - i % 2))", True),
    ("ties by descending value", "hist[order[j]] < hist[v]", "hist[order[j]] <= hist[v]", False),
    ("sign bit dropped from sm", "(((x >> 8) & 0x80u) | (x & 0x7Fu))", "((x & 0x7Fu))", False),
    ("exponent taken from bits 8..15", "((x >> 7) & 0xFFu)", "((x >> 8) & 0xFFu)", False),
    ("align4 rounds too far", "(v + 3u)", "(v + 4u)", False),
    ("only 15 codes", "distinct < 16u ? distinct : 16u", "distinct < 15u ? distinct : 15u", False),
    ("chunk of 512", "(uint32_t)(i / SZO_CHUNK)", "(uint32_t)(i / 512u)", False),
    ("local_pos modulo 512", "(uint32_t)(i % SZO_CHUNK)", "(uint32_t)(i % 512u)", False),
    ("coverage over n+1", "(double)top_count / (double)n", "(double)top_count / (double)(n + 1)", False),
    ("pads not zeroed", "memset(out, 0, m->comp_bytes)", "memset(out, 0x5A, m->comp_bytes)", False),
    ("no pad before esc_val", "m->off_ev = align4(m->off_lpos + 2 * n_esc)", "m->off_ev = m->off_lpos + 2 * n_esc", False),
    ("esc_val holds the code", "out[m->off_ev + k] = exp;", "out[m->off_ev + k] = code;", False),
    ("escape nibble kept as 15", "(uint8_t)(code & 0x0Fu)", "(uint8_t)(code == SZO_ESCAPE ? 15u : code)", False),
    ("merge shifts exponent by 8", "((uint32_t)exp << 7)", "((uint32_t)exp << 8)", False),
    ("escape patched one element late", "cid * SZO_CHUNK + pos;", "cid * SZO_CHUNK + pos + 1;", False),
    ("escape patch drops the sign", "out[idx] = merge(payload[m->off_sm + idx], payload[m->off_ev + k]);",
     "out[idx] = merge(payload[m->off_sm + idx] & 0x7Fu, payload[m->off_ev + k]);", False),
    ("dense decode reads the wrong sm byte", "out[i] = merge(payload[m->off_sm + i], exp);",
     "out[i] = merge(payload[m->off_sm + (i ^ 1) % (m->n ? m->n : 1)], exp);", False),
    ("top_count misses the last code", "top_count += hist[value];", "if (code + 1 < top) top_count += hist[value];", False),
]


class _Shim:
    """The oracle package's API bound to a mutant library."""

    def __init__(self, lib):
        self._lib = lib
        self.CHUNK = oracle_pkg.CHUNK

    def __getattr__(self, name):
        fn = getattr(oracle_pkg, name)
        return lambda *a, **k: fn(*a, lib=self._lib, **k)


PIN_TESTS = [
    lambda o, g: pins.test_golden_small_no_escape(o, g),
    lambda o, g: pins.test_golden_three_chunk_escapes(o, g),
    lambda o, g: pins.test_all_bit_patterns_closed_form(o, g),
    lambda o, g: pins.test_empty_tensor(o),
    lambda o, g: [pins.test_small_sizes_round_trip_and_layout(o, n) for n in (1, 3, 1025, 4097)],
    lambda o, g: pins.test_histogram_equals_bincount(o, "edge"),
    lambda o, g: pins.test_select_equals_stable_argsort(o),
    lambda o, g: pins.test_invariants_gaussian_and_ratio(o),
    lambda o, g: pins.test_invariants_edge_case_specials(o),
    lambda o, g: pins.test_codebook_from_other_data(o),
]


@pytest.mark.parametrize("name,old,new,everywhere", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, golden, name, old, new, everywhere):
    src = oracle_build.HERE / "sz_oracle.c"
    text = src.read_text()
    assert old in text, f"mutation anchor not found: {old!r}"
    mutated = text.replace(old, new) if everywhere else text.replace(old, new, 1)
    shutil.copy(oracle_build.HERE / "sz_oracle.h", tmp_path / "sz_oracle.h")
    (tmp_path / "sz_oracle.c").write_text(mutated)
    lib_path = oracle_build.build(force=True, sources=[tmp_path / "sz_oracle.c"], out=tmp_path / "libmut.so")
    shim = _Shim(oracle_pkg.load(lib_path))
    caught = 0
    for check in PIN_TESTS:
        try:
            check(shim, golden)
        except (AssertionError, ValueError, RuntimeError, IndexError):
            caught += 1
    assert caught >= 1, f"no pin caught the planted mistake: {name}"


def test_unmutated_copy_passes_every_pin(tmp_path, golden):
    shutil.copy(oracle_build.HERE / "sz_oracle.h", tmp_path / "sz_oracle.h")
    shutil.copy(oracle_build.HERE / "sz_oracle.c", tmp_path / "sz_oracle.c")
    lib_path = oracle_build.build(force=True, sources=[tmp_path / "sz_oracle.c"], out=tmp_path / "libcopy.so")
    shim = _Shim(oracle_pkg.load(lib_path))
    for check in PIN_TESTS:
        check(shim, golden)
