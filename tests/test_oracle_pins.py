"""Pins of the CPU oracle against what the SplitZip pages and plain mathematics fix.

Each check ties the oracle to something other than itself:
  * hand-worked golden payloads (tests/golden/*.json, each with its derivation);
  * the closed-form facts about all 65,536 BF16 bit patterns;
  * library routines (numpy.bincount for the histogram, a stable numpy argsort
    for the Top-16 order) and brute force on tiny inputs;
  * invariants the method guarantees (bitwise round trip, escape count =
    n - top_count, escape-stream order, code 0 at escapes, section sizes);
  * the ratio the pages print for weight-like data (0.750, "splitzip_codec.py"
    module docstring "Validated ... measured ratio 0.750").
"""
from __future__ import annotations

import numpy as np
import pytest

from weight_compression_codec_gb300 import inputs


def _bytes_hex(h: str) -> np.ndarray:
    return np.frombuffer(bytes.fromhex(h), dtype=np.uint8)


def _escape_streams(payload: np.ndarray, m):
    e = m.n_esc
    cid = payload[m.off_cid:m.off_cid + 4 * e].view("<i4")
    lpos = payload[m.off_lpos:m.off_lpos + 2 * e].view("<u2")
    ev = payload[m.off_ev:m.off_ev + e]
    return cid, lpos, ev


def _meta_dict(m):
    return {k: getattr(m, k) for k in ("n", "n_pairs", "n_esc", "comp_bytes", "off_pk", "off_sm",
                                       "off_cid", "off_lpos", "off_ev", "chunk_size")}


# --------------------------------------------------------------------------- golden payloads


def test_golden_small_no_escape(oracle, golden):
    g = golden("small_no_escape.json")
    x = np.array([int(h, 16) for h in g["x_hex"]], dtype=np.uint16)
    cb = oracle.calibrate(x)
    assert list(cb.dec_lut) == g["dec_lut"]
    assert cb.n_top == g["n_top"] and cb.top_count == g["top_count"] and cb.coverage == g["coverage"]
    payload, m = oracle.encode(x, cb)
    assert _meta_dict(m) == g["meta"]
    assert payload.tobytes() == bytes.fromhex(g["payload_hex"])
    # the other nibble order (element 2i high), as the page's own torch codec writes it
    p1 = oracle.to_p1_nibble_order(payload, m)
    assert p1.tobytes() == bytes.fromhex(g["payload_p1_nibble_order_hex"])
    # decode of the hand-written payload, independent of the encoder
    out = oracle.decode(_bytes_hex(g["payload_hex"]), m, np.array(g["dec_lut"], dtype=np.uint8))
    assert np.array_equal(out, x)


def _three_chunk_input(g) -> np.ndarray:
    x = np.full(g["n"], int(g["base_hex"], 16), dtype=np.uint16)
    for j in range(15):
        x[10 + j] = ((0x70 + j) << 7) | j
        x[1500 + j] = 0x8000 | ((0x70 + j) << 7) | (127 - j)
    x[5], x[1030], x[2050] = 0x7F80, 0x0081, 0xC801
    return x


def test_golden_three_chunk_escapes(oracle, golden):
    g = golden("three_chunk_escapes.json")
    x = _three_chunk_input(g)
    cb = oracle.calibrate(x)
    assert list(cb.dec_lut) == g["dec_lut"]
    assert cb.n_top == g["n_top"] and cb.top_count == g["top_count"]
    assert cb.coverage == g["coverage_num"] / g["coverage_den"]
    for v in g["escape_values"]:
        assert cb.enc_lut[v] == 16
    payload, m = oracle.encode(x, cb)
    assert _meta_dict(m) == g["meta"]
    expect = np.zeros(g["meta"]["comp_bytes"], dtype=np.uint8)
    for off, h in g["nonzero_runs_hex"]:
        b = _bytes_hex(h)
        expect[off:off + b.size] = b
    assert np.array_equal(payload, expect)
    p1 = oracle.to_p1_nibble_order(payload, m)
    expect_p1 = expect.copy()
    for off, h in g["p1_nibble_order_pk_runs_hex"]:
        b = _bytes_hex(h)
        expect_p1[off:off + b.size] = b
    assert np.array_equal(p1, expect_p1)
    assert np.array_equal(oracle.decode(expect, m, np.array(g["dec_lut"], dtype=np.uint8)), x)


def test_all_bit_patterns_closed_form(oracle, golden):
    g = golden("all_bit_patterns.json")
    x = inputs.all_bit_patterns()
    cb = oracle.calibrate(x)
    assert list(cb.dec_lut) == g["dec_lut"]
    assert cb.n_top == g["n_top"] and cb.top_count == g["top_count"] and cb.coverage == g["coverage"]
    payload, m = oracle.encode(x, cb)
    assert _meta_dict(m) == g["meta"]
    assert m.comp_bytes / (2 * m.n) == g["ratio"]
    cid, lpos, ev = _escape_streams(payload, m)
    for key, k in (("first_escape", 0), ("last_escape", m.n_esc - 1)):
        assert (int(cid[k]), int(lpos[k]), int(ev[k])) == tuple(g[key].values())
    elem = cid.astype(np.int64) * 1024 + lpos
    for k0, k1, first in g["escape_element_runs"]:
        assert np.array_equal(elem[k0:k1], np.arange(first, first + (k1 - k0)))
    pk = payload[:m.n_pairs]
    b = np.arange(m.n_pairs)
    want = np.zeros(m.n_pairs, dtype=np.uint8)
    lo = b < 1024
    want[lo] = 0x11 * (b[lo] >> 6)
    hi = (b >= 16384) & (b < 17408)
    want[hi] = 0x11 * ((b[hi] - 16384) >> 6)
    assert np.array_equal(pk, want)
    assert np.array_equal(oracle.decode(payload, m, cb.dec_lut), x)


def test_empty_tensor(oracle):
    x = np.zeros(0, dtype=np.uint16)
    cb = oracle.calibrate(x)
    assert cb.n_top == 0 and cb.top_count == 0 and cb.coverage == 1.0
    assert list(cb.enc_lut) == [16] * 256 and list(cb.dec_lut) == [0] * 16
    payload, m = oracle.encode(x, cb)
    assert payload.size == 0 and m.comp_bytes == 0 and m.n_esc == 0
    assert oracle.decode(payload, m, cb.dec_lut).size == 0


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 9, 1023, 1024, 1025, 2047, 2049, 4095, 4097])
def test_small_sizes_round_trip_and_layout(oracle, n):
    r = np.random.default_rng(n)
    x = r.integers(0, 65536, size=n, dtype=np.uint16)
    cb = oracle.calibrate(x)
    payload, m = oracle.encode(x, cb)
    # the payload size: the aligned sum of ceil(n/2) + n + 7 * n_esc; pads are below 4 bytes each
    raw = (n + 1) // 2 + n + 7 * m.n_esc
    assert 0 <= m.comp_bytes - raw <= 3 + 3 + 3
    for off in (m.off_sm, m.off_cid, m.off_lpos, m.off_ev):
        assert off % 4 == 0 or off == m.off_lpos  # off_lpos = off_cid + 4e is aligned too
    assert m.off_lpos % 4 == 0
    assert np.array_equal(oracle.decode(payload, m, cb.dec_lut), x)


# --------------------------------------------------------------------------- histogram and select


@pytest.mark.parametrize("maker", ["gauss", "uniform_bits", "edge"])
def test_histogram_equals_bincount(oracle, maker):
    n = 200_003
    if maker == "gauss":
        x = inputs.gaussian(n, 0.02, seed=7)
    elif maker == "uniform_bits":
        x = np.random.default_rng(3).integers(0, 65536, size=n, dtype=np.uint16)
    else:
        x = inputs.edge_case(n, seed=3)
    expo = (x.astype(np.uint32) >> 7) & 0xFF
    assert np.array_equal(oracle.histogram(x), np.bincount(expo, minlength=256).astype(np.uint64))


def test_histogram_brute_force_tiny(oracle):
    r = np.random.default_rng(11)
    for n in (0, 1, 2, 17, 300):
        x = r.integers(0, 65536, size=n, dtype=np.uint16)
        h = [0] * 256
        for v in x.tolist():
            h[(v // 128) % 256] += 1
        assert oracle.histogram(x).tolist() == h


def _stable_top(h: np.ndarray) -> list[int]:
    order = np.argsort(-h.astype(np.float64), kind="stable")
    return [int(v) for v in order if h[v] > 0][:16]


def test_select_equals_stable_argsort(oracle):
    r = np.random.default_rng(5)
    cases = []
    for _ in range(200):
        k = int(r.integers(0, 40))
        h = np.zeros(256, dtype=np.uint64)
        vals = r.choice(256, size=k, replace=False)
        h[vals] = r.integers(1, 6, size=k)  # small counts: many ties
        cases.append(h)
    cases.append(np.ones(256, dtype=np.uint64))
    cases.append(np.zeros(256, dtype=np.uint64))
    for h in cases:
        n = int(h.sum())
        cb = oracle.select(h, n)
        top = _stable_top(h)
        assert cb.n_top == len(top)
        assert list(cb.dec_lut[:len(top)]) == top and all(v == 0 for v in cb.dec_lut[len(top):])
        enc = np.full(256, 16, dtype=np.uint8)
        enc[top] = np.arange(len(top))
        assert np.array_equal(cb.enc_lut, enc)
        assert cb.top_count == int(h[top].sum())
        assert cb.coverage == (int(h[top].sum()) / n if n else 1.0)


# --------------------------------------------------------------------------- invariants on workloads


def _check_invariants(oracle, x, cb=None):
    cb = cb if cb is not None else oracle.calibrate(x)
    payload, m = oracle.encode(x, cb)
    expo = (x.astype(np.uint32) >> 7) & 0xFF
    in_top = np.zeros(256, dtype=bool)
    in_top[cb.dec_lut[:cb.n_top]] = True
    esc_mask = ~in_top[expo]
    assert m.n_esc == int(esc_mask.sum())
    cid, lpos, ev = _escape_streams(payload, m)
    idx = cid.astype(np.int64) * 1024 + lpos.astype(np.int64)
    assert np.array_equal(idx, np.nonzero(esc_mask)[0])  # ascending element order
    assert np.all(lpos < 1024)
    assert np.array_equal(ev, expo[esc_mask].astype(np.uint8))
    pk = payload[:m.n_pairs]
    nib = np.empty(2 * m.n_pairs, dtype=np.uint8)
    nib[0::2] = pk & 0xF
    nib[1::2] = pk >> 4
    assert np.all(nib[:m.n][esc_mask] == 0)
    if m.n % 2:
        assert nib[m.n] == 0
    # every pad byte is zero
    for a, b in ((m.n_pairs, m.off_sm), (m.off_sm + m.n, m.off_cid), (m.off_lpos + 2 * m.n_esc, m.off_ev)):
        assert np.all(payload[a:b] == 0)
    assert np.array_equal(oracle.decode(payload, m, cb.dec_lut), x)
    return payload, m, cb


def test_invariants_gaussian_and_ratio(oracle):
    x = inputs.gaussian(1 << 20, 0.02, seed=0)
    payload, m, cb = _check_invariants(oracle, x)
    assert m.n_esc == m.n - cb.top_count
    ratio = m.comp_bytes / (2 * m.n)
    assert abs(ratio - 0.750) < 0.0015  # the pages: "measured ratio 0.750 on gaussian/weight-like data"


def test_invariants_edge_case_specials(oracle):
    x = inputs.edge_case(300_007, seed=1)
    payload, m, cb = _check_invariants(oracle, x)
    assert cb.coverage < 0.5 and m.n_esc > m.n // 2
    for special in (0x0000, 0x8000, 0x7F80, 0xFF80):
        assert np.any(x == special)
    nan = ((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0)
    sub = ((x & 0x7F80) == 0) & ((x & 0x7F) != 0)
    assert nan.mean() > 0.005 and sub.mean() > 0.04


def test_codebook_from_other_data(oracle):
    """Encode must hold for any codebook, whatever the escape count."""
    x = inputs.gaussian(50_001, 1.0, seed=2)
    cb_other = oracle.calibrate(inputs.gaussian(4_096, 1e-3, seed=3))
    _check_invariants(oracle, x, cb_other)
    cb_few = oracle.calibrate(np.array([0x3F80, 0x3F80, 0x0000], dtype=np.uint16))
    payload, m, _ = _check_invariants(oracle, x, cb_few)
    assert m.n_esc > 0.5 * m.n  # only |x| in [1, 2) and zeros are covered


def test_kv_and_weight_recipes_small(oracle):
    for x in inputs.kv_cache(layers=1, tokens=64)[:2]:
        _check_invariants(oracle, x)
    small = inputs.weight_tensor(0, pairs=2, d_model=64, d_ff=224)
    last = inputs.weight_tensor(3, pairs=2, d_model=64, d_ff=224)
    _check_invariants(oracle, small)
    _, m, cb = _check_invariants(oracle, last)
    assert cb.coverage < 0.99  # the broad-exponent tensor of the weight recipe
    for blk in inputs.paged_kv(count=4):
        _check_invariants(oracle, blk)


# --------------------------------------------------------------------------- decode rejects malformed metas


def test_decode_rejects_bad_meta(oracle):
    import dataclasses

    x = inputs.edge_case(5000, seed=4)
    cb = oracle.calibrate(x)
    payload, m = oracle.encode(x, cb)
    assert m.n_esc > 0
    for field, delta in (("off_sm", 4), ("off_cid", -4), ("off_ev", 4), ("comp_bytes", 1), ("chunk_size", 1),
                         ("n_pairs", 1)):
        bad = dataclasses.replace(m, **{field: getattr(m, field) + delta})
        with pytest.raises(ValueError):
            oracle.decode(np.concatenate([payload, np.zeros(16, np.uint8)]), bad, cb.dec_lut)
    broken = payload.copy()
    broken[m.off_lpos:m.off_lpos + 2] = np.frombuffer(np.uint16(1024).tobytes(), np.uint8)
    with pytest.raises(ValueError):
        oracle.decode(broken, m, cb.dec_lut)


# ---------------------------------------------------------------------------- coverage gate


def test_gate_is_strictly_below_and_negative_gates_nothing(oracle):
    assert oracle.gated(0.98, 0.99) and not oracle.gated(0.99, 0.99) and not oracle.gated(1.0, 0.99)
    assert not oracle.gated(0.0, -1.0) and oracle.gated(0.0, 0.5)


def test_gate_report_by_hand(oracle):
    # three tensors: a Gaussian one (coverage ~1), the all-bit-patterns tensor
    # (coverage 1/16, payload 4.03 x raw) and an empty one (coverage 1.0)
    from weight_compression_codec_gb300 import inputs

    xs = [inputs.gaussian(10_000, 0.02, seed=3), inputs.all_bit_patterns(), np.zeros(0, np.uint16)]
    cbs = [oracle.calibrate(x) for x in xs]
    metas = [oracle.encode(x, cb)[1] for x, cb in zip(xs, cbs)]
    assert cbs[1].coverage == 0.0625 and metas[1].comp_bytes == 528_384
    r = oracle.gate_report([x.size for x in xs], [cb.coverage for cb in cbs], metas, 0.99)
    assert r["tensors_gated"] == 1 and r["raw_bytes_gated"] == 2 * 65_536
    assert r["tensors_encoded"] == 2 and r["raw_bytes_encoded"] == 20_000
    assert r["payload_bytes"] == metas[0].comp_bytes + 0 and r["escapes"] == metas[0].n_esc
    assert r["tensors_expanded"] == 0
    # without the gate the all-bit-patterns tensor is encoded and expands
    r = oracle.gate_report([x.size for x in xs], [cb.coverage for cb in cbs], metas, -1.0)
    assert r["tensors_gated"] == 0 and r["tensors_expanded"] == 1 and r["escapes"] == metas[0].n_esc + 61_440
    assert r["payload_bytes"] == metas[0].comp_bytes + 528_384


# ---------------------------------------------------------------------------- slot decode


def test_decode_slot_golden_payload_with_garbage_after_it(oracle, golden):
    # "splitzip_codec.py" GpuSplitZipDecoder: the payload sits in the slot's
    # leading comp_bytes, the rest of the raw-size slot is arbitrary, and the
    # weight is decoded over the whole slot
    g = golden("three_chunk_escapes.json")
    x = _three_chunk_input(g)
    expect = np.zeros(g["meta"]["comp_bytes"], dtype=np.uint8)
    for off, h in g["nonzero_runs_hex"]:
        b = _bytes_hex(h)
        expect[off:off + b.size] = b
    m = oracle.layout(g["n"], g["meta"]["n_esc"], 1.0)
    slot = np.random.default_rng(5).integers(0, 256, 2 * x.size, dtype=np.uint8)
    slot[:expect.size] = expect
    out = oracle.decode_slot(slot, m, np.array(g["dec_lut"], dtype=np.uint8))
    assert out is slot and np.array_equal(slot.view(np.uint16), x)


def test_decode_slot_needs_the_copy_aside(oracle):
    # decoding element by element straight over the slot would overwrite pk,
    # sm and escape bytes before they are read; the oracle's result must not
    # depend on that (it equals the out-of-place decode)
    x = inputs.gaussian(40_000, 0.02, seed=9)
    x[::997] = 0x7F80  # a few escapes
    cb = oracle.calibrate(x)
    payload, m = oracle.encode(x, cb)
    assert m.n_esc > 0 and m.comp_bytes <= 2 * x.size
    slot = np.zeros(2 * x.size, dtype=np.uint8)
    slot[:m.comp_bytes] = payload
    naive = slot.copy()
    nv = naive.view(np.uint16)
    for i in range(x.size):  # no stash: element i is written before later elements are read
        code = (naive[i // 2] >> (4 * (i % 2))) & 15
        s = int(naive[m.off_sm + i])
        nv[i] = ((s & 0x80) << 8) | (int(cb.dec_lut[code]) << 7) | (s & 0x7F)
    assert not np.array_equal(nv, x)
    oracle.decode_slot(slot, m, cb.dec_lut)
    assert np.array_equal(slot.view(np.uint16), x)


def test_decode_slot_rejects_a_payload_larger_than_the_slot(oracle):
    x = np.array([0x3F80], dtype=np.uint16)  # n = 1: comp_bytes = 8 > 2
    cb = oracle.calibrate(x)
    payload, m = oracle.encode(x, cb)
    assert m.comp_bytes == 8
    with pytest.raises(ValueError):
        oracle.decode_slot(np.zeros(2, np.uint8), m, cb.dec_lut)
    with pytest.raises(ValueError):
        oracle.decode_slot(np.zeros(8, np.uint8), m, cb.dec_lut)  # not a raw-size slot
