"""CPU-side checks of libsplitzip.so: it builds for sm_103a, loads, exports every
symbol include/splitzip.h declares, and its host-only calls (sizes, layout,
argument checks) behave -- no GPU needed, no kernel launched."""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B

HEADER = Path(__file__).resolve().parents[1] / "include" / "splitzip.h"


@pytest.fixture(scope="module")
def lib():
    sz.build()
    return B.lib()


def declared_symbols() -> list[str]:
    text = HEADER.read_text()
    return re.findall(r"SZ_API\s+[\w\s\*]+?\b(sz_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ("sz_calibrate", "sz_encode", "sz_decode", "sz_calibrate_many", "sz_encode_many",
                 "sz_decode_many", "sz_max_payload_bytes", "sz_workspace_flags"):
        assert must in names
    assert set(names) == set(B.SIGNATURES), "binding signatures and header declarations differ"


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.sz_version() == 1


def test_exports_are_only_the_abi(lib):
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", str(B.library_path())], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {s for s in exported if s.startswith("sz_")}
    assert ours == set(declared_symbols())


def test_struct_sizes_match_header(lib):
    assert ctypes.sizeof(B.SzCodebook) == 304 and ctypes.sizeof(B.SzMeta) == 96 and ctypes.sizeof(B.SzItem) == 64


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 1023, 1024, 1025, 8191, 8192, 8193, 65536, 100_000_003, 2**31, 2**32 - 1])
def test_layout_matches_oracle(lib, oracle, n):
    for e in sorted({0, 1, 3, n // 7, n}):
        if e > n:
            continue
        m = sz.sz_layout(n, e)
        o = oracle.layout(n, e)
        assert m.as_tuple() == o.as_tuple()
        assert sz.sz_payload_bytes(n, e) == o.comp_bytes
    assert sz.sz_max_payload_bytes(n) == oracle.layout(n, n).comp_bytes
    assert sz.sz_tiles(n) == (n + 8191) // 8192


def test_layout_rejects_bad_sizes(lib):
    m = B.SzMeta()
    assert lib.sz_layout(10, 11, ctypes.byref(m)) == B.SZ_ERR_ARG
    assert lib.sz_layout(2**32, 0, ctypes.byref(m)) == B.SZ_ERR_ARG
    assert lib.sz_layout(10, 0, None) == B.SZ_ERR_ARG


def test_items_prepare(lib):
    ns = [0, 5, 8192, 8193, 0, 1]
    arr = (B.SzItem * len(ns))()
    for i, n in enumerate(ns):
        arr[i].n = n
    total = ctypes.c_uint64()
    assert lib.sz_items_prepare(arr, len(ns), ctypes.byref(total)) == 0
    assert [arr[i].tile_begin for i in range(len(ns))] == [0, 0, 1, 2, 4, 4]
    assert total.value == 5


def test_workspace_sizes_monotone(lib):
    for f in (lambda c: lib.sz_calibrate_workspace_bytes(c),):
        assert f(1) <= f(2) <= f(100)
    assert lib.sz_encode_workspace_bytes(1, 10) < lib.sz_encode_workspace_bytes(1, 11)
    assert lib.sz_decode_workspace_bytes(1, 10) <= lib.sz_decode_workspace_bytes(1, 11)
    # encode staging holds local_pos and esc_val of every element of every tile
    assert lib.sz_encode_workspace_bytes(1, 100) >= 100 * 8192 * 3


def test_host_argument_checks_launch_nothing(lib):
    """Invalid arguments are rejected on the host before any CUDA call, so these
    run without a GPU."""
    ws = 4096  # fake aligned addresses: never dereferenced on these paths
    al = 1 << 20
    # null codebook / meta / data
    assert lib.sz_calibrate(al, 10, None, ws * 256, 1 << 20, None) == B.SZ_ERR_ARG
    assert lib.sz_calibrate(None, 10, al, ws * 256, 1 << 20, None) == B.SZ_ERR_ARG
    assert lib.sz_encode(al, 10, al, al, 1000, None, ws * 256, 1 << 20, None) == B.SZ_ERR_ARG
    assert lib.sz_decode(al, 1000, None, al, al, 10, ws * 256, 1 << 20, None) == B.SZ_ERR_ARG
    # misaligned pointers
    assert lib.sz_calibrate(al + 2, 10, al, ws * 256, 1 << 20, None) == B.SZ_ERR_ALIGN
    assert lib.sz_encode(al, 10, al + 8, al, 1000, al, ws * 256, 1 << 20, None) == B.SZ_ERR_ALIGN
    assert lib.sz_decode(al + 4, 1000, al, al, al, 10, ws * 256, 1 << 20, None) == B.SZ_ERR_ALIGN
    # too-large n
    assert lib.sz_calibrate(al, 2**32, al, ws * 256, 1 << 20, None) == B.SZ_ERR_ARG
    # capacity below the dense part of the layout
    assert lib.sz_encode(al, 1000, al, al, 1000, al, ws * 256, 1 << 30, None) == B.SZ_ERR_CAPACITY
    assert lib.sz_decode(al, 1000, al, al, al, 1000, ws * 256, 1 << 30, None) == B.SZ_ERR_CAPACITY
    # workspace missing / misaligned / too small
    assert lib.sz_calibrate(al, 10, al, None, 1 << 20, None) == B.SZ_ERR_WORKSPACE
    assert lib.sz_calibrate(al, 10, al, ws * 256 + 16, 1 << 20, None) == B.SZ_ERR_WORKSPACE
    assert lib.sz_encode(al, 10**6, al, al, 10**7, al, ws * 256, 1024, None) == B.SZ_ERR_WORKSPACE
    # *_many: count and table checks
    assert lib.sz_calibrate_many(al, 0, 1, ws * 256, 1 << 20, None) == B.SZ_ERR_ARG
    assert lib.sz_encode_many(None, 3, 1, ws * 256, 1 << 20, None) == B.SZ_ERR_ARG
    assert lib.sz_decode_many(al + 8, 3, 1, ws * 256, 1 << 20, None) == B.SZ_ERR_ALIGN
    assert lib.sz_decode_many(al, 70000, 1, ws * 256, 1 << 20, None) == B.SZ_ERR_ARG
    for s in range(8):
        assert lib.sz_strerror(s)


def test_python_binding_rejects_cpu_and_wrong_dtype(lib):
    import torch

    with pytest.raises(ValueError):
        sz.sz_calibrate(torch.zeros(8, dtype=torch.float32))
    with pytest.raises(ValueError):
        sz.sz_calibrate(torch.zeros(8, dtype=torch.bfloat16))  # not on a CUDA device


def test_meta_bytes_round_trip(lib, oracle):
    om = oracle.layout(12345, 67, 0.5)
    m = sz.meta_from_bytes(np.frombuffer(sz.meta_to_bytes(om), np.uint8))
    assert m.as_tuple() == om.as_tuple() and m.coverage == 0.5


def test_host_decode_planner_on_the_host():
    """sz_decode_many_host_scratch_bytes plans groups on the host only (the
    addresses below are never dereferenced)."""
    from weight_compression_codec_gb300 import binding as B

    lib = B.lib()
    n = 100_000
    layout = B.SzMeta()
    assert lib.sz_layout(n, 10, ctypes.byref(layout)) == 0
    comp = layout.comp_bytes
    count = 6
    items = (B.SzItem * count)()
    metas = (B.SzMeta * count)()
    base = 1 << 32
    for i in range(count):
        items[i].payload = base + i * ((comp + 255) // 256 * 256)  # back to back, 256-byte steps
        items[i].out = base
        items[i].codebook = base
        items[i].n = n
        items[i].capacity = comp
        metas[i] = layout
    step = (comp + 255) // 256 * 256  # halves are whole multiples of 256 bytes
    one = lib.sz_decode_many_host_scratch_bytes(items, metas, count, 2 * step)       # a tensor per group
    all6 = lib.sz_decode_many_host_scratch_bytes(items, metas, count, 2 * 6 * step)  # all in one group
    # metas, item tables and the decode workspace (its 256-byte status header, whatever the groups)
    r256 = lambda v: (v + 255) // 256 * 256
    assert one == all6 == r256(count * 96) + r256(count * 64) + 256
    assert lib.sz_decode_many_host_scratch_bytes(items, metas, count, comp) == 0  # a payload exceeds half
    metas[3].n = n + 1
    assert lib.sz_decode_many_host_scratch_bytes(items, metas, count, 2 * step) == 0  # meta disagrees with n
    assert lib.sz_decode_many_host_flags_offset(count) % 256 == 0
    # the pinned upload buffer: the metas (256-byte rounded) then the tables
    for c in (1, 2, 3, 6, 1000):
        assert lib.sz_decode_many_host_upload_bytes(c) == ((c * 96 + 255) // 256) * 256 + c * 64
    assert lib.sz_decode_many_host_upload_bytes(0) == 0


# ---------------------------------------------------------------------------- in-place slot decode schedule


def _inplace_cases():
    # (n, n_esc): one tile, ragged tails, tile boundaries, an odd off_sm, escape
    # counts up to the largest payload that still fits in the 2n-byte slot
    cases = []
    for n in (2, 3, 4, 7, 8191, 8192, 8193, 16384, 16385, 24577, 65536, 100_003, 262_144, 1_000_001, 2_097_152):
        for frac in (0.0, 1e-4, 0.01, 0.0714):
            e = int(n * frac)
            cases.append((n, e))
    return cases


@pytest.mark.parametrize("n,e", _inplace_cases())
def test_inplace_schedule_covers_every_payload_byte(lib, n, e):
    """For the decode over the slot, in the plan's order: every payload byte
    read in place is overwritten (slot byte b belongs to output tile
    b // 16384) only by its own reader's tile or by a later tile that waits
    for its reader; every other byte read is in the stash; every tile waited
    for comes earlier in the order (so the schedule cannot deadlock); the
    order is a permutation; the stash fits its budget."""
    m = sz.sz_layout(n, e)
    if m.comp_bytes > 2 * n:
        with pytest.raises(B.SplitZipError):
            sz.inplace_plan(n, e, 0)
        return
    T = (n + 8191) // 8192
    plans = [sz.inplace_plan(n, e, u) for u in range(T)]
    p0 = plans[0]
    for p in plans:
        for k in ("tiles", "phase_a_first", "phase_b_end", "stash_pk_from", "stash_pk_to", "stash_esc_from",
                  "stash_esc_to", "stash_bytes", "stash_budget"):
            assert p[k] == p0[k]
    assert p0["tiles"] == T and p0["stash_bytes"] <= p0["stash_budget"]
    tA, tB = p0["phase_a_first"], p0["phase_b_end"]
    assert 0 <= tB <= tA <= T
    rank = np.array([p["rank"] for p in plans], dtype=np.int64)
    assert sorted(rank.tolist()) == list(range(T))
    ranges = np.array([[p["pk_lo"], p["pk_hi"], p["pk2_lo"], p["pk2_hi"], p["sm_lo"], p["sm_hi"]] for p in plans],
                      dtype=np.int64)
    for u in range(T):
        for lo, hi in ranges[u].reshape(3, 2):
            for d in range(lo, hi + 1):
                assert 0 <= d < T and (d == u or rank[d] < rank[u]), (u, d)

    def check_in_place(b, r):
        w = b // 16384
        assert np.all(w < T)
        other = w != r
        ww, rr = w[other], r[other]
        assert np.all(rank[rr] < rank[ww]), "a byte is overwritten by a tile decoded before its reader"
        rg = ranges[ww]
        ok = np.zeros(ww.size, dtype=bool)
        for k in range(3):
            ok |= (rg[:, 2 * k] <= rr) & (rr <= rg[:, 2 * k + 1])
        assert np.all(ok), "a tile stores over bytes whose reader it does not wait for"

    # pk: element i's code is in byte i // 2, read by tile i // 8192; phase C's
    # pk comes from the stash, but tile 0's (under tile 0 itself)
    b = np.arange(m.n_pairs, dtype=np.int64)
    r = b // 4096
    stashed = (tB <= r) & (r < tA) & (r > 0)
    assert np.all((p0["stash_pk_from"] <= b[stashed]) & (b[stashed] < p0["stash_pk_to"]))
    check_in_place(b[~stashed], r[~stashed])
    # sm: element i's byte at off_sm + i, read by tile i // 8192, always in place
    i = np.arange(n, dtype=np.int64)
    check_in_place(m.off_sm + i, i // 8192)
    # escape streams: stashed whole
    if e:
        assert p0["stash_esc_from"] <= m.off_cid and p0["stash_esc_to"] >= m.off_ev + e
    else:
        assert p0["stash_esc_to"] == p0["stash_esc_from"]
    # the stash is about n / 8 + 7 e bytes (the whole payload is 1.5 n + 7 e)
    assert p0["stash_pk_to"] - p0["stash_pk_from"] <= n // 8 + 8200


def test_inplace_plan_rejects_bad_arguments(lib):
    t = B.SzInplaceTile()
    assert lib.sz_inplace_plan(0, 0, 0, ctypes.byref(t)) == B.SZ_ERR_ARG
    assert lib.sz_inplace_plan(8192, 0, 1, ctypes.byref(t)) == B.SZ_ERR_ARG  # one tile only
    assert lib.sz_inplace_plan(100, 101, 0, ctypes.byref(t)) == B.SZ_ERR_ARG
    assert lib.sz_inplace_plan(1, 0, 0, ctypes.byref(t)) == B.SZ_ERR_CAPACITY  # 8-byte payload, 2-byte slot
    assert lib.sz_inplace_plan(8192, 0, 0, None) == B.SZ_ERR_ARG
    # header, item flags, escape ranges and tile map (256 bytes each here), read_done, stash
    assert lib.sz_decode_inplace_workspace_bytes(3, 10) == 4 * 256 + 256 + 10 * 8192 + 3 * 4352
    # the out-of-place decode finds everything in the kernel: its workspace is the status header
    assert lib.sz_decode_workspace_bytes(3, 10) == lib.sz_decode_workspace_bytes(1, 1 << 19) == 256
