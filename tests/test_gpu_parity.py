"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer work, so the bar is exact: codebooks, metas and payload bytes
identical to the oracle's, decodes bit-identical to the input.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

from gpu_util import DEV, check_codebook, roundtrip_single, to_dev, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    sz.lib()
    torch.cuda.set_device(DEV)


SIZES = [0, 1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 1023, 1024, 1025, 2047, 4095, 4096, 8191, 8192, 8193,
         16383, 16384, 16385, 24577, 40961, 100_003]


@pytest.mark.parametrize("n", SIZES)
def test_gaussian_sizes(n):
    roundtrip_single(inputs.gaussian(n, 0.02, seed=n))


@pytest.mark.parametrize("n", SIZES)
def test_escape_heavy_sizes(n):
    roundtrip_single(inputs.edge_case(n, seed=n))


def test_all_bit_patterns():
    r = roundtrip_single(inputs.all_bit_patterns())
    assert r["meta"].n_esc == 61440 and r["meta"].comp_bytes == 528384


@pytest.mark.parametrize("shift", [0, 1, 2, 3, 4, 5, 6, 7])
def test_sm_section_alignment_classes(shift):
    """off_sm = align4(ceil(n/2)) takes every residue mod 16 as n varies; the
    decoder stages sm through 16-byte-aligned copies and must handle each."""
    n = 3 * 8192 + 8 * shift + (shift % 3)
    x = inputs.gaussian(n, 1.0, seed=shift)
    x[::301] = inputs.edge_case(x[::301].size, seed=shift)
    m = roundtrip_single(x)["meta"]
    assert m.n == n


def test_codebook_from_other_tensor():
    x = inputs.gaussian(50_001, 1.0, seed=2)
    roundtrip_single(x, codebook_from=inputs.gaussian(4_096, 1e-3, seed=3))
    roundtrip_single(x, codebook_from=np.array([0x3F80, 0x3F80, 0x0000], dtype=np.uint16))


def test_out_of_contract_enc_lut_stays_in_bounds():
    """enc_lut entries other than 0..15 and SZ_ESCAPE_CODE are not checked: the
    payload is then unspecified, but encode and decode stay within their
    buffers, flag nothing and agree with the layout of the escape count."""
    from weight_compression_codec_gb300 import binding as B

    x = inputs.gaussian(3 * 8192 + 77, 1.0, seed=21)  # full tiles and a ragged one
    rng = np.random.default_rng(21)
    c = B.SzCodebook()
    c.enc_lut[:] = rng.integers(0, 256, 256).tolist()
    c.dec_lut[:] = rng.integers(0, 256, 16).tolist()
    c.n_top, c.top_count, c.n, c.coverage = 16, 0, x.size, 0.5
    cb = torch.frombuffer(bytearray(bytes(c)), dtype=torch.uint8).to(DEV)
    ws = sz.Workspace(DEV)
    payload, meta = sz.sz_encode(to_dev(x), cb, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    m = sz.read_meta(meta)
    assert m.status == 0 and m.n_esc <= x.size
    assert m.as_tuple() == oracle.layout(x.size, m.n_esc).as_tuple()
    sz.sz_decode(payload, meta, cb, x.size, workspace=ws)
    torch.cuda.synchronize()
    assert sz.sz_workspace_flags(ws.buf) == 0


def test_dense_escapes_spill_path():
    """Tiles with more escapes than the decoder stages in shared memory."""
    x = inputs.edge_case(3 * 8192 + 77, seed=11)
    r = roundtrip_single(x, codebook_from=np.array([0x3F80], dtype=np.uint16))
    assert r["meta"].n_esc > 0.9 * x.size


def test_repeated_calls_reuse_workspace():
    ws = sz.Workspace(DEV)
    x = inputs.gaussian(70_001, 0.5, seed=4)
    xd = to_dev(x)
    for _ in range(3):
        cb = sz.sz_calibrate(xd, workspace=ws)
        payload, meta = sz.sz_encode(xd, cb, workspace=ws)
        out = sz.sz_decode(payload, meta, cb, x.size, workspace=ws)
        assert sz.sz_workspace_flags(ws.buf) == 0
        assert np.array_equal(to_np_u16(out), x)


def test_nondefault_stream():
    s = torch.cuda.Stream()
    x = inputs.edge_case(33_333, seed=8)
    xd = to_dev(x)
    with torch.cuda.stream(s):
        cb = sz.sz_calibrate(xd, stream=s)
        payload, meta = sz.sz_encode(xd, cb, stream=s)
        out = sz.sz_decode(payload, meta, cb, x.size, stream=s)
    s.synchronize()
    assert np.array_equal(to_np_u16(out), x)


# ---------------------------------------------------------------------------- device-side errors


def test_capacity_overrun_is_flagged_and_bounded():
    x = inputs.edge_case(20_000, seed=1)
    xd = to_dev(x)
    cb = sz.sz_calibrate(xd)
    full = oracle.encode(x, oracle.calibrate(x))[1]
    cap = full.off_cid + 4 * 100  # room for the dense part and 100 chunk ids only
    buf = torch.full((cap + 4096,), 0xA5, dtype=torch.uint8, device=DEV)
    meta = torch.empty(96, dtype=torch.uint8, device=DEV)
    ws = sz.Workspace(DEV)
    sz.sz_encode(xd, cb, payload=buf[:cap], meta=meta, workspace=ws)
    flags = sz.sz_workspace_flags(ws.buf)
    assert flags & B.SZ_FLAG_CAPACITY
    m = sz.read_meta(meta)
    assert m.status & B.SZ_FLAG_CAPACITY and m.n_esc == full.n_esc
    assert torch.all(buf[cap:] == 0xA5), "bytes beyond capacity were written"


def test_malformed_meta_is_flagged_and_output_untouched():
    x = inputs.gaussian(30_000, 1.0, seed=3)
    xd = to_dev(x)
    cb = sz.sz_calibrate(xd)
    payload, meta = sz.sz_encode(xd, cb)
    good = sz.read_meta(meta)
    import dataclasses

    for field, delta in (("off_sm", 4), ("comp_bytes", 1), ("chunk_size", 1), ("n_esc", 1)):
        bad = dataclasses.replace(good, **{field: getattr(good, field) + delta})
        mb = torch.frombuffer(bytearray(sz.meta_to_bytes(bad)), dtype=torch.uint8).to(DEV)
        out = torch.full((x.size,), 7, dtype=torch.int16, device=DEV)
        ws = sz.Workspace(DEV)
        sz.sz_decode(payload, mb, cb, x.size, out=out, workspace=ws)
        assert sz.sz_workspace_flags(ws.buf) & B.SZ_FLAG_META
        assert torch.all(out == 7)
    # a payload shorter than comp_bytes is rejected the same way
    ws = sz.Workspace(DEV)
    out = torch.full((x.size,), 7, dtype=torch.int16, device=DEV)
    sz.sz_decode(payload[:good.comp_bytes - 1], meta, cb, x.size, out=out, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) & B.SZ_FLAG_META and torch.all(out == 7)


def test_out_of_range_escape_is_flagged():
    x = inputs.edge_case(9_000, seed=2)
    xd = to_dev(x)
    cb = sz.sz_calibrate(xd)
    payload, meta = sz.sz_encode(xd, cb)
    m = sz.read_meta(meta)
    assert m.n_esc > 10
    bad = payload.clone()
    bad[m.off_lpos:m.off_lpos + 2] = torch.tensor([0x00, 0x04], dtype=torch.uint8)  # local_pos 1024
    ws = sz.Workspace(DEV)
    out = sz.sz_decode(bad, meta, cb, x.size, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) & B.SZ_FLAG_ESCAPE
    y = to_np_u16(out)
    assert np.count_nonzero(y != x) <= 1  # only the corrupted escape is missing


# ---------------------------------------------------------------------------- many tensors


def _check_batch(batch: "sz.Batch", arrays: list[np.ndarray]) -> None:
    torch.cuda.synchronize()
    for i, x in enumerate(arrays):
        ocb = oracle.calibrate(x)
        check_codebook(sz.codebook_from_bytes(batch.codebooks[i].cpu().numpy()), ocb, x.size)
        opay, om = oracle.encode(x, ocb)
        m = sz.meta_from_bytes(batch.metas[i].cpu().numpy())
        assert m.status == 0 and m.as_tuple() == om.as_tuple(), (i, m, om)
        assert np.array_equal(batch.payload_view(i, m.comp_bytes).cpu().numpy(), opay), f"payload {i}"
        assert np.array_equal(to_np_u16(batch.out_view(i)), x), f"decode {i}"


def test_many_ragged_with_empty_items():
    arrays = [inputs.gaussian(n, 0.02, seed=n) for n in (0, 1, 8191, 8192, 8193, 0, 100_003, 3, 0)]
    arrays[6][::97] = inputs.edge_case(arrays[6][::97].size, seed=6)
    xs = [to_dev(a) for a in arrays]
    b = sz.Batch(xs)
    ws = sz.Workspace(DEV)
    sz.sz_calibrate_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    sz.sz_encode_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    sz.sz_decode_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    _check_batch(b, arrays)


def test_many_kv_cache_reduced():
    arrays = inputs.kv_cache(layers=3, tokens=512)
    b = sz.Batch([to_dev(a) for a in arrays])
    sz.sz_calibrate_many(b.table)
    sz.sz_encode_many(b.table)
    sz.sz_decode_many(b.table)
    _check_batch(b, arrays)


def test_many_item_table_errors_are_flagged():
    arrays = [inputs.gaussian(5000, 1.0, seed=1), inputs.gaussian(7000, 1.0, seed=2)]
    b = sz.Batch([to_dev(a) for a in arrays])
    # corrupt tile_begin of item 1 in the device table
    host = bytearray(bytes(b.table.host))
    host[64 + 56:64 + 64] = (5).to_bytes(8, "little")
    bad_table = torch.frombuffer(host, dtype=torch.uint8).to(DEV)
    ws = sz.Workspace(DEV)
    buf = ws.get(B.lib().sz_encode_workspace_bytes(2, b.table.total_tiles), DEV)
    rc = B.lib().sz_encode_many(bad_table.data_ptr(), 2, b.table.total_tiles, buf.data_ptr(), buf.numel(),
                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert sz.sz_workspace_flags(buf) & B.SZ_FLAG_ITEMS
