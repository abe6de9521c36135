"""Tables of small tensors (at most two tiles on average, such as the blocks of a
paged KV cache) take the whole-tensor paths of sz_encode_many,
sz_calibrate_encode_many and sz_decode_many: each tensor held in shared
memory.  Their results are checked here against the CPU oracle tensor by
tensor at ragged sizes, escape-heavy inputs, flagged items, the coverage
gate, and tables with a tensor the whole-tensor kernels leave to the tile
kernels."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

import gpu_util
from gpu_util import DEV, check_codebook, to_dev, to_np_u16

pytestmark = pytest.mark.gpu

SMALL_MAX = 2 * 8192  # elements of the largest tensor held whole


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)


def _tiles(n: int) -> int:
    return (n + 8191) // 8192


def _small_routed(arrays) -> bool:
    return sum(_tiles(a.size) for a in arrays) <= 2 * len(arrays)


def _encode_both_ways(arrays):
    """Calibrate + encode of the table as one fused call and as two calls."""
    xs = [to_dev(a) for a in arrays]
    out = []
    for fused in (True, False):
        b = sz.Batch(xs)
        ws = sz.Workspace(DEV)
        if fused:
            sz.sz_calibrate_encode_many(b.table, workspace=ws)
            flags = sz.sz_workspace_flags(ws.buf)
        else:
            sz.sz_calibrate_many(b.table, workspace=ws)
            flags = sz.sz_workspace_flags(ws.buf)
            sz.sz_encode_many(b.table, workspace=ws)
            flags |= sz.sz_workspace_flags(ws.buf)
        torch.cuda.synchronize()
        assert flags == 0
        out.append(b)
    return out


def _check_against_oracle(b: "sz.Batch", arrays) -> None:
    cbs = b.codebooks.cpu().numpy()
    for i, x in enumerate(arrays):
        ocb = oracle.calibrate(x)
        check_codebook(sz.codebook_from_bytes(cbs[i]), ocb, x.size)
        opay, om = oracle.encode(x, ocb)
        m = sz.meta_from_bytes(b.metas[i].cpu().numpy())
        assert m.status == 0 and m.as_tuple() == om.as_tuple(), (i, x.size, m, om)
        assert m.coverage == ocb.coverage
        gp = b.payload_view(i, om.comp_bytes).cpu().numpy()
        assert np.array_equal(gp, opay), f"tensor {i} (n={x.size}): payload differs"


def _ragged_table():
    sizes = [0, 1, 2, 3, 7, 8, 9, 15, 16, 17, 255, 1023, 1024, 1025, 4097, 8191, 8192, 8193, 12_345, 16_383, 16_384]
    arrays = []
    for k, n in enumerate(sizes):
        kind = k % 3
        if kind == 0:
            arrays.append(inputs.gaussian(n, 0.02, seed=700 + k))
        elif kind == 1:
            arrays.append(inputs.edge_case(n, seed=700 + k))  # broad exponents: many escapes
        else:
            a = inputs.gaussian(n, 1.0, seed=700 + k)
            a[::97] = inputs.edge_case(a[::97].size, seed=800 + k)  # sparse escapes
            arrays.append(a)
    return arrays


def test_small_table_ragged_sizes_match_the_oracle():
    arrays = _ragged_table()
    assert _small_routed(arrays)
    fused, separate = _encode_both_ways(arrays)
    for b in (fused, separate):
        _check_against_oracle(b, arrays)
    # and decode back
    sz.sz_decode_many(fused.table)
    torch.cuda.synchronize()
    for i, x in enumerate(arrays):
        assert np.array_equal(to_np_u16(fused.out_view(i)), x), f"decode {i}"


def test_small_table_many_blocks_and_escape_heavy_blocks():
    arrays = [inputs.paged_kv_block(i) for i in range(400)]
    for k in range(0, 400, 37):  # every 37th block escape-heavy
        arrays[k] = inputs.edge_case(SMALL_MAX, seed=900 + k)
    assert _small_routed(arrays)
    fused, separate = _encode_both_ways(arrays)
    assert torch.equal(fused.codebooks, separate.codebooks) and torch.equal(fused.metas, separate.metas)
    for i in range(len(arrays)):
        m = sz.meta_from_bytes(fused.metas[i].cpu().numpy())
        assert torch.equal(fused.payload_view(i, m.comp_bytes), separate.payload_view(i, m.comp_bytes)), i
    sample = [0, 1, 37, 74, 200, 399]
    sub = sz.Batch([to_dev(arrays[i]) for i in sample])
    sz.sz_calibrate_encode_many(sub.table)
    torch.cuda.synchronize()
    _check_against_oracle(sub, [arrays[i] for i in sample])


def _tie_tensor(n: int, bins: int, seed: int) -> np.ndarray:
    """n patterns spread evenly over `bins` exponents (equal counts where n
    allows: ties broken by ascending exponent), random sign and mantissa."""
    rng = np.random.default_rng(seed)
    e = (90 + np.arange(n) % bins).astype(np.uint16)
    rng.shuffle(e)
    return (rng.integers(0, 2, n, dtype=np.uint16) << 15) | (e << 7) | rng.integers(0, 128, n, dtype=np.uint16)


def test_small_table_calibrate_alone_matches_the_oracle():
    # sz_calibrate_many on its own: every codebook byte against the oracle's,
    # over paged blocks, ragged sizes, one-bin, tied and escape-heavy tensors
    arrays = [inputs.paged_kv_block(i) for i in range(600)]
    arrays += _ragged_table()
    arrays += [np.full(n, v, np.uint16) for n, v in ((16_384, 0x3F80), (5, 0x0000), (9, 0x8001))]
    arrays += [_tie_tensor(n, bins, 990 + k) for k, (n, bins) in
               enumerate(((16_384, 16), (16_384, 17), (16_000, 20), (8_191, 40), (12_289, 256), (33, 33)))]
    assert _small_routed(arrays) and max(a.size for a in arrays) <= SMALL_MAX
    b = sz.Batch([to_dev(a) for a in arrays])
    b.codebooks.fill_(0xAB)
    ws = sz.Workspace(DEV)
    sz.sz_calibrate_many(b.table, workspace=ws)
    torch.cuda.synchronize()
    assert sz.sz_workspace_flags(ws.buf) == 0
    cbs = b.codebooks.cpu().numpy()
    for i, x in enumerate(arrays):
        want = np.frombuffer(gpu_util.oracle_codebook_bytes(oracle.calibrate(x), x.size), np.uint8)
        assert np.array_equal(cbs[i][:want.size], want), f"codebook {i} (n={x.size})"


def test_small_table_with_one_large_tensor_goes_to_the_general_kernels():
    arrays = [inputs.gaussian(40_000, 0.02, seed=950)] + [inputs.edge_case(1000 + 37 * k, seed=951 + k)
                                                           for k in range(30)]
    assert _small_routed(arrays) and arrays[0].size > SMALL_MAX
    fused, separate = _encode_both_ways(arrays)
    for b in (fused, separate):
        _check_against_oracle(b, arrays)


def test_small_table_flags_match_between_the_calls():
    # item 1's input is misaligned (skipped by both passes), item 2's payload
    # is too small (calibrated, not encoded), item 3 is empty
    arrays = [inputs.gaussian(5000, 0.02, seed=960 + k) for k in range(3)] + [np.zeros(0, np.uint16)]
    assert _small_routed(arrays)
    xs = [to_dev(a) for a in arrays]
    base = torch.zeros(5000 + 8, dtype=torch.int16, device=DEV)
    base[1:5001] = xs[1]
    xs[1] = base[1:5001]  # 2-byte offset: not 16-byte aligned
    outs = []
    for fused in (False, True):
        b = sz.Batch(xs, capacity=[sz.sz_max_payload_bytes(5000), sz.sz_max_payload_bytes(5000), 500, 16])
        b.codebooks.fill_(0xAB)
        ws = sz.Workspace(DEV)
        if fused:
            sz.sz_calibrate_encode_many(b.table, workspace=ws)
            flags = sz.sz_workspace_flags(ws.buf)
        else:
            sz.sz_calibrate_many(b.table, workspace=ws)
            flags = sz.sz_workspace_flags(ws.buf)
            sz.sz_encode_many(b.table, workspace=ws)
            flags |= sz.sz_workspace_flags(ws.buf)
        torch.cuda.synchronize()
        outs.append((flags, b.codebooks.cpu().clone(), b.metas.cpu().clone(), b.payload_view(0).cpu().clone()))
    (f1, c1, m1, p1), (f2, c2, m2, p2) = outs
    assert f1 == f2 and f1 & B.SZ_FLAG_ALIGN and f1 & B.SZ_FLAG_CAPACITY
    assert torch.equal(c1, c2) and torch.equal(m1, m2)
    n0 = sz.meta_from_bytes(m1[0].numpy()).comp_bytes
    assert torch.equal(p1[:n0], p2[:n0])
    # item 0 is right; item 2 got its codebook but no payload; item 3 is empty
    ocb = oracle.calibrate(arrays[0])
    check_codebook(sz.codebook_from_bytes(c2[0].numpy()), ocb, 5000)
    opay, om = oracle.encode(arrays[0], ocb)
    assert sz.meta_from_bytes(m2[0].numpy()).as_tuple() == om.as_tuple() and np.array_equal(p2[:n0].numpy(), opay)
    check_codebook(sz.codebook_from_bytes(c2[2].numpy()), oracle.calibrate(arrays[2]), 5000)
    assert sz.meta_from_bytes(m2[2].numpy()).status & B.SZ_FLAG_CAPACITY
    m3 = sz.meta_from_bytes(m2[3].numpy())
    assert m3.status == 0 and m3.n == 0 and m3.comp_bytes == 0


@pytest.mark.parametrize("gate", [0.99, -1.0])
def test_small_table_gate_matches_the_oracle(gate):
    arrays = [inputs.paged_kv_block(i) for i in range(40)] + [inputs.edge_case(3000 + k, seed=970 + k)
                                                              for k in range(8)]
    assert _small_routed(arrays)
    xs = [to_dev(a) for a in arrays]
    b = sz.Batch(xs)
    sz.sz_calibrate_many(b.table)
    b.payload.fill_(0x5A)
    ws = sz.Workspace(DEV)
    report = sz.sz_encode_gated_many(b.table, gate, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    cbs = [sz.codebook_from_bytes(c) for c in b.codebooks.cpu().numpy()]
    ometas = []
    for i, x in enumerate(arrays):
        ocb = oracle.calibrate(x)
        assert cbs[i].coverage == ocb.coverage
        opay, om = oracle.encode(x, ocb)
        ometas.append(om)
        m = sz.meta_from_bytes(b.metas[i].cpu().numpy())
        if oracle.gated(ocb.coverage, gate):
            assert m.status == B.SZ_META_GATED and m.n == x.size and m.coverage == ocb.coverage
            assert bool(torch.all(b.payload_view(i) == 0x5A)), f"gated tensor {i}: payload written"
        else:
            assert m.status == 0 and m.as_tuple() == om.as_tuple()
            assert np.array_equal(b.payload_view(i, om.comp_bytes).cpu().numpy(), opay)
    expect = oracle.gate_report([a.size for a in arrays], [c.coverage for c in cbs], ometas, gate)
    assert sz.read_gate_report(report) == expect
    if gate > 0:
        assert any(oracle.gated(c.coverage, gate) for c in cbs) and not all(oracle.gated(c.coverage, gate)
                                                                           for c in cbs)


def _decode_table(b: "sz.Batch", fill: int = 7) -> int:
    b.out.view(torch.int16).fill_(fill)
    ws = sz.Workspace(DEV)
    sz.sz_decode_many(b.table, workspace=ws)
    flags = sz.sz_workspace_flags(ws.buf)
    torch.cuda.synchronize()
    return flags


def test_small_table_decode_of_the_oracle_payloads():
    """Payloads written by the CPU oracle (not by this library), decoded as a
    table of small tensors: ragged sizes, escapes, and tensors whose payload
    is too large for the whole-tensor kernel (left to the tile kernel)."""
    arrays = _ragged_table() + [inputs.edge_case(SMALL_MAX, seed=990), inputs.edge_case(9000, seed=991)]
    assert _small_routed(arrays)
    b = sz.Batch([to_dev(a) for a in arrays])
    for i, x in enumerate(arrays):
        ocb = oracle.calibrate(x)
        opay, om = oracle.encode(x, ocb)
        b.codebooks[i].copy_(torch.frombuffer(bytearray(gpu_util.oracle_codebook_bytes(ocb, x.size)),
                                              dtype=torch.uint8).to(DEV))
        b.metas[i].copy_(torch.frombuffer(bytearray(sz.meta_to_bytes(om)), dtype=torch.uint8).to(DEV))
        if om.comp_bytes:
            b.payload_view(i, om.comp_bytes).copy_(torch.from_numpy(opay).to(DEV))
    assert _decode_table(b) == 0
    for i, x in enumerate(arrays):
        assert np.array_equal(to_np_u16(b.out_view(i)), x), f"tensor {i} (n={x.size})"


def test_small_table_decode_with_one_large_tensor_and_flags():
    arrays = [inputs.gaussian(40_000, 0.02, seed=992)] + [inputs.gaussian(5000 + 7 * k, 0.5, seed=1000 + k)
                                                           for k in range(20)]
    assert _small_routed(arrays) and arrays[0].size > SMALL_MAX
    b = sz.Batch([to_dev(a) for a in arrays])
    sz.sz_calibrate_encode_many(b.table)
    torch.cuda.synchronize()
    assert _decode_table(b) == 0
    for i, x in enumerate(arrays):
        assert np.array_equal(to_np_u16(b.out_view(i)), x), f"tensor {i}"
    # a meta that disagrees with the layout: that tensor is flagged and left untouched, the rest decoded
    import dataclasses

    m3 = sz.meta_from_bytes(b.metas[3].cpu().numpy())
    b.metas[3].copy_(torch.frombuffer(bytearray(sz.meta_to_bytes(dataclasses.replace(m3, off_sm=m3.off_sm + 4))),
                                      dtype=torch.uint8).to(DEV))
    flags = _decode_table(b)
    assert flags & B.SZ_FLAG_META
    assert bool(torch.all(b.out_view(3).view(torch.int16) == 7))
    for i, x in enumerate(arrays):
        if i != 3:
            assert np.array_equal(to_np_u16(b.out_view(i)), x), f"tensor {i}"


def test_small_table_decode_flags_an_escape_outside_its_chunk():
    arrays = [inputs.edge_case(2000, seed=993 + k) for k in range(3)]
    assert _small_routed(arrays)
    b = sz.Batch([to_dev(a) for a in arrays])
    sz.sz_calibrate_encode_many(b.table)
    torch.cuda.synchronize()
    m = sz.meta_from_bytes(b.metas[1].cpu().numpy())
    assert m.n_esc > 0 and m.comp_bytes <= 26_624  # decoded whole (its payload fits a buffer)
    lpos = b.payload_view(1, m.comp_bytes)[m.off_lpos:m.off_lpos + 2]
    lpos.copy_(torch.tensor([0x00, 0x04], dtype=torch.uint8, device=DEV))  # local_pos 1024
    flags = _decode_table(b)
    assert flags & B.SZ_FLAG_ESCAPE
    for i in (0, 2):
        assert np.array_equal(to_np_u16(b.out_view(i)), arrays[i]), f"tensor {i}"


def test_small_table_decode_leaves_gated_tensors_untouched():
    arrays = [inputs.paged_kv_block(i) for i in range(10)] + [inputs.edge_case(6000, seed=996)]
    assert _small_routed(arrays)
    b = sz.Batch([to_dev(a) for a in arrays])
    sz.sz_calibrate_many(b.table)
    sz.sz_encode_gated_many(b.table, 0.99)
    torch.cuda.synchronize()
    assert sz.meta_from_bytes(b.metas[10].cpu().numpy()).status == B.SZ_META_GATED
    assert _decode_table(b) == 0
    assert bool(torch.all(b.out_view(10).view(torch.int16) == 7))
    for i in range(10):
        assert np.array_equal(to_np_u16(b.out_view(i)), arrays[i]), f"tensor {i}"
