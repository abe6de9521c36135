"""sz_calibrate_encode(_many): one call, results identical to
sz_calibrate(_many) followed by sz_encode(_many) and to the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

from gpu_util import DEV, check_codebook, to_dev, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)


def _fused_vs_separate(arrays: list[np.ndarray], oracle_check: bool = True) -> list:
    xs = [to_dev(a) for a in arrays]
    sep, fus = sz.Batch(xs), sz.Batch(xs)
    ws1, ws2 = sz.Workspace(DEV), sz.Workspace(DEV)
    sz.sz_calibrate_many(sep.table, workspace=ws1)
    assert sz.sz_workspace_flags(ws1.buf) == 0
    sz.sz_encode_many(sep.table, workspace=ws1)
    assert sz.sz_workspace_flags(ws1.buf) == 0
    sz.sz_calibrate_encode_many(fus.table, workspace=ws2)
    assert sz.sz_workspace_flags(ws2.buf) == 0
    torch.cuda.synchronize()
    assert torch.equal(sep.codebooks, fus.codebooks), "codebooks differ"
    assert torch.equal(sep.metas, fus.metas), "metas differ"
    metas = []
    for i in range(len(arrays)):
        m = sz.meta_from_bytes(fus.metas[i].cpu().numpy())
        assert m.status == 0
        assert torch.equal(sep.payload_view(i, m.comp_bytes), fus.payload_view(i, m.comp_bytes)), f"payload {i}"
        metas.append(m)
    if oracle_check:
        cbs = fus.codebooks.cpu().numpy()
        for i, x in enumerate(arrays):
            ocb = oracle.calibrate(x)
            check_codebook(sz.codebook_from_bytes(cbs[i]), ocb, x.size)
            opay, om = oracle.encode(x, ocb)
            assert metas[i].as_tuple() == om.as_tuple()
            assert np.array_equal(fus.payload_view(i, om.comp_bytes).cpu().numpy(), opay), f"oracle payload {i}"
    # the fused payloads decode back exactly
    sz.sz_decode_many(fus.table)
    torch.cuda.synchronize()
    for i, x in enumerate(arrays):
        assert np.array_equal(to_np_u16(fus.out_view(i)), x), f"decode {i}"
    return metas


def test_fused_kv_cache_spans_groups():
    # 8 KV tensors of 512 tiles = 2 groups of 2048 tiles
    arrays = [inputs.kv_cache_tensor(l, kv) for l in range(4) for kv in range(2)]
    _fused_vs_separate(arrays)


def test_fused_tensor_larger_than_a_group_then_small_ones():
    arrays = [inputs.gaussian(20_000_017, 1.0, seed=31)] + [inputs.gaussian(n, 0.02, seed=32 + n) for n in
                                                            (0, 1, 8191, 8193, 300_001, 0, 2_000_000)]
    _fused_vs_separate(arrays)


def test_fused_tensors_each_spanning_several_groups():
    # 3 tensors of 6,244 tiles: each covers the start of three 2048-tile
    # groups, so most groups are empty and the schedule runs over the others
    arrays = [inputs.gaussian(6244 * 8192 - 5 * i, 0.02, seed=40 + i) for i in range(3)]
    _fused_vs_separate(arrays)


def test_fused_many_small_tensors():
    arrays = [inputs.paged_kv_block(i) for i in range(3000)]
    _fused_vs_separate(arrays, oracle_check=False)
    # the oracle on a sample
    sample = [inputs.paged_kv_block(i) for i in (0, 1, 1499, 2999)]
    _fused_vs_separate(sample)


def test_fused_escape_heavy_and_all_bit_patterns():
    _fused_vs_separate([inputs.edge_case(3_000_001, seed=33), inputs.all_bit_patterns(),
                        inputs.edge_case(12_345, seed=34)])


def test_fused_single_tensor_call():
    x = inputs.edge_case(1_234_567, seed=35)
    cb, payload, meta = sz.sz_calibrate_encode(to_dev(x))
    torch.cuda.synchronize()
    ocb = oracle.calibrate(x)
    check_codebook(sz.read_codebook(cb), ocb, x.size)
    opay, om = oracle.encode(x, ocb)
    m = sz.read_meta(meta)
    assert m.status == 0 and m.as_tuple() == om.as_tuple()
    assert np.array_equal(payload[:m.comp_bytes].cpu().numpy(), opay)
    # empty tensor
    cb0, _, meta0 = sz.sz_calibrate_encode(torch.empty(0, dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert sz.read_codebook(cb0).coverage == 1.0 and sz.read_meta(meta0).comp_bytes == 0


def test_fused_flags_match_the_separate_calls():
    # item 1's input is misaligned (both passes skip it), item 2's payload is
    # too small (calibrated, not encoded): same flags, metas and codebooks
    arrays = [inputs.gaussian(50_000, 0.02, seed=36 + k) for k in range(3)]
    xs = [to_dev(a) for a in arrays]
    base = torch.zeros(50_000 + 8, dtype=torch.int16, device=DEV)
    base[1:50_001] = xs[1]
    xs[1] = base[1:50_001]  # 2-byte offset: not 16-byte aligned
    outs = []
    for fused in (False, True):
        b = sz.Batch(xs, capacity=[sz.sz_max_payload_bytes(50_000), sz.sz_max_payload_bytes(50_000), 1000])
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
    assert torch.equal(p1[:sz.meta_from_bytes(m1[0].numpy()).comp_bytes], p2[:sz.meta_from_bytes(m2[0].numpy()).comp_bytes])


def test_fused_rejects_an_inconsistent_table():
    arrays = [inputs.gaussian(20_000, 0.02, seed=40 + k) for k in range(4)]
    b = sz.Batch([to_dev(a) for a in arrays])
    host = bytearray(bytes(b.table.host))
    host[2 * 64 + 56:2 * 64 + 64] = (b.table.host[2].tile_begin + 1).to_bytes(8, "little")  # item 2's tile_begin
    bad_table = torch.frombuffer(host, dtype=torch.uint8).to(DEV)
    ws = sz.Workspace(DEV)
    buf = ws.get(B.lib().sz_calibrate_encode_workspace_bytes(4, b.table.total_tiles), DEV)
    rc = B.lib().sz_calibrate_encode_many(bad_table.data_ptr(), 4, b.table.total_tiles, buf.data_ptr(),
                                          buf.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert sz.sz_workspace_flags(buf) & B.SZ_FLAG_ITEMS
