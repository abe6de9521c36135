"""sz_encode_gated_many: the coverage gate of the shard-cache builder on the GPU,
against the oracle's gate and report and against the ungated call."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

from gpu_util import DEV, to_dev, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)


def _arrays():
    # coverages ~1 (Gaussian), 0.9999.. (KV slice), 1/16 (all patterns), ~0.22
    # (escape-heavy), 1.0 (empty) and a mix in between
    mix = inputs.gaussian(300_001, 0.02, seed=51)
    broad = inputs.edge_case(300_001, seed=52)
    mix[::50] = broad[::50]  # 2 % broad exponents: coverage just below 0.99
    return [inputs.gaussian(100_003, 0.02, seed=50), inputs.kv_cache_tensor(0, 1)[:2_000_000],
            inputs.all_bit_patterns(), inputs.edge_case(200_001, seed=53), np.zeros(0, np.uint16), mix]


@pytest.mark.parametrize("gate", [0.99, 0.5, -1.0, 1.0])
def test_gate_matches_oracle_and_ungated_encode(gate):
    arrays = _arrays()
    xs = [to_dev(a) for a in arrays]
    plain, gated = sz.Batch(xs), sz.Batch(xs)
    for b in (plain, gated):
        sz.sz_calibrate_many(b.table)
    torch.cuda.synchronize()
    assert torch.equal(plain.codebooks, gated.codebooks)
    sz.sz_encode_many(plain.table)
    gated.payload.fill_(0x5A)
    ws = sz.Workspace(DEV)
    report = sz.sz_encode_gated_many(gated.table, gate, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    cbs = [sz.codebook_from_bytes(c) for c in gated.codebooks.cpu().numpy()]
    ometas = []
    for i, x in enumerate(arrays):
        ocb = oracle.calibrate(x)
        assert cbs[i].coverage == ocb.coverage
        opay, om = oracle.encode(x, ocb)
        ometas.append(om)
        m = sz.meta_from_bytes(gated.metas[i].cpu().numpy())
        if oracle.gated(ocb.coverage, gate):
            assert m.status == B.SZ_META_GATED and m.n == x.size and m.coverage == ocb.coverage
            assert (m.n_pairs, m.n_esc, m.comp_bytes, m.off_sm, m.off_cid, m.off_lpos, m.off_ev) == (0,) * 7
            assert bool(torch.all(gated.payload_view(i) == 0x5A)), f"gated tensor {i}: payload written"
        else:
            assert m.status == 0 and m.as_tuple() == om.as_tuple()
            assert torch.equal(gated.metas[i], plain.metas[i])
            assert np.array_equal(gated.payload_view(i, om.comp_bytes).cpu().numpy(), opay)
    expect = oracle.gate_report([a.size for a in arrays], [c.coverage for c in cbs], ometas, gate)
    assert sz.read_gate_report(report) == expect
    # decode: gated tensors are left untouched, with no flag
    gated.out.view(torch.int16).fill_(7)
    wd = sz.Workspace(DEV)
    sz.sz_decode_many(gated.table, workspace=wd)
    assert sz.sz_workspace_flags(wd.buf) == 0
    torch.cuda.synchronize()
    for i, x in enumerate(arrays):
        y = to_np_u16(gated.out_view(i))
        if oracle.gated(cbs[i].coverage, gate):
            assert np.all(y == 7)
        else:
            assert np.array_equal(y, x)


def test_gate_coverage_values_of_the_batch():
    # the batch spans both sides of 0.99 and of 0.5, so every gate above is exercised
    covs = [oracle.calibrate(a).coverage for a in _arrays()]
    assert min(covs) < 0.5 < 0.99 < max(covs)
    assert any(0.5 <= c < 0.99 for c in covs)


def test_gate_rejects_bad_arguments():
    b = sz.Batch([to_dev(inputs.gaussian(1000, 0.02, seed=54))])
    ws = sz.Workspace(DEV).get(B.lib().sz_encode_workspace_bytes(1, b.table.total_tiles), DEV)
    s = torch.cuda.current_stream().cuda_stream
    rep = torch.empty(64, dtype=torch.uint8, device=DEV)
    lib = B.lib()
    assert lib.sz_encode_gated_many(b.table.ptr(), 1, b.table.total_tiles, 0.99, None, ws.data_ptr(), ws.numel(),
                                    s) == B.SZ_ERR_ARG
    assert lib.sz_encode_gated_many(b.table.ptr(), 1, b.table.total_tiles, float("nan"), rep.data_ptr(),
                                    ws.data_ptr(), ws.numel(), s) == B.SZ_ERR_ARG
    assert lib.sz_encode_gated_many(b.table.ptr(), 1, b.table.total_tiles, 0.99, rep.data_ptr() + 8,
                                    ws.data_ptr(), ws.numel(), s) == B.SZ_ERR_ALIGN
