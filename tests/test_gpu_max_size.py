"""The largest tensor the ABI takes: n = SZ_MAX_ELEMS = 2^32 - 1 elements (8 GiB of BF16).

At this size the byte offsets of the sm and escape sections pass 2^32 and the
chunk ids reach 2^22, so every offset the kernels form must be 64-bit. The
input repeats one 64 Mi-element block whose sign and mantissa bits change with
each repeat, so a tile read or written at the wrong place shows up. Calibrate
and encode are compared with the oracle byte for byte; decode and in-place
decode must give the input back bit for bit.

Memory: about 15 GB on the host (input and the oracle's payload) and about
55 GB on the device.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

from gpu_util import DEV, check_codebook

pytestmark = pytest.mark.gpu

BLOCK = 1 << 26


def _max_input() -> np.ndarray:
    n = B.SZ_MAX_ELEMS
    base = inputs.gaussian(BLOCK, 1.0, seed=77)
    heavy = np.random.default_rng(78).random(BLOCK) < 0.004  # escapes in every region
    base[heavy] = inputs.edge_case(BLOCK, seed=79)[heavy]
    reps = -(-n // BLOCK)
    x = np.tile(base, reps)
    # each repeat gets its own low mantissa bits (exponents, hence codebook and escapes, unchanged)
    x.reshape(reps, BLOCK)[...] ^= (np.arange(reps, dtype=np.uint16) * 37 % 128)[:, None]
    return x[:n]


def test_max_elements_round_trip_and_in_place():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)
    x = _max_input()
    n = x.size
    ocb = oracle.calibrate(x)
    opay, om = oracle.encode(x, ocb)
    assert om.off_ev + om.n_esc > 1 << 32 and om.n_esc > 0
    xd = torch.from_numpy(x.view(np.int16)).to(DEV)
    del x

    ws = sz.Workspace(DEV)
    cb = sz.sz_calibrate(xd, workspace=ws)
    torch.cuda.synchronize()
    check_codebook(sz.read_codebook(cb), ocb, n)

    payload = torch.empty(om.comp_bytes + 16, dtype=torch.uint8, device=DEV)
    payload, meta = sz.sz_encode(xd, cb, payload=payload, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    m = sz.read_meta(meta)
    assert m.status == 0 and m.as_tuple() == om.as_tuple()
    step = 1 << 28
    for a in range(0, om.comp_bytes, step):
        b = min(a + step, om.comp_bytes)
        assert np.array_equal(payload[a:b].cpu().numpy(), opay[a:b]), f"payload bytes [{a}, {b})"
    del opay, ws
    torch.cuda.empty_cache()

    wd = sz.Workspace(DEV)
    out = sz.sz_decode(payload, meta, cb, n, workspace=wd)
    assert sz.sz_workspace_flags(wd.buf) == 0
    assert torch.equal(out.view(torch.int16), xd), "decode"
    del out

    slot = torch.empty_like(xd)
    slot.view(torch.uint8)[:m.comp_bytes].copy_(payload[:m.comp_bytes])
    del payload
    sz.sz_decode_inplace(slot, meta, cb, workspace=wd)
    assert sz.sz_workspace_flags(wd.buf) == 0
    assert torch.equal(slot, xd), "in-place decode"
    del slot, xd, wd
    torch.cuda.empty_cache()


def test_max_item_count_round_trip_and_in_place():
    """SZ_MANY_MAX_ITEMS (65,535) tensors in one table: 1 to 4,000 elements
    each (some at tile edges, a few of one element). Separate calls, the fused
    calibrate + encode and the gated encode give every codebook, meta, payload
    and report the oracle gives; every decode and in-place decode is exact."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)
    count = B.SZ_MANY_MAX_ITEMS
    rng = np.random.default_rng(91)
    sizes = rng.integers(1, 4_000, count)
    sizes[::97] = 8192
    sizes[1::97] = 8193
    sizes[2::997] = 1
    offs = np.concatenate([[0], np.cumsum((sizes + 7) // 8 * 8)])  # 16-byte aligned views
    flat = np.zeros(int(offs[-1]), np.uint16)
    for i in range(0, count, 4096):  # a few distributions, changing along the table
        j = min(count, i + 4096)
        a, b = int(offs[i]), int(offs[j])
        flat[a:b] = inputs.gaussian(b - a, float(10 ** rng.uniform(-3, 0.5)), seed=100 + i)
        heavy = rng.random(b - a) < rng.uniform(0, 0.05)
        flat[a:b][heavy] = inputs.edge_case(b - a, seed=200 + i)[heavy]
    arrays = [flat[offs[i]:offs[i] + sizes[i]] for i in range(count)]
    dflat = torch.from_numpy(flat.view(np.int16)).to(DEV)
    views = [dflat[int(offs[i]):int(offs[i]) + int(sizes[i])] for i in range(count)]
    b = sz.Batch(views)
    ws = sz.Workspace(DEV)
    sz.sz_calibrate_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    sz.sz_encode_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    sz.sz_decode_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    cbs = b.codebooks.cpu().numpy()
    metas = b.metas.cpu().numpy()
    pay = b.payload.cpu().numpy()
    out = b.out.view(torch.int16).cpu().numpy().view(np.uint16)
    om_list, ocbs = [], []
    for i, x in enumerate(arrays):
        ocb = oracle.calibrate(x)
        check_codebook(sz.codebook_from_bytes(cbs[i]), ocb, x.size)
        opay, om = oracle.encode(x, ocb)
        m = sz.meta_from_bytes(metas[i])
        assert m.status == 0 and m.as_tuple() == om.as_tuple(), i
        po = b.payload_off[i]
        assert np.array_equal(pay[po:po + om.comp_bytes], opay), f"payload {i}"
        oo = b.out_off[i] // 2
        assert np.array_equal(out[oo:oo + x.size], x), f"decode {i}"
        om_list.append((opay, om))
        ocbs.append(ocb)

    # in place: every tensor whose payload fits its slot, slots packed in one buffer
    fit = [i for i, (_, om) in enumerate(om_list) if om.comp_bytes <= 2 * arrays[i].size]
    soffs = np.concatenate([[0], np.cumsum([(sizes[i] + 7) // 8 * 8 for i in fit])])
    host_slots = np.full(int(soffs[-1]), 0x5A5A, np.uint16)
    for k, i in enumerate(fit):
        opay, om = om_list[i]
        host_slots[soffs[k]:soffs[k] + sizes[i]].view(np.uint8)[:om.comp_bytes] = opay
    dslots = torch.from_numpy(host_slots.view(np.int16)).to(DEV)
    slots = [dslots[int(soffs[k]):int(soffs[k]) + int(sizes[i])] for k, i in enumerate(fit)]
    t = sz.slot_table(slots, [b.codebooks[i] for i in fit], [b.metas[i] for i in fit])
    sz.sz_decode_inplace_many(t, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    back = dslots.cpu().numpy().view(np.uint16)
    for k, i in enumerate(fit):
        assert np.array_equal(back[soffs[k]:soffs[k] + sizes[i]], arrays[i]), f"slot of tensor {i}"
    assert len(fit) > count // 2

    # the fused calibrate + encode over the same table
    fus = sz.Batch(views)
    sz.sz_calibrate_encode_many(fus.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    fcbs, fmetas, fpay = fus.codebooks.cpu().numpy(), fus.metas.cpu().numpy(), fus.payload.cpu().numpy()
    for i, x in enumerate(arrays):
        opay, om = om_list[i]
        check_codebook(sz.codebook_from_bytes(fcbs[i]), ocbs[i], x.size)
        assert sz.meta_from_bytes(fmetas[i]).as_tuple() == om.as_tuple(), f"fused meta {i}"
        po = fus.payload_off[i]
        assert np.array_equal(fpay[po:po + om.comp_bytes], opay), f"fused payload {i}"
    del fus, fpay

    # the coverage gate at 0.99, with its report
    g = sz.Batch(views)
    sz.sz_calibrate_many(g.table, workspace=ws)
    report = sz.sz_encode_gated_many(g.table, 0.99, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    gmetas = g.metas.cpu().numpy()
    gpay = g.payload.cpu().numpy()
    for i, x in enumerate(arrays):
        opay, om = om_list[i]
        m = sz.meta_from_bytes(gmetas[i])
        if oracle.gated(ocbs[i].coverage, 0.99):
            assert m.status == B.SZ_META_GATED and m.comp_bytes == 0, f"gated meta {i}"
        else:
            assert m.status == 0 and m.as_tuple() == om.as_tuple(), f"gated-call meta {i}"
            po = g.payload_off[i]
            assert np.array_equal(gpay[po:po + om.comp_bytes], opay), f"gated-call payload {i}"
    expect = oracle.gate_report([x.size for x in arrays], [c.coverage for c in ocbs], [om for _, om in om_list], 0.99)
    assert sz.read_gate_report(report) == expect
    assert 0 < expect["tensors_gated"] < count
