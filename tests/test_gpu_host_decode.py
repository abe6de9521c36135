"""sz_decode_many_host: payloads in pinned host memory, copied in groups
through a device staging buffer and decoded on the GPU."""
from __future__ import annotations

import numpy as np
import pytest
import torch

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


def _encoded(arrays):
    b = sz.Batch([to_dev(a) for a in arrays])
    sz.sz_calibrate_many(b.table)
    sz.sz_encode_many(b.table)
    torch.cuda.synchronize()
    metas = [sz.meta_from_bytes(b.metas[i].cpu().numpy()) for i in range(len(arrays))]
    return b, metas


def _host_blob(b, metas):
    """The whole payload buffer in one pinned host tensor (payloads back to
    back at 256-byte offsets, as in a packed blob) and a view per tensor."""
    blob = b.payload.cpu().pin_memory()
    views = [blob[o:o + m.comp_bytes] for o, m in zip(b.payload_off, metas)]
    return blob, views


def _decode_from_host(payloads, metas, b, staging_bytes):
    outs = [torch.full((n,), 7, dtype=torch.int16, device=DEV) for n in b.n]
    hd = sz.HostDecode(payloads, metas, [b.codebooks[i] for i in range(len(metas))], outs, staging_bytes)
    hd.run()
    flags = hd.flags()
    torch.cuda.synchronize()
    return outs, flags, hd


@pytest.mark.parametrize("staging_mib", [16, 64])
def test_host_decode_kv_groups(staging_mib):
    arrays = [inputs.kv_cache_tensor(l, kv) for l in range(2) for kv in range(2)]
    b, metas = _encoded(arrays)
    blob, views = _host_blob(b, metas)
    outs, flags, _ = _decode_from_host(views, metas, b, staging_mib << 20)
    assert flags == 0
    for x, y in zip(arrays, outs):
        assert np.array_equal(to_np_u16(y), x)


def test_host_decode_many_small_tensors_few_copies():
    arrays = [inputs.paged_kv_block(i) for i in range(2000)] + [inputs.edge_case(5000, seed=60), np.zeros(0, np.uint16)]
    b, metas = _encoded(arrays)
    blob, views = _host_blob(b, metas)
    outs, flags, hd = _decode_from_host(views, metas, b, 1 << 20)  # ~40 tensors per group
    assert flags == 0
    for x, y in zip(arrays, outs):
        assert np.array_equal(to_np_u16(y), x)


def test_host_decode_scattered_payloads():
    arrays = [inputs.gaussian(n, 0.02, seed=61 + n) for n in (1, 8193, 300_001, 77)]
    b, metas = _encoded(arrays)
    views = [b.payload_view(i, m.comp_bytes).cpu().pin_memory() for i, m in enumerate(metas)]  # one allocation each
    outs, flags, _ = _decode_from_host(views, metas, b, 1 << 20)
    assert flags == 0
    for x, y in zip(arrays, outs):
        assert np.array_equal(to_np_u16(y), x)


def test_host_decode_flags_and_gated_tensors():
    arrays = [inputs.gaussian(20_000, 0.02, seed=70), inputs.edge_case(20_000, seed=71),
              inputs.gaussian(30_000, 0.02, seed=72)]
    b = sz.Batch([to_dev(a) for a in arrays])
    sz.sz_calibrate_many(b.table)
    sz.sz_encode_gated_many(b.table, 0.99)  # the escape-heavy tensor is kept raw
    torch.cuda.synchronize()
    metas = [sz.meta_from_bytes(b.metas[i].cpu().numpy()) for i in range(3)]
    assert metas[1].status == B.SZ_META_GATED and metas[1].comp_bytes == 0
    import dataclasses

    metas[2] = dataclasses.replace(metas[2], off_sm=metas[2].off_sm + 4)  # disagrees with the layout
    blob, views = _host_blob(b, metas)
    outs, flags, _ = _decode_from_host(views, metas, b, 1 << 20)
    assert flags & B.SZ_FLAG_META
    assert np.array_equal(to_np_u16(outs[0]), arrays[0])
    assert torch.all(outs[1] == 7) and torch.all(outs[2] == 7)


def test_host_decode_rejects_a_small_staging_buffer():
    arrays = [inputs.gaussian(500_000, 0.02, seed=73)]
    b, metas = _encoded(arrays)
    blob, views = _host_blob(b, metas)
    with pytest.raises(B.SplitZipError):
        sz.HostDecode(views, metas, [b.codebooks[0]], [torch.empty(500_000, dtype=torch.int16, device=DEV)],
                      metas[0].comp_bytes)  # each half smaller than the payload


def test_host_decode_runs_back_to_back_and_allocates_nothing():
    """Repeated runs alternate the two pinned upload buffers; after the first
    run the calls change neither the device's free memory nor torch's
    allocations (the library allocates nothing and releases its events)."""
    arrays = [inputs.paged_kv_block(i) for i in range(300)]
    b, metas = _encoded(arrays)
    blob, views = _host_blob(b, metas)
    outs, flags, hd = _decode_from_host(views, metas, b, 1 << 20)
    assert flags == 0
    torch.cuda.synchronize()
    free0, allocated0 = torch.cuda.mem_get_info(DEV)[0], torch.cuda.memory_allocated(DEV)
    for _ in range(6):
        for y in outs:
            y.fill_(7)
        hd.run()
    assert hd.flags() == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(DEV)[0] == free0 and torch.cuda.memory_allocated(DEV) == allocated0
    for x, y in zip(arrays, outs):
        assert np.array_equal(to_np_u16(y), x)


def test_host_decode_rejects_pageable_or_short_upload_buffers():
    arrays = [inputs.gaussian(20_000, 0.02, seed=74), inputs.gaussian(3000, 0.02, seed=75)]
    b, metas = _encoded(arrays)
    blob, views = _host_blob(b, metas)
    outs = [torch.empty(n, dtype=torch.int16, device=DEV) for n in b.n]
    hd = sz.HostDecode(views, metas, [b.codebooks[i] for i in range(2)], outs, 1 << 20)
    lib = B.lib()
    need = lib.sz_decode_many_host_upload_bytes(2)
    s = torch.cuda.current_stream().cuda_stream
    pageable = torch.empty(need, dtype=torch.uint8)
    assert not pageable.is_pinned()

    def call(up, nbytes):
        return lib.sz_decode_many_host(hd.items, hd.metas, 2, hd.staging.data_ptr(), hd.staging.numel(),
                                       hd.scratch.data_ptr(), hd.scratch.numel(), up, nbytes, s,
                                       hd.copy_stream.cuda_stream)

    assert call(pageable.data_ptr(), need) == B.SZ_ERR_ARG
    pinned = torch.empty(need, dtype=torch.uint8).pin_memory()
    assert call(pinned.data_ptr(), need - 1) == B.SZ_ERR_WORKSPACE
    assert call(None, need) == B.SZ_ERR_ARG
    assert call(pinned.data_ptr(), need) == B.SZ_OK
    torch.cuda.synchronize()
    assert hd.flags() == 0
    for x, y in zip(arrays, outs):
        assert np.array_equal(to_np_u16(y), x)
