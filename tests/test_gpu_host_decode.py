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
