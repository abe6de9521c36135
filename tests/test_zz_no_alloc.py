"""sz_decode_noalloc: decode for callers that cannot allocate device memory when
they decode (a framework that owns all device memory, or a latency-critical
path that must not call cudaMalloc).  It keeps its scratch in a fixed array
inside the library instead of taking a workspace.

Checked through the C ABI against sz_decode (which takes a caller workspace):
identical output on two calls in a row (the second reuses the array the first
left behind), the status word reported through d_flags, the size limit, a
tensor of exactly the largest size it takes, and that calls leave the device's
free memory and torch's allocations unchanged.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)
    return B.lib()


def _encoded(x: np.ndarray):
    xd = torch.from_numpy(x.view(np.int16)).to(DEV)
    cb = sz.sz_calibrate(xd)
    payload, meta = sz.sz_encode(xd, cb)
    return payload, meta, cb


def _noalloc(lib, payload, meta, cb, n, out, flags):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.sz_decode_noalloc(payload.data_ptr(), payload.numel(), meta.data_ptr(), cb.data_ptr(),
                                 out.data_ptr() if n else None, n, flags.data_ptr(), stream)


def test_noalloc_decode_matches_workspace_decode_twice(lib):
    cases = [inputs.gaussian(3 * 8192 + 555, 0.02, seed=21), inputs.edge_case(40_001, seed=22)]
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    for x in cases:  # two calls in a row; the second finds the first one's scratch contents
        payload, meta, cb = _encoded(x)
        ref = sz.sz_decode(payload, meta, cb, x.size)
        out = torch.full((x.size,), 7, dtype=torch.int16, device=DEV)
        flags.fill_(-1)
        assert _noalloc(lib, payload, meta, cb, x.size, out, flags) == B.SZ_OK
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        assert torch.equal(out, ref.view(torch.int16))
        assert np.array_equal(out.cpu().numpy().view(np.uint16), x)


def test_noalloc_reports_device_flags_and_recovers(lib):
    x = inputs.gaussian(20_000, 1.0, seed=23)
    payload, meta, cb = _encoded(x)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = sz.read_meta(meta)
    import dataclasses

    bad_meta = torch.frombuffer(bytearray(sz.meta_to_bytes(dataclasses.replace(bad, off_sm=bad.off_sm + 4))),
                                dtype=torch.uint8).to(DEV)
    out = torch.full((x.size,), 7, dtype=torch.int16, device=DEV)
    assert _noalloc(lib, payload, bad_meta, cb, x.size, out, flags) == B.SZ_OK
    torch.cuda.synchronize()
    assert int(flags.item()) & B.SZ_FLAG_META and torch.all(out == 7)
    # the next call starts from a clean status word
    assert _noalloc(lib, payload, meta, cb, x.size, out, flags) == B.SZ_OK
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), x)


def test_noalloc_rejects_tensors_over_the_limit(lib):
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: the call returns before any launch
    assert lib.sz_decode_noalloc(p, 1 << 40, p, p, p, B.SZ_NOALLOC_MAX_ELEMS + 1, None, None) == B.SZ_ERR_ARG


def test_noalloc_at_the_size_limit_decodes_the_oracle_payload(lib):
    """n = SZ_NOALLOC_MAX_ELEMS exactly, with escapes in the last tile: the
    oracle's payload (written by the CPU codec, not by this library) decodes
    bit for bit."""
    n = B.SZ_NOALLOC_MAX_ELEMS
    x = inputs.gaussian(n, 0.02, seed=24)
    x[-8192::37] = inputs.edge_case(x[-8192::37].size, seed=25)  # escapes in the last tile
    ocb = oracle.calibrate(x)
    opay, om = oracle.encode(x, ocb)
    assert om.n_esc > 0 and om.n == n
    payload = torch.from_numpy(np.concatenate([opay, np.zeros(16, np.uint8)])).to(DEV)
    meta = torch.frombuffer(bytearray(sz.meta_to_bytes(om)), dtype=torch.uint8).to(DEV)
    cb = torch.frombuffer(bytearray(_oracle_codebook(ocb, n)), dtype=torch.uint8).to(DEV)
    out = torch.empty(n, dtype=torch.int16, device=DEV)
    flags = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    assert _noalloc(lib, payload, meta, cb, n, out, flags) == B.SZ_OK
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    y = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(y[-8192:], x[-8192:]), "last tile"
    assert np.array_equal(y, x)


def test_noalloc_calls_allocate_nothing(lib):
    """After a first call (which looks up the array's address), further calls
    change neither the device's free memory nor torch's allocations."""
    x = inputs.edge_case(3 * 8192 + 17, seed=26)
    payload, meta, cb = _encoded(x)
    out = torch.empty(x.size, dtype=torch.int16, device=DEV)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _noalloc(lib, payload, meta, cb, x.size, out, flags) == B.SZ_OK
    torch.cuda.synchronize()
    free0, allocated0 = torch.cuda.mem_get_info(DEV)[0], torch.cuda.memory_allocated(DEV)
    for _ in range(5):
        assert _noalloc(lib, payload, meta, cb, x.size, out, flags) == B.SZ_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(DEV)[0] == free0
    assert torch.cuda.memory_allocated(DEV) == allocated0
    assert int(flags.item()) == 0 and np.array_equal(out.cpu().numpy().view(np.uint16), x)


def _oracle_codebook(ocb, n: int) -> bytes:
    c = B.SzCodebook()
    c.enc_lut[:] = list(ocb.enc_lut)
    c.dec_lut[:] = list(ocb.dec_lut)
    c.n_top = ocb.n_top
    c.top_count = ocb.top_count
    c.n = n
    c.coverage = ocb.coverage
    return bytes(c)
