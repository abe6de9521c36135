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
