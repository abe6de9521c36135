"""Failure detection on the GPU without a fault: every wait inside the kernels
is bounded, gives up with SZ_FLAG_TIMEOUT and leaves the context usable."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

from gpu_util import DEV, roundtrip_single

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)


def test_bounded_waits_give_up_and_leave_the_context_usable():
    # an mbarrier phase that never completes, a word one thread polls and
    # words a warp polls, none of them ever set: each wait must end on its own
    ws = torch.full((B.SZ_CHECK_WAITS_WORKSPACE_BYTES,), 0xAB, dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    rc = B.lib().sz_check_bounded_waits(ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == B.SZ_OK
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert sz.sz_workspace_flags(ws) == B.SZ_FLAG_TIMEOUT
    words = ws[256:272].cpu().numpy().view(np.uint32)
    assert words[0] == 0, "nothing ever set the word the waits watched"
    assert list(words[1:4]) == [1, 1, 1], "every kind of wait gave up"
    assert 1.0 < elapsed < 30.0, elapsed
    # the context is still usable: a full round trip and an in-place decode
    roundtrip_single(inputs.gaussian(100_003, 0.02, seed=96))
    x = inputs.kv_cache_tensor(1, 0)[:1_000_000]
    xd = torch.from_numpy(x.view(np.int16)).to(DEV)
    cb = sz.sz_calibrate(xd)
    payload, meta = sz.sz_encode(xd, cb)
    m = sz.read_meta(meta)
    slot = torch.empty_like(xd)
    slot.view(torch.uint8)[:m.comp_bytes].copy_(payload[:m.comp_bytes])
    sz.sz_decode_inplace(slot, meta, cb)
    torch.cuda.synchronize()
    assert torch.equal(slot, xd)


def test_bounded_waits_check_rejects_a_small_workspace():
    ws = torch.empty(B.SZ_CHECK_WAITS_WORKSPACE_BYTES, dtype=torch.uint8, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    assert B.lib().sz_check_bounded_waits(ws.data_ptr(), 256, s) == B.SZ_ERR_WORKSPACE
    assert B.lib().sz_check_bounded_waits(None, ws.numel(), s) == B.SZ_ERR_WORKSPACE
