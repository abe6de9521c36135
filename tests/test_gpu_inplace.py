"""sz_decode_inplace(_many): a payload held in the leading bytes of the tensor's
own BF16 buffer (its slot, "splitzip_codec.py" GpuSplitZipDecoder) decoded
over that buffer, against the oracle's slot decode."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

from gpu_util import DEV, oracle_codebook_bytes, to_dev, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)


def _dev_bytes(b: bytes) -> torch.Tensor:
    return torch.frombuffer(bytearray(b), dtype=torch.uint8).to(DEV)


def _slot_case(x: np.ndarray, seed: int):
    """The oracle's payload in a slot of random bytes, and the oracle's slot decode of it."""
    ocb = oracle.calibrate(x)
    opay, om = oracle.encode(x, ocb)
    assert om.comp_bytes <= 2 * x.size, "test input does not fit its slot"
    slot_np = np.random.default_rng(seed).integers(0, 256, 2 * x.size, dtype=np.uint8)
    slot_np[:om.comp_bytes] = opay
    expect = oracle.decode_slot(slot_np.copy(), om, ocb.dec_lut)
    slot = torch.from_numpy(slot_np.view(np.int16)).to(DEV)
    return slot, _dev_bytes(sz.meta_to_bytes(om)), _dev_bytes(oracle_codebook_bytes(ocb, x.size)), expect, om


def _exact_escapes(n: int, e: int, seed: int) -> np.ndarray:
    """n values whose Top-16 exponents are 100..115 (equal shares) and whose e
    other elements spread over the 240 remaining exponents, fewer per value
    than any Top-16 share: exactly e escapes."""
    rng = np.random.default_rng(seed)
    exp = np.repeat(np.arange(100, 116, dtype=np.uint16), -(-(n - e) // 16))[:n - e]
    others = np.concatenate([np.arange(0, 100), np.arange(116, 256)]).astype(np.uint16)
    esc = others[np.arange(e) % others.size]
    assert (n - e) // 16 > -(-e // others.size)
    allexp = np.concatenate([exp, esc])
    rng.shuffle(allexp)
    low = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16) & np.uint16(0x807F)
    return (allexp << np.uint16(7)) | low


def _single(x: np.ndarray, seed: int) -> None:
    slot, meta, cb, expect, om = _slot_case(x, seed)
    ws = sz.Workspace(DEV)
    sz.sz_decode_inplace(slot, meta, cb, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    got = slot.cpu().numpy().view(np.uint8)
    if not np.array_equal(got, expect):
        bad = np.nonzero(got != expect)[0]
        raise AssertionError(f"slot differs at {bad.size} bytes, first at {bad[:8]} ({om})")
    assert np.array_equal(got.view(np.uint16), x)


@pytest.mark.parametrize("n", [4, 8, 4099, 8192, 8193, 16384, 16385, 24577, 100_003, 1_000_001])
def test_inplace_gaussian_sizes(n):
    _single(inputs.gaussian(n, 0.02, seed=80 + n % 97), seed=n)


def test_inplace_kv_cache_tensor():
    _single(inputs.kv_cache_tensor(3, 1), seed=81)


@pytest.mark.parametrize("n,e", [(114_688, 8192), (114_688, 8190), (16_384, 1170), (1_400_000, 99_000)])
def test_inplace_largest_payloads_that_fit(n, e):
    # (114688, 8192): comp_bytes == 2n exactly, every slot byte is payload
    x = _exact_escapes(n, e, seed=n + e)
    m = oracle.layout(n, e)
    assert oracle.count_escapes(x, oracle.calibrate(x)) == e and m.comp_bytes <= 2 * n
    if (n, e) == (114_688, 8192):
        assert m.comp_bytes == 2 * n
    _single(x, seed=e)


def test_inplace_tile_with_thousands_of_escapes():
    # 3000 escapes in one tile: the tile's escapes arrive in three stages
    x = inputs.gaussian(60_000, 0.02, seed=82)
    broad = inputs.edge_case(3000, seed=83)
    x[8192:11192] = broad
    _single(x, seed=84)


def test_inplace_empty_tensor_and_repeated_calls():
    ws = sz.Workspace(DEV)
    x = inputs.gaussian(300_001, 0.02, seed=85)
    for rep in range(3):
        slot, meta, cb, expect, _ = _slot_case(x, seed=rep)
        sz.sz_decode_inplace(slot, meta, cb, workspace=ws)
        assert sz.sz_workspace_flags(ws.buf) == 0
        assert np.array_equal(slot.cpu().numpy().view(np.uint8), expect)
    empty = torch.empty(0, dtype=torch.int16, device=DEV)
    m0 = oracle.layout(0, 0, 1.0)
    sz.sz_decode_inplace(empty, _dev_bytes(sz.meta_to_bytes(m0)), _dev_bytes(oracle_codebook_bytes(
        oracle.calibrate(np.zeros(0, np.uint16)), 0)), workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0


def _encode_into_slots(arrays):
    """GPU calibrate + encode of the arrays, each payload copied into the
    leading bytes of a fresh slot of its raw size (random bytes after it)."""
    b = sz.Batch([to_dev(a) for a in arrays])
    sz.sz_calibrate_many(b.table)
    sz.sz_encode_many(b.table)
    torch.cuda.synchronize()
    metas = [sz.meta_from_bytes(b.metas[i].cpu().numpy()) for i in range(len(arrays))]
    gen = torch.Generator(device=DEV).manual_seed(7)
    slots = []
    for i, (a, m) in enumerate(zip(arrays, metas)):
        s = torch.randint(-32768, 32767, (a.size,), dtype=torch.int16, device=DEV, generator=gen)
        if m.comp_bytes <= 2 * a.size:
            s.view(torch.uint8)[:m.comp_bytes].copy_(b.payload_view(i, m.comp_bytes))
        slots.append(s)
    return b, metas, slots


def test_inplace_many_mixed_sizes_against_oracle():
    arrays = ([inputs.kv_cache_tensor(l, kv) for l in range(2) for kv in range(2)] +
              [inputs.gaussian(n, 0.02, seed=86 + n % 13) for n in (8192, 8193, 300_001, 4, 77_777)] +
              [np.zeros(0, np.uint16), _exact_escapes(114_688, 8192, seed=87)] +
              [inputs.paged_kv_block(i) for i in range(40)])
    b, metas, slots = _encode_into_slots(arrays)
    t = sz.slot_table(slots, [b.codebooks[i] for i in range(len(arrays))], [b.metas[i] for i in range(len(arrays))])
    ws = sz.Workspace(DEV)
    sz.sz_decode_inplace_many(t, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    for i, x in enumerate(arrays):
        assert np.array_equal(to_np_u16(slots[i]), x), f"slot {i}"
    # the oracle's slot decode of a sample gives the same bytes
    for i in (0, 5, 10, 20):
        ocb = oracle.calibrate(arrays[i])
        opay, om = oracle.encode(arrays[i], ocb)
        s = np.zeros(2 * arrays[i].size, np.uint8)
        s[:om.comp_bytes] = opay
        assert np.array_equal(oracle.decode_slot(s, om, ocb.dec_lut).view(np.uint16), to_np_u16(slots[i]))


def test_inplace_many_flags_expanded_gated_and_foreign_payload():
    # item 0: fine; item 1: n = 2 (payload 8 bytes > 4-byte slot) -> META, untouched;
    # item 2: kept raw by the gate -> untouched, no flag; item 3: payload not at the slot -> META
    arrays = [inputs.gaussian(50_000, 0.02, seed=88), np.array([0x3F80, 0x4000], np.uint16),
              inputs.edge_case(20_000, seed=89), inputs.gaussian(30_000, 0.02, seed=90)]
    b = sz.Batch([to_dev(a) for a in arrays])
    sz.sz_calibrate_many(b.table)
    sz.sz_encode_gated_many(b.table, 0.99)
    torch.cuda.synchronize()
    metas = [sz.meta_from_bytes(b.metas[i].cpu().numpy()) for i in range(4)]
    assert metas[1].comp_bytes == 8 and metas[2].status == B.SZ_META_GATED
    slots = [to_dev(arrays[0]).fill_(0), torch.full((2,), 5, dtype=torch.int16, device=DEV), to_dev(arrays[2]),
             torch.full((30_000,), 9, dtype=torch.int16, device=DEV)]
    slots[0].view(torch.uint8)[:metas[0].comp_bytes].copy_(b.payload_view(0, metas[0].comp_bytes))
    items = sz.make_items([a.size for a in arrays], out=slots,
                          payload=[slots[0], slots[1], slots[2], b.payload_view(3)],
                          capacity=[2 * a.size for a in arrays], codebook=[b.codebooks[i] for i in range(4)],
                          meta=[b.metas[i] for i in range(4)])
    t = sz.ItemTable(items, DEV)
    ws = sz.Workspace(DEV)
    sz.sz_decode_inplace_many(t, workspace=ws)
    flags = sz.sz_workspace_flags(ws.buf)
    torch.cuda.synchronize()
    assert flags == B.SZ_FLAG_META
    assert np.array_equal(to_np_u16(slots[0]), arrays[0])
    assert torch.all(slots[1] == 5) and torch.all(slots[3] == 9)
    assert np.array_equal(to_np_u16(slots[2]), arrays[2])


def test_inplace_kv_cache_full_size():
    # the 64 x 4 Mi-element KV cache: every slot decoded in place, exact
    arrays = inputs.kv_cache()
    b, metas, slots = _encode_into_slots(arrays)
    assert all(m.comp_bytes <= 2 * a.size for m, a in zip(metas, arrays))
    t = sz.slot_table(slots, [b.codebooks[i] for i in range(len(arrays))], [b.metas[i] for i in range(len(arrays))])
    ws = sz.Workspace(DEV)
    for rep in range(2):
        if rep:  # again, from freshly placed payloads with the same workspace
            for i, m in enumerate(metas):
                slots[i].view(torch.uint8)[:m.comp_bytes].copy_(b.payload_view(i, m.comp_bytes))
        sz.sz_decode_inplace_many(t, workspace=ws)
        assert sz.sz_workspace_flags(ws.buf) == 0
        torch.cuda.synchronize()
        for i in range(len(arrays)):
            assert torch.equal(slots[i], b.xs[i]), f"slot {i}"


def test_inplace_rejects_bad_arguments():
    lib = B.lib()
    s = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    slot = torch.empty(8192, dtype=torch.int16, device=DEV)
    meta = torch.empty(B.META_BYTES, dtype=torch.uint8, device=DEV)
    cb = torch.empty(B.CODEBOOK_BYTES, dtype=torch.uint8, device=DEV)
    assert lib.sz_decode_inplace(slot.data_ptr(), 8192, None, cb.data_ptr(), ws.data_ptr(), ws.numel(), s) == \
        B.SZ_ERR_ARG
    assert lib.sz_decode_inplace(slot.data_ptr() + 2, 8192, meta.data_ptr(), cb.data_ptr(), ws.data_ptr(),
                                 ws.numel(), s) == B.SZ_ERR_ALIGN
    need = lib.sz_decode_inplace_workspace_bytes(1, 1)
    assert lib.sz_decode_inplace(slot.data_ptr(), 8192, meta.data_ptr(), cb.data_ptr(), ws.data_ptr(), need - 1,
                                 s) == B.SZ_ERR_WORKSPACE
