"""Seeded random batches through the whole path, every result against the oracle.

Each batch draws:
- a tensor count;
- sizes: empty, tiny, around chunk and tile edges, or up to a few hundred
  thousand elements;
- value distributions: Gaussians of any scale, escape-heavy bit patterns,
  mixtures of the two, constant tensors and uniform bit patterns.

Some tensors are encoded with a codebook calibrated on another tensor of the
batch, which forces escapes.  The batch is calibrated, encoded, decoded out of
place, and decoded in place for the tensors whose payload fits their raw size.
Other batches go through the fused calibrate + encode, the decode from pinned
host memory and the coverage gate.  Every codebook, meta, payload, report and
decode is compared with the oracle.
"""
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

EDGE_SIZES = [0, 1, 2, 3, 5, 1023, 1024, 1025, 4095, 4096, 8191, 8192, 8193, 16383, 16384, 16385, 24577, 65536]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)


def _tensor(rng: np.random.Generator, n: int, seed: int) -> np.ndarray:
    kind = int(rng.integers(0, 5))
    if n == 0:
        return np.zeros(0, np.uint16)
    if kind == 0:
        return inputs.gaussian(n, float(10 ** rng.uniform(-3, 1)), seed=seed)
    if kind == 1:
        return inputs.edge_case(n, seed=seed)
    if kind == 2:
        x = inputs.gaussian(n, 0.05, seed=seed)
        mask = rng.random(n) < rng.uniform(0.0, 0.3)
        x[mask] = inputs.edge_case(n, seed=seed + 1)[mask]
        return x
    if kind == 3:
        return np.full(n, int(rng.integers(0, 65536)), dtype=np.uint16)
    return rng.integers(0, 65536, n, dtype=np.uint16)  # every exponent occurs


def _batch(seed: int) -> list[np.ndarray]:
    rng = np.random.default_rng(1000 + seed)
    count = int(rng.integers(1, 25))
    sizes = [int(rng.choice(EDGE_SIZES)) if rng.random() < 0.6 else int(rng.integers(1, 300_000))
             for _ in range(count)]
    return [_tensor(rng, n, seed * 100 + i) for i, n in enumerate(sizes)]


@pytest.mark.parametrize("seed", range(16))
def test_random_batch_matches_oracle(seed):
    arrays = _batch(seed)
    count = len(arrays)
    b = sz.Batch([to_dev(a) if a.size else torch.empty(0, dtype=torch.int16, device=DEV) for a in arrays])
    ws = sz.Workspace(DEV)
    sz.sz_calibrate_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    ocbs = [oracle.calibrate(a) for a in arrays]
    cbs = b.codebooks.cpu().numpy()
    for i, a in enumerate(arrays):
        check_codebook(sz.codebook_from_bytes(cbs[i]), ocbs[i], a.size)

    # a third of the tensors take another tensor's codebook: row i copies row
    # j as it is now, which may already hold a third tensor's codebook
    rng = np.random.default_rng(2000 + seed)
    use = list(range(count))  # use[i]: the tensor whose oracle codebook row i holds
    for i in range(count):
        if count > 1 and rng.random() < 1 / 3:
            j = int(rng.integers(0, count))
            b.codebooks[i].copy_(b.codebooks[j])
            use[i] = use[j]
    sz.sz_encode_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    sz.sz_decode_many(b.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    metas = b.metas.cpu().numpy()
    expect = []
    for i, a in enumerate(arrays):
        opay, om = oracle.encode(a, ocbs[use[i]])
        m = sz.meta_from_bytes(metas[i])
        assert m.status == 0 and m.as_tuple() == om.as_tuple(), (seed, i, m, om)
        assert np.array_equal(b.payload_view(i, m.comp_bytes).cpu().numpy(), opay), f"payload {i}"
        assert np.array_equal(to_np_u16(b.out_view(i)), a), f"decode {i}"
        expect.append((opay, om))

    # in place, for every tensor whose payload fits its raw size
    fit = [i for i, (_, om) in enumerate(expect) if om.comp_bytes <= 2 * arrays[i].size]
    if not fit:
        return
    gen = torch.Generator(device=DEV).manual_seed(seed)
    slots = []
    for i in fit:
        s = torch.randint(-32768, 32767, (arrays[i].size,), dtype=torch.int16, device=DEV, generator=gen)
        om = expect[i][1]
        s.view(torch.uint8)[:om.comp_bytes].copy_(b.payload_view(i, om.comp_bytes))
        slots.append(s)
    t = sz.slot_table(slots, [b.codebooks[i] for i in fit], [b.metas[i] for i in fit])
    sz.sz_decode_inplace_many(t, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    for k, i in enumerate(fit):
        assert np.array_equal(to_np_u16(slots[k]), arrays[i]), f"slot of tensor {i}"


@pytest.mark.parametrize("seed", range(8))
def test_random_batch_fused_from_host_and_gated(seed):
    arrays = _batch(100 + seed)
    count = len(arrays)
    ocbs = [oracle.calibrate(a) for a in arrays]
    oenc = [oracle.encode(a, c) for a, c in zip(arrays, ocbs)]
    devs = [to_dev(a) if a.size else torch.empty(0, dtype=torch.int16, device=DEV) for a in arrays]
    ws = sz.Workspace(DEV)

    # fused calibrate + encode
    fus = sz.Batch(devs)
    sz.sz_calibrate_encode_many(fus.table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    cbs = fus.codebooks.cpu().numpy()
    metas = [sz.meta_from_bytes(fus.metas[i].cpu().numpy()) for i in range(count)]
    for i, a in enumerate(arrays):
        check_codebook(sz.codebook_from_bytes(cbs[i]), ocbs[i], a.size)
        opay, om = oenc[i]
        assert metas[i].status == 0 and metas[i].as_tuple() == om.as_tuple(), (seed, i)
        assert np.array_equal(fus.payload_view(i, om.comp_bytes).cpu().numpy(), opay), f"fused payload {i}"

    # decode from pinned host memory, the payloads back to back in one blob
    blob = fus.payload.cpu().pin_memory()
    views = [blob[o:o + m.comp_bytes] for o, m in zip(fus.payload_off, metas)]
    outs = [torch.full((a.size,), 7, dtype=torch.int16, device=DEV) for a in arrays]
    staging = max(4 * max(m.comp_bytes for m in metas), 1 << 20)
    hd = sz.HostDecode(views, metas, [fus.codebooks[i] for i in range(count)], outs, staging)
    hd.run()
    assert hd.flags() == 0
    torch.cuda.synchronize()
    for i, a in enumerate(arrays):
        assert np.array_equal(to_np_u16(outs[i]), a), f"decode from host {i}"

    # coverage gate at a random threshold
    gate = float(np.random.default_rng(3000 + seed).uniform(0.2, 1.0))
    g = sz.Batch(devs)
    g.payload.fill_(0x5A)
    sz.sz_calibrate_many(g.table, workspace=ws)
    report = sz.sz_encode_gated_many(g.table, gate, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    for i, a in enumerate(arrays):
        m = sz.meta_from_bytes(g.metas[i].cpu().numpy())
        opay, om = oenc[i]
        if oracle.gated(ocbs[i].coverage, gate):
            assert m.status == B.SZ_META_GATED and m.comp_bytes == 0, (seed, i)
            assert bool(torch.all(g.payload_view(i) == 0x5A)), f"gated tensor {i}: payload written"
        else:
            assert m.status == 0 and m.as_tuple() == om.as_tuple(), (seed, i)
            assert np.array_equal(g.payload_view(i, om.comp_bytes).cpu().numpy(), opay), f"gated payload {i}"
    expect = oracle.gate_report([a.size for a in arrays], [c.coverage for c in ocbs], [om for _, om in oenc], gate)
    assert sz.read_gate_report(report) == expect


@pytest.mark.parametrize("seed", range(12))
def test_inplace_random_sizes_and_escape_rates(seed):
    """In-place decode of the oracle's payloads: tensors of up to ~730 tiles,
    with escape rates up to what still fits the slot (comp_bytes <= 2n), so the
    three decode phases and the stash take every proportion."""
    from gpu_util import oracle_codebook_bytes

    rng = np.random.default_rng(4000 + seed)
    count = int(rng.integers(1, 7))
    arrays, slots, cbs, metas = [], [], [], []
    while len(arrays) < count:
        k = len(arrays)
        n = int(rng.integers(1, 6_000_000)) if rng.random() < 0.7 else \
            max(1, int(rng.integers(1, 40)) * 8192 + int(rng.integers(-2, 3)))
        x = inputs.gaussian(n, 0.02, seed=seed * 10 + k)
        mask = rng.random(n) < rng.uniform(0.0, 0.12)
        x[mask] = inputs.edge_case(n, seed=seed * 10 + k)[mask]
        cb = oracle.calibrate(x)
        pay, m = oracle.encode(x, cb)
        if m.comp_bytes > 2 * n:
            continue  # an expanding tensor cannot sit in its slot
        s = torch.randint(-32768, 32767, (n,), dtype=torch.int16, device=DEV)
        s.view(torch.uint8)[:m.comp_bytes].copy_(torch.from_numpy(pay).to(DEV))
        arrays.append(x)
        slots.append(s)
        cbs.append(torch.frombuffer(bytearray(oracle_codebook_bytes(cb, n)), dtype=torch.uint8).to(DEV))
        metas.append(torch.frombuffer(bytearray(sz.meta_to_bytes(m)), dtype=torch.uint8).to(DEV))
    t = sz.slot_table(slots, cbs, metas)
    ws = sz.Workspace(DEV)
    sz.sz_decode_inplace_many(t, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    for k, x in enumerate(arrays):
        assert np.array_equal(to_np_u16(slots[k]), x), f"slot {k} (n = {x.size})"
