"""Calibration parity across the calibrate kernel's hand-over paths.

Each CTA of the calibrate kernel counts a contiguous run of tiles and, at each
tensor change, either ranks a tensor it counted whole or adds its counts to the
tensor's global histogram, the last CTA to add ranking it.  These cases cover:
- long tensors counted whole by one CTA;
- tensors split over CTAs at ragged points;
- long runs of one- and two-tile tensors, ragged and empty ones mixed in.
Each codebook is compared with the oracle's.

The item tables point several items at the same device tensor: calibration only
reads x, and the oracle's codebook is computed once per distinct tensor.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import weight_compression_codec_gb300 as sz
from weight_compression_codec_gb300 import binding as B
from weight_compression_codec_gb300 import inputs

from gpu_util import DEV, check_codebook, to_dev

pytestmark = pytest.mark.gpu

TILE = 8192


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    torch.cuda.set_device(DEV)


def _ctas() -> int:
    """Persistent CTAs of the calibrate kernel: two per SM."""
    return 2 * torch.cuda.get_device_properties(DEV).multi_processor_count


def _calibrate_reused(bases: list[np.ndarray], pick: list[int]) -> None:
    """Calibrates items i -> bases[pick[i]] in one sz_calibrate_many call and
    checks every codebook against the oracle's for its base tensor."""
    xd = [to_dev(b) for b in bases]
    count = len(pick)
    cbs = torch.empty((count, B.CODEBOOK_BYTES), dtype=torch.uint8, device=DEV)
    items = sz.make_items([bases[p].size for p in pick], x=[xd[p] for p in pick],
                          codebook=[cbs[i] for i in range(count)])
    table = sz.ItemTable(items, DEV)
    ws = sz.Workspace(DEV)
    sz.sz_calibrate_many(table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    host = cbs.cpu().numpy()
    ocbs = [oracle.calibrate(b) for b in bases]
    for i, p in enumerate(pick):
        check_codebook(sz.codebook_from_bytes(host[i]), ocbs[p], bases[p].size)


def _bases(n: int, sigmas=(0.02, 0.3, 1e-3, 4.0)) -> list[np.ndarray]:
    return [inputs.gaussian(n, s, seed=10 + i) for i, s in enumerate(sigmas)]


def test_long_tensors_counted_whole_by_one_cta():
    # 2 tensors of 300 tiles per CTA: each counted whole by one CTA and handed
    # to its select warp without the global histogram
    R = _ctas()
    bases = _bases(300 * TILE)
    _calibrate_reused(bases, [i % 4 for i in range(2 * R)])


def test_tensors_split_over_ctas():
    # ragged 900-tile tensors over ~590-tile CTA ranges: runs that start or end
    # inside a tensor, merged through the global histogram
    R = _ctas()
    bases = _bases(900 * TILE - 77)
    _calibrate_reused(bases, [(3 * i) % 4 for i in range(2 * R // 3)])


def test_runs_of_one_and_two_tile_tensors():
    # a tensor change every one or two tiles, with ragged and empty ones mixed in
    sizes = [TILE, 2 * TILE, 5, TILE + 1, 0, 2 * TILE - 3, 1]
    bases = [inputs.gaussian(n, 0.05 * (1 + i), seed=30 + i) if n else np.zeros(0, np.uint16)
             for i, n in enumerate(sizes)]
    rng = np.random.default_rng(7)
    pick = rng.integers(0, len(sizes), size=6 * _ctas()).tolist()
    xd = [to_dev(b) if b.size else torch.empty(8, dtype=torch.int16, device=DEV) for b in bases]
    count = len(pick)
    cbs = torch.empty((count, B.CODEBOOK_BYTES), dtype=torch.uint8, device=DEV)
    items = sz.make_items([sizes[p] for p in pick], x=[xd[p] for p in pick],
                          codebook=[cbs[i] for i in range(count)])
    table = sz.ItemTable(items, DEV)
    ws = sz.Workspace(DEV)
    sz.sz_calibrate_many(table, workspace=ws)
    assert sz.sz_workspace_flags(ws.buf) == 0
    torch.cuda.synchronize()
    host = cbs.cpu().numpy()
    ocbs = [oracle.calibrate(b) for b in bases]
    for i, p in enumerate(pick):
        check_codebook(sz.codebook_from_bytes(host[i]), ocbs[p], sizes[p])
