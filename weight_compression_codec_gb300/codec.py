"""PyTorch-facing binding of the SplitZip codec.

The functions carry the C ABI's names (sz_calibrate, sz_encode, sz_decode and
the *_many variants) and only marshal arguments: they check dtype, device,
contiguity and alignment, allocate outputs and workspaces with torch (device
memory), pass raw pointers and the current CUDA stream to libsplitzip.so, and
return tensors.  Codebooks and metas stay on the device as uint8 tensors of
304 and 96 bytes (the sz_codebook / sz_meta structs); ``read_codebook`` and
``read_meta`` copy one to the host when needed.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import binding as B

_BF16_LIKE = (torch.bfloat16, torch.int16, torch.uint16)


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _bits(x: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if x.dtype not in _BF16_LIKE:
        raise ValueError(f"SplitZip expects bfloat16 data for {name}, got {x.dtype}")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return x.reshape(-1)


def _u8(t: torch.Tensor, name: str, nbytes: int | None = None) -> torch.Tensor:
    if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor")
    if nbytes is not None and t.numel() < nbytes:
        raise ValueError(f"{name} needs at least {nbytes} bytes, has {t.numel()}")
    return t


class Workspace:
    """A device scratch buffer that grows on demand (one per stream of use)."""

    def __init__(self, device: torch.device | str | None = None):
        self.device = torch.device(device) if device is not None else None
        self.buf: torch.Tensor | None = None

    def get(self, nbytes: int, device: torch.device) -> torch.Tensor:
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        return self.buf


_default_ws: dict = {}


def _workspace(ws, nbytes: int, device: torch.device) -> torch.Tensor:
    if isinstance(ws, torch.Tensor):
        return _u8(ws, "workspace", nbytes)
    if ws is None:
        ws = _default_ws.setdefault(device, Workspace(device))
    return ws.get(nbytes, device)


# ---------------------------------------------------------------------------- host views


@dataclass(frozen=True)
class Codebook:
    enc_lut: np.ndarray
    dec_lut: np.ndarray
    n_top: int
    top_count: int
    n: int
    coverage: float


@dataclass(frozen=True)
class Meta:
    n: int
    n_pairs: int
    n_esc: int
    comp_bytes: int
    off_pk: int
    off_sm: int
    off_cid: int
    off_lpos: int
    off_ev: int
    chunk_size: int
    status: int
    coverage: float

    def as_tuple(self) -> tuple:
        return (self.n, self.n_pairs, self.n_esc, self.comp_bytes, self.off_pk, self.off_sm,
                self.off_cid, self.off_lpos, self.off_ev, self.chunk_size)


def codebook_from_bytes(b) -> Codebook:
    c = B.SzCodebook.from_buffer_copy(bytes(np.asarray(b, dtype=np.uint8).tobytes()[:B.CODEBOOK_BYTES]))
    return Codebook(np.frombuffer(bytes(c.enc_lut), np.uint8).copy(), np.frombuffer(bytes(c.dec_lut), np.uint8).copy(),
                    int(c.n_top), int(c.top_count), int(c.n), float(c.coverage))


def meta_from_bytes(b) -> Meta:
    m = B.SzMeta.from_buffer_copy(bytes(np.asarray(b, dtype=np.uint8).tobytes()[:B.META_BYTES]))
    return Meta(int(m.n), int(m.n_pairs), int(m.n_esc), int(m.comp_bytes), int(m.off_pk), int(m.off_sm),
                int(m.off_cid), int(m.off_lpos), int(m.off_ev), int(m.chunk_size), int(m.status), float(m.coverage))


def meta_to_bytes(m) -> bytes:
    s = B.SzMeta()
    for f in ("n", "n_pairs", "n_esc", "comp_bytes", "off_pk", "off_sm", "off_cid", "off_lpos", "off_ev",
              "chunk_size"):
        setattr(s, f, int(getattr(m, f)))
    s.status = int(getattr(m, "status", 0))
    s.coverage = float(getattr(m, "coverage", 0.0))
    return bytes(s)


def read_codebook(cb: torch.Tensor) -> Codebook:
    return codebook_from_bytes(cb.reshape(-1)[:B.CODEBOOK_BYTES].cpu().numpy())


def read_meta(meta: torch.Tensor) -> Meta:
    return meta_from_bytes(meta.reshape(-1)[:B.META_BYTES].cpu().numpy())


# ---------------------------------------------------------------------------- host queries


def sz_tiles(n: int) -> int:
    return int(B.lib().sz_tiles(n))


def sz_layout(n: int, n_esc: int) -> Meta:
    m = B.SzMeta()
    B.check(B.lib().sz_layout(n, n_esc, ctypes.byref(m)), "sz_layout")
    return meta_from_bytes(np.frombuffer(bytes(m), np.uint8))


def sz_payload_bytes(n: int, n_esc: int) -> int:
    return int(B.lib().sz_payload_bytes(n, n_esc))


def sz_max_payload_bytes(n: int) -> int:
    return int(B.lib().sz_max_payload_bytes(n))


def sz_workspace_flags(workspace: torch.Tensor, stream=None) -> int:
    f = ctypes.c_uint32(0)
    rc = B.lib().sz_workspace_flags(ctypes.c_void_p(workspace.data_ptr()), ctypes.byref(f),
                                    ctypes.c_void_p(_stream_handle(stream)))
    if rc not in (B.SZ_OK, B.SZ_ERR_DEVICE):
        B.check(rc, "sz_workspace_flags")
    return int(f.value)


def sz_set_timing_events(before, after) -> None:
    """Record torch.cuda.Event `before`/`after` around the next main kernels (None clears)."""
    b = ctypes.c_void_p(before.cuda_event) if before is not None else None
    a = ctypes.c_void_p(after.cuda_event) if after is not None else None
    B.lib().sz_set_timing_events(b, a)


# ---------------------------------------------------------------------------- single tensor


def sz_calibrate(x: torch.Tensor, codebook: torch.Tensor | None = None, workspace=None, stream=None) -> torch.Tensor:
    """Top-16 exponent codebook of ``x`` (BF16, CUDA), as a 304-byte device tensor."""
    xb = _bits(x, "x")
    dev = xb.device
    if codebook is None:
        codebook = torch.empty(B.CODEBOOK_BYTES, dtype=torch.uint8, device=dev)
    _u8(codebook, "codebook", B.CODEBOOK_BYTES)
    need = B.lib().sz_calibrate_workspace_bytes(1)
    ws = _workspace(workspace, need, dev)
    rc = B.lib().sz_calibrate(xb.data_ptr(), xb.numel(), codebook.data_ptr(), ws.data_ptr(), ws.numel(),
                              _stream_handle(stream))
    B.check(rc, "sz_calibrate")
    return codebook


def sz_encode(x: torch.Tensor, codebook: torch.Tensor, payload: torch.Tensor | None = None,
              meta: torch.Tensor | None = None, workspace=None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Encode ``x`` with ``codebook`` (device tensors).  Returns (payload, meta) on the device;
    the payload buffer defaults to the worst-case size, the valid bytes are meta.comp_bytes."""
    xb = _bits(x, "x")
    dev = xb.device
    n = xb.numel()
    _u8(codebook, "codebook", B.CODEBOOK_BYTES)
    if payload is None:
        payload = torch.empty(max(sz_max_payload_bytes(n), 16), dtype=torch.uint8, device=dev)
    _u8(payload, "payload")
    if meta is None:
        meta = torch.empty(B.META_BYTES, dtype=torch.uint8, device=dev)
    _u8(meta, "meta", B.META_BYTES)
    need = B.lib().sz_encode_workspace_bytes(1, sz_tiles(n))
    ws = _workspace(workspace, need, dev)
    rc = B.lib().sz_encode(xb.data_ptr(), n, codebook.data_ptr(), payload.data_ptr(), payload.numel(),
                           meta.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(stream))
    B.check(rc, "sz_encode")
    return payload, meta


def sz_calibrate_encode(x: torch.Tensor, codebook: torch.Tensor | None = None, payload: torch.Tensor | None = None,
                        meta: torch.Tensor | None = None, workspace=None,
                        stream=None) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """sz_calibrate then sz_encode in one pass over HBM.  Returns (codebook, payload, meta)."""
    xb = _bits(x, "x")
    dev = xb.device
    n = xb.numel()
    if codebook is None:
        codebook = torch.empty(B.CODEBOOK_BYTES, dtype=torch.uint8, device=dev)
    _u8(codebook, "codebook", B.CODEBOOK_BYTES)
    if payload is None:
        payload = torch.empty(max(sz_max_payload_bytes(n), 16), dtype=torch.uint8, device=dev)
    _u8(payload, "payload")
    if meta is None:
        meta = torch.empty(B.META_BYTES, dtype=torch.uint8, device=dev)
    _u8(meta, "meta", B.META_BYTES)
    ws = _workspace(workspace, B.lib().sz_calibrate_encode_workspace_bytes(1, sz_tiles(n)), dev)
    rc = B.lib().sz_calibrate_encode(xb.data_ptr(), n, codebook.data_ptr(), payload.data_ptr(), payload.numel(),
                                     meta.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(stream))
    B.check(rc, "sz_calibrate_encode")
    return codebook, payload, meta


def sz_decode(payload: torch.Tensor, meta: torch.Tensor, codebook: torch.Tensor, n: int,
              out: torch.Tensor | None = None, workspace=None, stream=None) -> torch.Tensor:
    """Decode a payload (device tensors) into ``out`` (BF16, n elements)."""
    _u8(payload, "payload")
    _u8(meta, "meta", B.META_BYTES)
    _u8(codebook, "codebook", B.CODEBOOK_BYTES)
    dev = payload.device
    if out is None:
        out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    ob = _bits(out, "out")
    if ob.numel() != n:
        raise ValueError(f"out has {ob.numel()} elements, expected {n}")
    need = B.lib().sz_decode_workspace_bytes(1, sz_tiles(n))
    ws = _workspace(workspace, need, dev)
    rc = B.lib().sz_decode(payload.data_ptr(), payload.numel(), meta.data_ptr(), codebook.data_ptr(),
                           ob.data_ptr(), n, ws.data_ptr(), ws.numel(), _stream_handle(stream))
    B.check(rc, "sz_decode")
    return out


def sz_decode_inplace(slot: torch.Tensor, meta: torch.Tensor, codebook: torch.Tensor, workspace=None,
                      stream=None) -> torch.Tensor:
    """Decode the payload held in the leading meta.comp_bytes of ``slot`` (the
    BF16 destination, n elements) over the slot itself."""
    sb = _bits(slot, "slot")
    _u8(meta, "meta", B.META_BYTES)
    _u8(codebook, "codebook", B.CODEBOOK_BYTES)
    n = sb.numel()
    ws = _workspace(workspace, B.lib().sz_decode_inplace_workspace_bytes(1, sz_tiles(n)), slot.device)
    rc = B.lib().sz_decode_inplace(sb.data_ptr(), n, meta.data_ptr(), codebook.data_ptr(), ws.data_ptr(),
                                   ws.numel(), _stream_handle(stream))
    B.check(rc, "sz_decode_inplace")
    return slot


def inplace_plan(n: int, n_esc: int, tile: int) -> dict:
    """The in-place decode's schedule of one tile (stash ranges, tiles waited for)."""
    t = B.SzInplaceTile()
    B.check(B.lib().sz_inplace_plan(int(n), int(n_esc), int(tile), ctypes.byref(t)), "sz_inplace_plan")
    return {name: int(getattr(t, name)) for name, _ in B.SzInplaceTile._fields_}


# ---------------------------------------------------------------------------- many tensors


class ItemTable:
    """Host-built, device-resident sz_item table for the *_many calls."""

    def __init__(self, items: list[B.SzItem], device):
        arr = (B.SzItem * len(items))(*items)
        total = ctypes.c_uint64(0)
        B.check(B.lib().sz_items_prepare(arr, len(items), ctypes.byref(total)), "sz_items_prepare")
        self.count = len(items)
        self.total_tiles = int(total.value)
        self.host = arr
        self.device = torch.frombuffer(bytearray(bytes(arr)), dtype=torch.uint8).to(device)

    def ptr(self) -> int:
        return self.device.data_ptr()


def make_items(n: list[int], x=None, out=None, payload=None, capacity=None, codebook=None, meta=None) -> list:
    """sz_item structs from per-item pointers (ints or tensors) and sizes."""
    def p(v, i):
        if v is None:
            return None
        e = v[i]
        return e.data_ptr() if isinstance(e, torch.Tensor) else (int(e) if e is not None else None)

    items = []
    for i, ni in enumerate(n):
        it = B.SzItem()
        it.x, it.out, it.payload = p(x, i), p(out, i), p(payload, i)
        it.codebook, it.meta = p(codebook, i), p(meta, i)
        it.n = int(ni)
        it.capacity = int(capacity[i]) if capacity is not None else 0
        items.append(it)
    return items


def _rows(t: torch.Tensor, count: int, stride: int) -> list[int]:
    base = t.data_ptr()
    return [base + i * stride for i in range(count)]


def sz_calibrate_many(table: ItemTable, workspace=None, stream=None) -> None:
    dev = table.device.device
    ws = _workspace(workspace, B.lib().sz_calibrate_workspace_bytes(table.count), dev)
    rc = B.lib().sz_calibrate_many(table.ptr(), table.count, table.total_tiles, ws.data_ptr(), ws.numel(),
                                   _stream_handle(stream))
    B.check(rc, "sz_calibrate_many")


def sz_encode_many(table: ItemTable, workspace=None, stream=None) -> None:
    dev = table.device.device
    ws = _workspace(workspace, B.lib().sz_encode_workspace_bytes(table.count, table.total_tiles), dev)
    rc = B.lib().sz_encode_many(table.ptr(), table.count, table.total_tiles, ws.data_ptr(), ws.numel(),
                                _stream_handle(stream))
    B.check(rc, "sz_encode_many")


def sz_encode_gated_many(table: ItemTable, min_coverage: float, report: torch.Tensor | None = None, workspace=None,
                         stream=None) -> torch.Tensor:
    """sz_encode_many with the coverage gate: tensors below min_coverage are left
    uncompressed (meta status SZ_META_GATED).  Returns the build report (64-byte
    device tensor; read_gate_report turns it into a dict)."""
    dev = table.device.device
    if report is None:
        report = torch.empty(B.GATE_REPORT_BYTES, dtype=torch.uint8, device=dev)
    _u8(report, "report", B.GATE_REPORT_BYTES)
    ws = _workspace(workspace, B.lib().sz_encode_workspace_bytes(table.count, table.total_tiles), dev)
    rc = B.lib().sz_encode_gated_many(table.ptr(), table.count, table.total_tiles, float(min_coverage),
                                      report.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(stream))
    B.check(rc, "sz_encode_gated_many")
    return report


def slot_table(slots: list[torch.Tensor], codebooks, metas) -> ItemTable:
    """Item table for sz_decode_inplace_many: item i decodes over slots[i]
    (its payload in the slot's leading bytes); codebooks[i] / metas[i] are
    device tensors or addresses."""
    sb = [_bits(s, f"slot[{i}]") for i, s in enumerate(slots)]
    n = [s.numel() for s in sb]
    items = make_items(n, out=sb, payload=sb, capacity=[2 * k for k in n], codebook=codebooks, meta=metas)
    t = ItemTable(items, sb[0].device)
    t.keep = sb
    return t


def sz_decode_inplace_many(table: ItemTable, workspace=None, stream=None) -> None:
    dev = table.device.device
    ws = _workspace(workspace, B.lib().sz_decode_inplace_workspace_bytes(table.count, table.total_tiles), dev)
    rc = B.lib().sz_decode_inplace_many(table.ptr(), table.count, table.total_tiles, ws.data_ptr(), ws.numel(),
                                        _stream_handle(stream))
    B.check(rc, "sz_decode_inplace_many")


def read_gate_report(report: torch.Tensor) -> dict:
    r = B.SzGateReport.from_buffer_copy(bytes(report.reshape(-1)[:B.GATE_REPORT_BYTES].cpu().numpy().tobytes()))
    return {name: int(getattr(r, name)) for name, _ in B.SzGateReport._fields_}


class HostDecode:
    """sz_decode_many_host over tensors whose payloads are in pinned host memory.

    payloads[i]: pinned host uint8 tensor (or a view into one) holding the
    payload; metas[i]: its Meta; codebooks[i] / outs[i]: device tensors.  The
    staging buffer, the scratch and two pinned upload buffers are allocated
    once and reused by run(): a run writes one upload buffer while the copy
    out of the other (the run before) may still be queued, and waits for the
    run two back to have passed its upload before reusing that one."""

    def __init__(self, payloads, metas, codebooks, outs, staging_bytes: int):
        count = len(payloads)
        dev = outs[0].device
        self.items = (B.SzItem * count)()
        self.metas = (B.SzMeta * count)()
        for i in range(count):
            if payloads[i].numel() and not (payloads[i].dtype == torch.uint8 and payloads[i].is_pinned()):
                raise ValueError(f"payloads[{i}] must be a pinned host uint8 tensor")
            it = self.items[i]
            it.payload = payloads[i].data_ptr() if payloads[i].numel() else None
            it.out = _bits(outs[i], f"out[{i}]").data_ptr() if outs[i].numel() else None
            it.codebook = _u8(codebooks[i], f"codebook[{i}]", B.CODEBOOK_BYTES).data_ptr()
            it.n = outs[i].numel()
            it.capacity = payloads[i].numel()
            self.metas[i] = B.SzMeta.from_buffer_copy(meta_to_bytes(metas[i]))
        self.count = count
        self.keep = (payloads, codebooks, outs)
        self.staging = torch.empty(staging_bytes, dtype=torch.uint8, device=dev)
        need = B.lib().sz_decode_many_host_scratch_bytes(self.items, self.metas, count, staging_bytes)
        if need == 0:
            raise B.SplitZipError(B.SZ_ERR_WORKSPACE, "sz_decode_many_host_scratch_bytes")
        self.scratch = torch.empty(need, dtype=torch.uint8, device=dev)
        up = B.lib().sz_decode_many_host_upload_bytes(count)
        self.uploads = [torch.empty(up, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.uploaded = [None, None]  # event after the run that last used each upload buffer
        self.next = 0
        self.copy_stream = torch.cuda.Stream(device=dev)

    def run(self, stream=None) -> None:
        k = self.next
        self.next ^= 1
        if self.uploaded[k] is not None:
            self.uploaded[k].synchronize()
        up = self.uploads[k]
        rc = B.lib().sz_decode_many_host(self.items, self.metas, self.count, self.staging.data_ptr(),
                                         self.staging.numel(), self.scratch.data_ptr(), self.scratch.numel(),
                                         up.data_ptr(), up.numel(), _stream_handle(stream),
                                         self.copy_stream.cuda_stream)
        B.check(rc, "sz_decode_many_host")
        ev = torch.cuda.Event()
        ev.record(stream if stream is not None else torch.cuda.current_stream())
        self.uploaded[k] = ev

    def flags(self, stream=None) -> int:
        off = B.lib().sz_decode_many_host_flags_offset(self.count)
        return sz_workspace_flags(self.scratch[off:], stream)


def sz_calibrate_encode_many(table: ItemTable, workspace=None, stream=None) -> None:
    """sz_calibrate_many then sz_encode_many in one pass over HBM (same results)."""
    dev = table.device.device
    ws = _workspace(workspace, B.lib().sz_calibrate_encode_workspace_bytes(table.count, table.total_tiles), dev)
    rc = B.lib().sz_calibrate_encode_many(table.ptr(), table.count, table.total_tiles, ws.data_ptr(), ws.numel(),
                                          _stream_handle(stream))
    B.check(rc, "sz_calibrate_encode_many")


def sz_decode_many(table: ItemTable, workspace=None, stream=None) -> None:
    dev = table.device.device
    ws = _workspace(workspace, B.lib().sz_decode_workspace_bytes(table.count, table.total_tiles), dev)
    rc = B.lib().sz_decode_many(table.ptr(), table.count, table.total_tiles, ws.data_ptr(), ws.numel(),
                                _stream_handle(stream))
    B.check(rc, "sz_decode_many")


def _aligned_offsets(sizes: list[int], align: int = 256) -> tuple[list[int], int]:
    offs, o = [], 0
    for s in sizes:
        offs.append(o)
        o += (int(s) + align - 1) // align * align
    return offs, max(o, align)


class Batch:
    """Device buffers for round-tripping a list of BF16 tensors through the *_many calls.

    x[i] are the inputs (kept by reference); payloads are carved from one
    buffer at 256-byte offsets with worst-case capacities; codebooks and metas
    are rows of [count, 304] / [count, 96] uint8 tensors; outputs are carved
    from one BF16 buffer at 256-byte offsets.
    """

    def __init__(self, xs: list[torch.Tensor], capacity: list[int] | None = None):
        self.xs = [_bits(x, f"x[{i}]") for i, x in enumerate(xs)]
        dev = self.xs[0].device
        self.n = [x.numel() for x in self.xs]
        count = len(self.xs)
        cap = capacity if capacity is not None else [max(sz_max_payload_bytes(n), 16) for n in self.n]
        self.capacity = [int(c) for c in cap]
        self.payload_off, total = _aligned_offsets(self.capacity)
        self.payload = torch.empty(total, dtype=torch.uint8, device=dev)
        self.codebooks = torch.empty((count, B.CODEBOOK_BYTES), dtype=torch.uint8, device=dev)
        self.metas = torch.empty((count, B.META_BYTES), dtype=torch.uint8, device=dev)
        self.out_off, out_bytes = _aligned_offsets([2 * n for n in self.n])
        self.out = torch.empty(out_bytes // 2, dtype=torch.bfloat16, device=dev)
        pbase, obase = self.payload.data_ptr(), self.out.data_ptr()
        items = make_items(
            self.n, x=self.xs, out=[obase + o for o in self.out_off], payload=[pbase + o for o in self.payload_off],
            capacity=self.capacity, codebook=_rows(self.codebooks, count, B.CODEBOOK_BYTES),
            meta=_rows(self.metas, count, B.META_BYTES))
        self.table = ItemTable(items, dev)

    def out_view(self, i: int) -> torch.Tensor:
        o = self.out_off[i] // 2
        return self.out[o:o + self.n[i]]

    def payload_view(self, i: int, nbytes: int | None = None) -> torch.Tensor:
        o = self.payload_off[i]
        return self.payload[o:o + (self.capacity[i] if nbytes is None else nbytes)]
