"""CPU oracle of the SplitZip BF16 codec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import this package.  The library in
``weight_compression_codec_gb300`` never does, and shares no code with it.

This module is a ctypes wrapper around ``sz_oracle.c`` (a plain single-threaded
C restatement of the method of "splitzip_codec.py": calibrate_codebook,
assemble_payload, encode_torch, decode_torch).  Arrays are numpy.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from pathlib import Path

import numpy as np

from . import build as _build

CHUNK = 1024
ESCAPE = 16


class _Codebook(ctypes.Structure):
    _fields_ = [
        ("enc_lut", ctypes.c_uint8 * 256),
        ("dec_lut", ctypes.c_uint8 * 16),
        ("n_top", ctypes.c_uint32),
        ("top_count", ctypes.c_uint64),
        ("coverage", ctypes.c_double),
    ]


class _Meta(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_uint64),
        ("n_pairs", ctypes.c_uint64),
        ("n_esc", ctypes.c_uint64),
        ("comp_bytes", ctypes.c_uint64),
        ("off_pk", ctypes.c_uint64),
        ("off_sm", ctypes.c_uint64),
        ("off_cid", ctypes.c_uint64),
        ("off_lpos", ctypes.c_uint64),
        ("off_ev", ctypes.c_uint64),
        ("chunk_size", ctypes.c_uint32),
        ("coverage", ctypes.c_double),
    ]


@dataclass(frozen=True)
class Codebook:
    enc_lut: np.ndarray  # uint8[256], code 0..15 or 16 = escape
    dec_lut: np.ndarray  # uint8[16]
    n_top: int
    top_count: int
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
    coverage: float

    def as_tuple(self) -> tuple:
        return (self.n, self.n_pairs, self.n_esc, self.comp_bytes, self.off_pk, self.off_sm,
                self.off_cid, self.off_lpos, self.off_ev, self.chunk_size)


_lib = None


def load(lib_path: Path | None = None):
    """Load (building if needed) the oracle library; returns the ctypes handle."""
    global _lib
    if lib_path is None and _lib is not None:
        return _lib
    path = Path(lib_path) if lib_path is not None else _build.build()
    lib = ctypes.CDLL(str(path))
    u16p = ctypes.POINTER(ctypes.c_uint16)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.szo_histogram.argtypes = [u16p, ctypes.c_uint64, u64p]
    lib.szo_histogram.restype = None
    lib.szo_select.argtypes = [u64p, ctypes.c_uint64, ctypes.POINTER(_Codebook)]
    lib.szo_select.restype = None
    lib.szo_calibrate.argtypes = [u16p, ctypes.c_uint64, ctypes.POINTER(_Codebook)]
    lib.szo_calibrate.restype = None
    lib.szo_layout.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double, ctypes.POINTER(_Meta)]
    lib.szo_layout.restype = None
    lib.szo_count_escapes.argtypes = [u16p, ctypes.c_uint64, ctypes.POINTER(_Codebook)]
    lib.szo_count_escapes.restype = ctypes.c_uint64
    lib.szo_encode.argtypes = [u16p, ctypes.c_uint64, ctypes.POINTER(_Codebook), u8p, ctypes.c_uint64,
                               ctypes.POINTER(_Meta)]
    lib.szo_encode.restype = ctypes.c_int
    lib.szo_decode.argtypes = [u8p, ctypes.POINTER(_Meta), u8p, u16p]
    lib.szo_decode.restype = ctypes.c_int
    lib.szo_to_p1_nibble_order.argtypes = [u8p, ctypes.POINTER(_Meta)]
    lib.szo_to_p1_nibble_order.restype = None
    if lib_path is None:
        _lib = lib
    return lib


def _u16(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError(f"expected BF16 bit patterns as uint16, got {a.dtype}")
    return a.reshape(-1)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _cb_to_c(cb: Codebook) -> _Codebook:
    c = _Codebook()
    ctypes.memmove(c.enc_lut, np.ascontiguousarray(cb.enc_lut, dtype=np.uint8).ctypes.data, 256)
    ctypes.memmove(c.dec_lut, np.ascontiguousarray(cb.dec_lut, dtype=np.uint8).ctypes.data, 16)
    c.n_top = cb.n_top
    c.top_count = cb.top_count
    c.coverage = cb.coverage
    return c


def _cb_from_c(c: _Codebook) -> Codebook:
    return Codebook(
        enc_lut=np.frombuffer(bytes(c.enc_lut), dtype=np.uint8).copy(),
        dec_lut=np.frombuffer(bytes(c.dec_lut), dtype=np.uint8).copy(),
        n_top=int(c.n_top),
        top_count=int(c.top_count),
        coverage=float(c.coverage),
    )


def _meta_to_c(m: Meta) -> _Meta:
    c = _Meta()
    for f, _ in _Meta._fields_:
        setattr(c, f, getattr(m, f))
    return c


def _meta_from_c(c: _Meta) -> Meta:
    return Meta(**{f: (float(getattr(c, f)) if f == "coverage" else int(getattr(c, f))) for f, _ in _Meta._fields_})


def histogram(x, lib=None) -> np.ndarray:
    lib = lib or load()
    a = _u16(x)
    h = np.zeros(256, dtype=np.uint64)
    lib.szo_histogram(_ptr(a, ctypes.c_uint16), a.size, _ptr(h, ctypes.c_uint64))
    return h


def select(hist, n: int, lib=None) -> Codebook:
    lib = lib or load()
    h = np.ascontiguousarray(hist, dtype=np.uint64)
    c = _Codebook()
    lib.szo_select(_ptr(h, ctypes.c_uint64), n, ctypes.byref(c))
    return _cb_from_c(c)


def calibrate(x, lib=None) -> Codebook:
    lib = lib or load()
    a = _u16(x)
    c = _Codebook()
    lib.szo_calibrate(_ptr(a, ctypes.c_uint16), a.size, ctypes.byref(c))
    return _cb_from_c(c)


def layout(n: int, n_esc: int, coverage: float = 1.0, lib=None) -> Meta:
    lib = lib or load()
    c = _Meta()
    lib.szo_layout(n, n_esc, coverage, ctypes.byref(c))
    return _meta_from_c(c)


def count_escapes(x, cb: Codebook, lib=None) -> int:
    lib = lib or load()
    a = _u16(x)
    c = _cb_to_c(cb)
    return int(lib.szo_count_escapes(_ptr(a, ctypes.c_uint16), a.size, ctypes.byref(c)))


def encode(x, cb: Codebook, lib=None) -> tuple[np.ndarray, Meta]:
    """Returns (payload bytes as uint8 array of length comp_bytes, meta)."""
    lib = lib or load()
    a = _u16(x)
    c = _cb_to_c(cb)
    n_esc = int(lib.szo_count_escapes(_ptr(a, ctypes.c_uint16), a.size, ctypes.byref(c)))
    m = layout(a.size, n_esc, cb.coverage, lib=lib)
    out = np.empty(max(m.comp_bytes, 1), dtype=np.uint8)
    cm = _Meta()
    rc = lib.szo_encode(_ptr(a, ctypes.c_uint16), a.size, ctypes.byref(c), _ptr(out, ctypes.c_uint8),
                        m.comp_bytes, ctypes.byref(cm))
    if rc != 0:
        raise RuntimeError(f"oracle encode failed with status {rc}")
    return out[: m.comp_bytes], _meta_from_c(cm)


def decode(payload, meta: Meta, dec_lut, lib=None) -> np.ndarray:
    lib = lib or load()
    p = np.ascontiguousarray(payload, dtype=np.uint8).reshape(-1)
    if p.size < meta.comp_bytes:
        raise ValueError("payload shorter than meta.comp_bytes")
    if p.size == 0:
        p = np.zeros(1, dtype=np.uint8)
    d = np.ascontiguousarray(dec_lut, dtype=np.uint8)
    out = np.empty(max(meta.n, 1), dtype=np.uint16)
    cm = _meta_to_c(meta)
    rc = lib.szo_decode(_ptr(p, ctypes.c_uint8), ctypes.byref(cm), _ptr(d, ctypes.c_uint8),
                        _ptr(out, ctypes.c_uint16))
    if rc != 0:
        raise ValueError(f"oracle decode rejected the payload (status {rc})")
    return out[: meta.n]


def to_p1_nibble_order(payload, meta: Meta, lib=None) -> np.ndarray:
    """Copy of ``payload`` with the pk nibbles swapped (element 2i -> high nibble)."""
    lib = lib or load()
    p = np.array(payload, dtype=np.uint8, copy=True).reshape(-1)
    if meta.n_pairs:
        cm = _meta_to_c(meta)
        lib.szo_to_p1_nibble_order(_ptr(p, ctypes.c_uint8), ctypes.byref(cm))
    return p


# ---------------------------------------------------------------------------- coverage gate
# "docs/developer/splitzip.md" (the shard-cache builder): tensors whose Top-16
# exponent coverage falls below 0.99 are left uncompressed, so the worst case
# is parity; the builder reports the tensors encoded and skipped for coverage
# and the payload ratio.  Reading: "below" is strict (coverage == gate is
# encoded); a negative gate gates nothing; a tensor that still expands is
# counted, not dropped.


def gated(coverage: float, min_coverage: float) -> bool:
    """True if the coverage gate leaves the tensor uncompressed."""
    return min_coverage >= 0.0 and coverage < min_coverage


def gate_report(ns, coverages, metas, min_coverage: float) -> dict:
    """Build report over tensors of sizes ns, codebook coverages and the metas
    their plain encode gives (meta i is used only when tensor i is encoded)."""
    r = dict(tensors_encoded=0, tensors_gated=0, raw_bytes_encoded=0, payload_bytes=0, raw_bytes_gated=0,
             tensors_expanded=0, escapes=0, tensors_failed=0)
    for n, cov, m in zip(ns, coverages, metas):
        if gated(cov, min_coverage):
            r["tensors_gated"] += 1
            r["raw_bytes_gated"] += 2 * n
        else:
            r["tensors_encoded"] += 1
            r["raw_bytes_encoded"] += 2 * n
            r["payload_bytes"] += m.comp_bytes
            r["tensors_expanded"] += int(m.comp_bytes > 2 * n)
            r["escapes"] += m.n_esc
    return r


# ---------------------------------------------------------------------------- slot decode
# "splitzip_codec.py" GpuSplitZipDecoder.decode_slot_into and
# "docs/developer/splitzip.md" (how a compressed fault is served; staging
# invariants): the destination of a weight is a slot of its RAW size (2n
# bytes); the compressed payload was copied into the slot's leading
# comp_bytes; the decoder first copies those bytes aside (the slot is about to
# be overwritten) and then decodes the full BF16 weight over the slot.  Bytes
# of the slot past comp_bytes carry nothing.  Reading: a payload larger than
# the slot cannot have been placed there and is rejected.


def decode_slot(slot, meta: Meta, dec_lut, lib=None) -> np.ndarray:
    """Decode the payload in slot[:meta.comp_bytes] over the slot (uint8, 2n
    bytes).  Returns the slot, which then holds the BF16 bit patterns."""
    s = np.asarray(slot)
    if s.dtype != np.uint8 or s.ndim != 1 or s.size != 2 * meta.n:
        raise ValueError("the slot must be a flat uint8 array of 2n bytes")
    if meta.comp_bytes > s.size:
        raise ValueError("payload larger than the slot")
    stash = s[: meta.comp_bytes].copy()  # step 1: the payload copied aside
    x = decode(stash, meta, dec_lut, lib=lib)  # step 2: decode over the slot
    s[:] = x.view(np.uint8)
    return s
