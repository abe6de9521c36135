"""ctypes binding of libsplitzip.so (include/splitzip.h).

Argument marshalling only: every step of calibrate / encode / decode runs in
the library's CUDA kernels.  PyTorch provides device memory (tensors) and
streams; nothing here computes codec results on the host.  If the library is
missing, ``lib()`` raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

from . import buildlib as _build

SZ_CHUNK_SIZE = 1024
SZ_TILE_ELEMS = 8192
SZ_ESCAPE_CODE = 16
SZ_MAX_ELEMS = 4294967295
SZ_MANY_MAX_ITEMS = 65535

SZ_OK, SZ_ERR_ARG, SZ_ERR_ALIGN, SZ_ERR_CAPACITY, SZ_ERR_META, SZ_ERR_WORKSPACE, SZ_ERR_CUDA, SZ_ERR_DEVICE = range(8)

SZ_FLAG_CAPACITY = 0x01
SZ_FLAG_META = 0x02
SZ_FLAG_ESCAPE = 0x04
SZ_FLAG_TIMEOUT = 0x08
SZ_FLAG_ALIGN = 0x10
SZ_FLAG_ITEMS = 0x20
SZ_FLAG_SIZE = 0x40
SZ_META_GATED = 0x100  # sz_meta.status: kept raw by the coverage gate (not an error)


class SzCodebook(ctypes.Structure):
    _fields_ = [
        ("enc_lut", ctypes.c_uint8 * 256),
        ("dec_lut", ctypes.c_uint8 * 16),
        ("n_top", ctypes.c_uint32),
        ("reserved0", ctypes.c_uint32),
        ("top_count", ctypes.c_uint64),
        ("n", ctypes.c_uint64),
        ("coverage", ctypes.c_double),
    ]


class SzMeta(ctypes.Structure):
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
        ("status", ctypes.c_uint32),
        ("coverage", ctypes.c_double),
        ("reserved1", ctypes.c_uint64),
    ]


class SzItem(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("payload", ctypes.c_void_p),
        ("codebook", ctypes.c_void_p),
        ("meta", ctypes.c_void_p),
        ("n", ctypes.c_uint64),
        ("capacity", ctypes.c_uint64),
        ("tile_begin", ctypes.c_uint64),
    ]


assert ctypes.sizeof(SzCodebook) == 304
assert ctypes.sizeof(SzMeta) == 96
assert ctypes.sizeof(SzItem) == 64

class SzGateReport(ctypes.Structure):
    _fields_ = [(name, ctypes.c_uint64) for name in (
        "tensors_encoded", "tensors_gated", "raw_bytes_encoded", "payload_bytes", "raw_bytes_gated",
        "tensors_expanded", "escapes", "tensors_failed")]


class SzInplaceTile(ctypes.Structure):
    _fields_ = [(name, ctypes.c_uint64) for name in (
        "tiles", "phase_a_first", "phase_b_end", "rank", "stash_pk_from", "stash_pk_to", "stash_esc_from",
        "stash_esc_to", "stash_bytes", "stash_budget", "pk_lo", "pk_hi", "pk2_lo", "pk2_hi", "sm_lo", "sm_hi")]


CODEBOOK_BYTES = 304
META_BYTES = 96
GATE_REPORT_BYTES = 64
ITEM_BYTES = 64

# Every symbol of include/splitzip.h with its ctypes signature.
_VP, _U64, _U32, _SZ, _INT = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_size_t, ctypes.c_int
SIGNATURES = {
    "sz_version": (_INT, []),
    "sz_strerror": (ctypes.c_char_p, [_INT]),
    "sz_tiles": (_U64, [_U64]),
    "sz_layout": (_INT, [_U64, _U64, ctypes.POINTER(SzMeta)]),
    "sz_payload_bytes": (_U64, [_U64, _U64]),
    "sz_max_payload_bytes": (_U64, [_U64]),
    "sz_items_prepare": (_INT, [ctypes.POINTER(SzItem), _U32, ctypes.POINTER(_U64)]),
    "sz_calibrate_workspace_bytes": (_SZ, [_U32]),
    "sz_encode_workspace_bytes": (_SZ, [_U32, _U64]),
    "sz_decode_workspace_bytes": (_SZ, [_U32, _U64]),
    "sz_calibrate_encode_workspace_bytes": (_SZ, [_U32, _U64]),
    "sz_workspace_flags": (_INT, [_VP, ctypes.POINTER(_U32), _VP]),
    "sz_calibrate": (_INT, [_VP, _U64, _VP, _VP, _SZ, _VP]),
    "sz_encode": (_INT, [_VP, _U64, _VP, _VP, _U64, _VP, _VP, _SZ, _VP]),
    "sz_decode": (_INT, [_VP, _U64, _VP, _VP, _VP, _U64, _VP, _SZ, _VP]),
    "sz_calibrate_many": (_INT, [_VP, _U32, _U64, _VP, _SZ, _VP]),
    "sz_encode_many": (_INT, [_VP, _U32, _U64, _VP, _SZ, _VP]),
    "sz_decode_many": (_INT, [_VP, _U32, _U64, _VP, _SZ, _VP]),
    "sz_calibrate_encode": (_INT, [_VP, _U64, _VP, _VP, _U64, _VP, _VP, _SZ, _VP]),
    "sz_calibrate_encode_many": (_INT, [_VP, _U32, _U64, _VP, _SZ, _VP]),
    "sz_encode_gated_many": (_INT, [_VP, _U32, _U64, ctypes.c_double, _VP, _VP, _SZ, _VP]),
    "sz_check_bounded_waits": (_INT, [_VP, _SZ, _VP]),
    "sz_decode_inplace": (_INT, [_VP, _U64, _VP, _VP, _VP, _SZ, _VP]),
    "sz_decode_inplace_many": (_INT, [_VP, _U32, _U64, _VP, _SZ, _VP]),
    "sz_decode_inplace_workspace_bytes": (_SZ, [_U32, _U64]),
    "sz_inplace_plan": (_INT, [_U64, _U64, _U64, ctypes.POINTER(SzInplaceTile)]),
    "sz_decode_many_host_scratch_bytes": (_SZ, [_VP, _VP, _U32, _U64]),
    "sz_decode_many_host_upload_bytes": (_SZ, [_U32]),
    "sz_decode_many_host": (_INT, [_VP, _VP, _U32, _VP, _U64, _VP, _SZ, _VP, _SZ, _VP, _VP]),
    "sz_decode_many_host_flags_offset": (_SZ, [_U32]),
    "sz_set_timing_events": (_INT, [_VP, _VP]),
    "sz_decode_noalloc": (_INT, [_VP, _U64, _VP, _VP, _VP, _U64, _VP, _VP]),
}

SZ_NOALLOC_MAX_ELEMS = 268435456
SZ_CHECK_WAITS_WORKSPACE_BYTES = 512

_LIB = None


class SplitZipError(RuntimeError):
    def __init__(self, status: int, where: str, flags: int | None = None):
        self.status = status
        self.flags = flags
        msg = f"{where}: status {status} ({strerror(status)})"
        if flags is not None:
            msg += f", device flags 0x{flags:02x}"
        super().__init__(msg)


def library_path() -> Path:
    return _build.LIB_PATH


def lib(path: Path | None = None):
    """The loaded library.  Raises if it has not been built."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = Path(path) if path is not None else library_path()
    if not p.exists():
        raise RuntimeError(
            f"libsplitzip.so not found at {p}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    handle = ctypes.CDLL(str(p))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = handle
    return handle


def strerror(status: int) -> str:
    try:
        return lib().sz_strerror(status).decode()
    except Exception:  # library missing: still give a readable message
        return "unknown"


def check(status: int, where: str) -> None:
    if status != SZ_OK:
        raise SplitZipError(status, where)
