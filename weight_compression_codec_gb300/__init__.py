"""SplitZip lossless BF16 codec for GB300 (sm_103a).

Per-tensor Top-16 exponent calibration, encode into the split payload
(4-bit exponent codes, verbatim sign+mantissa bytes, ordered escape stream)
and bitwise-exact decode, as hand-written CUDA kernels behind the C ABI of
``include/splitzip.h``.  This package is the thin Python binding: argument
marshalling over ctypes, with PyTorch supplying device memory and streams.
"""
from .binding import SplitZipError, lib, library_path  # noqa: F401
from .codec import (  # noqa: F401
    Batch,
    Codebook,
    HostDecode,
    ItemTable,
    Meta,
    Workspace,
    codebook_from_bytes,
    inplace_plan,
    make_items,
    meta_from_bytes,
    meta_to_bytes,
    read_codebook,
    read_gate_report,
    read_meta,
    slot_table,
    sz_calibrate,
    sz_calibrate_encode,
    sz_calibrate_encode_many,
    sz_calibrate_many,
    sz_decode,
    sz_decode_inplace,
    sz_decode_inplace_many,
    sz_decode_many,
    sz_encode,
    sz_encode_gated_many,
    sz_encode_many,
    sz_layout,
    sz_max_payload_bytes,
    sz_payload_bytes,
    sz_set_timing_events,
    sz_tiles,
    sz_workspace_flags,
)


def build(force: bool = False) -> str:
    """Compile libsplitzip.so for sm_103a (in-tree) and return its path."""
    from .buildlib import build as _b

    return str(_b(force=force))
