"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, and compare every byte with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import weight_compression_codec_gb300 as sz

DEV = torch.device("cuda:0")


def to_dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(DEV)


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_codebook(gcb: "sz.Codebook", ocb: "oracle.Codebook", n: int) -> None:
    assert np.array_equal(gcb.enc_lut, ocb.enc_lut), "enc_lut differs"
    assert np.array_equal(gcb.dec_lut, ocb.dec_lut), "dec_lut differs"
    assert gcb.n_top == ocb.n_top and gcb.top_count == ocb.top_count and gcb.n == n
    assert gcb.coverage == ocb.coverage  # one IEEE double division on both sides


def oracle_codebook_bytes(ocb: "oracle.Codebook", n: int) -> bytes:
    from weight_compression_codec_gb300 import binding as B

    c = B.SzCodebook()
    c.enc_lut[:] = list(ocb.enc_lut)
    c.dec_lut[:] = list(ocb.dec_lut)
    c.n_top = ocb.n_top
    c.top_count = ocb.top_count
    c.n = n
    c.coverage = ocb.coverage
    return bytes(c)


def roundtrip_single(x: np.ndarray, codebook_from: np.ndarray | None = None) -> dict:
    """calibrate -> encode -> decode on the GPU, each result compared with the oracle.
    With ``codebook_from``, the codebook is calibrated on that array instead."""
    n = x.size
    xd = to_dev(x)
    src = x if codebook_from is None else codebook_from
    cb = sz.sz_calibrate(to_dev(src))
    payload, meta = sz.sz_encode(xd, cb)
    out = sz.sz_decode(payload, meta, cb, n)
    torch.cuda.synchronize()
    ocb = oracle.calibrate(src)
    check_codebook(sz.read_codebook(cb), ocb, src.size)
    opay, om = oracle.encode(x, ocb)
    m = sz.read_meta(meta)
    assert m.status == 0, f"device status 0x{m.status:x}"
    assert m.as_tuple() == om.as_tuple(), (m, om)
    assert m.coverage == ocb.coverage
    gp = payload[:m.comp_bytes].cpu().numpy()
    if not np.array_equal(gp, opay):
        bad = np.nonzero(gp != opay)[0]
        raise AssertionError(f"payload differs at {bad.size} bytes, first at {bad[:8]} (layout {om})")
    y = to_np_u16(out)
    assert np.array_equal(y, x), f"decode differs at {np.count_nonzero(y != x)} elements"
    # the GPU decoder also reads the oracle's payload
    p2 = torch.from_numpy(np.concatenate([opay, np.zeros(16, np.uint8)])).to(DEV)
    meta2 = torch.frombuffer(bytearray(sz.meta_to_bytes(om)), dtype=torch.uint8).to(DEV)
    cb2 = torch.frombuffer(bytearray(oracle_codebook_bytes(ocb, src.size)), dtype=torch.uint8).to(DEV)
    out2 = sz.sz_decode(p2[:max(om.comp_bytes, 1)], meta2, cb2, n)
    assert np.array_equal(to_np_u16(out2), x)
    return {"meta": m, "codebook": ocb}
