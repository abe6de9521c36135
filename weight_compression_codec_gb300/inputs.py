"""Seeded synthetic BF16 inputs for the codec's tests and benchmark.

This module only builds input values; it holds none of the codec's arithmetic
(no exponent split, no codebook, no layout), so both the CUDA path and the CPU
oracle can take their inputs from it.  Every generator returns BF16 bit
patterns as ``numpy.uint16`` arrays, one per tensor, created from a fixed seed
with numpy's PCG64 generator.  float32 values are rounded to BF16 with
round-to-nearest-even.

The workloads stand in for the data the SplitZip pages measure on (LLM KV
activations and model weights), which are not available here:

* ``gaussian``      -- one weight-like tensor, N(0, sigma).
* ``kv_cache``      -- a [layers, K/V, tokens, kv_heads, head_dim] cache,
  N(0, 1) times a per-(layer, K/V, head, channel) scale, log-uniform in
  [0.1, 20], with 1 % of the channels given a 30x outlier scale; one tensor per
  (layer, K/V) slice.
* ``weight_pairs``  -- pairs of 4096x14336 / 14336x4096 matrices, N(0, 0.02)
  with 0.1 % of entries replaced by N(0, 1); the last tensor additionally has
  3 % of entries replaced by +-m * 2^U (U uniform in [-60, 20], m in [1, 2)) so
  that its exponent distribution is broad.
* ``edge_case``     -- magnitudes 2^U (U uniform integer in [-140, 40]) with
  random signs, plus 5 % subnormals, +-0, +-Inf and NaNs with random payloads.
* ``paged_kv``      -- many independent [16, 8, 128] blocks, each N(0, s) with s
  log-uniform in [0.01, 10] per block.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BASE_SEED = 1000
BLOCK = 1 << 24  # elements per independently seeded block of the large generators


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([BASE_SEED, *key]))


def _blocks(n: int, key: tuple, fill) -> np.ndarray:
    """n BF16 patterns made block by block: block b (elements [b BLOCK, (b + 1)
    BLOCK)) is ``fill(rng, count)`` with its own generator seeded by key + (b,),
    so the values do not depend on how many threads make them."""
    out = np.empty(n, dtype=np.uint16)
    nb = (n + BLOCK - 1) // BLOCK

    def work(b: int) -> None:
        lo = b * BLOCK
        hi = min(n, lo + BLOCK)
        out[lo:hi] = fill(_rng(*key, b), hi - lo)

    if nb <= 1:
        for b in range(nb):
            work(b)
    else:
        with ThreadPoolExecutor(max_workers=min(nb, os.cpu_count() or 1, 16)) as ex:
            list(ex.map(work, range(nb)))
    return out


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (round to nearest, ties to even); NaNs stay NaN."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    out = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    if nan.any():
        out[nan] = ((u[nan] >> np.uint32(16)) | np.uint32(0x0040)).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def all_bit_patterns() -> np.ndarray:
    """Every one of the 65,536 BF16 bit patterns, in ascending order."""
    return np.arange(65536, dtype=np.uint16)


def gaussian(n: int, sigma: float = 0.02, seed: int = 0) -> np.ndarray:
    return _blocks(n, (1, seed),
                   lambda r, k: f32_to_bf16_bits(r.standard_normal(k, dtype=np.float32) * np.float32(sigma)))


def kv_cache_shape(layers=32, tokens=4096, kv_heads=8, head_dim=128):
    return (layers, 2, tokens, kv_heads, head_dim)


def kv_cache_tensor(layer: int, kv: int, tokens=4096, kv_heads=8, head_dim=128) -> np.ndarray:
    """One [tokens, kv_heads, head_dim] slice of the KV cache (K for kv=0, V for kv=1)."""
    r = _rng(2, layer, kv)
    scale = np.exp(r.uniform(np.log(0.1), np.log(20.0), size=(kv_heads, head_dim))).astype(np.float32)
    outlier = r.random(size=(kv_heads, head_dim)) < 0.01
    scale[outlier] *= np.float32(30.0)
    v = r.standard_normal((tokens, kv_heads, head_dim), dtype=np.float32) * scale[None, :, :]
    return f32_to_bf16_bits(v).reshape(-1)


def kv_cache(layers=32, tokens=4096, kv_heads=8, head_dim=128) -> list[np.ndarray]:
    """All (layer, K/V) slices, layer-major: tensor 2*l + kv."""
    return [kv_cache_tensor(l, kv, tokens, kv_heads, head_dim) for l in range(layers) for kv in range(2)]


def weight_tensor(index: int, pairs=8, d_model=4096, d_ff=14336) -> np.ndarray:
    """Tensor ``index`` of ``pairs`` (d_model x d_ff, d_ff x d_model) matrices."""

    def fill(r: np.random.Generator, n: int) -> np.ndarray:
        v = r.standard_normal(n, dtype=np.float32) * np.float32(0.02)
        big = r.random(n) < 0.001
        v[big] = r.standard_normal(int(big.sum()), dtype=np.float32)
        if index == 2 * pairs - 1:
            broad = r.random(n) < 0.03
            k = int(broad.sum())
            u = r.integers(-60, 21, size=k)
            m = r.uniform(1.0, 2.0, size=k)
            s = np.where(r.random(k) < 0.5, -1.0, 1.0)
            v[broad] = (s * m * np.exp2(u.astype(np.float64))).astype(np.float32)
        return f32_to_bf16_bits(v)

    return _blocks(d_model * d_ff, (3, index), fill)


def weight_shapes(pairs=8, d_model=4096, d_ff=14336):
    return [(d_model, d_ff) if i % 2 == 0 else (d_ff, d_model) for i in range(2 * pairs)]


def weight_pairs(pairs=8, d_model=4096, d_ff=14336) -> list[np.ndarray]:
    return [weight_tensor(i, pairs, d_model, d_ff) for i in range(2 * pairs)]


def edge_case(n: int = 100_000_003, seed: int = 0) -> np.ndarray:
    """Escape-heavy tensor with special values mixed in (see module docstring)."""
    return _blocks(n, (4, seed), _edge_block)


def _edge_block(r: np.random.Generator, n: int) -> np.ndarray:
    u = r.integers(-140, 41, size=n)
    m = r.uniform(1.0, 2.0, size=n)
    s = np.where(r.random(n) < 0.5, -1.0, 1.0)
    out = f32_to_bf16_bits((s * m * np.exp2(u.astype(np.float64))).astype(np.float32))
    cat = r.random(n)
    sign = (r.random(n) < 0.5).astype(np.uint16) << np.uint16(15)
    mant = r.integers(1, 128, size=n).astype(np.uint16)
    # [0, 0.05): subnormal (exponent field 0, non-zero mantissa, random sign)
    sel = cat < 0.05
    out[sel] = sign[sel] | mant[sel]
    # +0, -0, +Inf, -Inf: 0.5 % each
    for lo, bits in ((0.050, 0x0000), (0.055, 0x8000), (0.060, 0x7F80), (0.065, 0xFF80)):
        out[(cat >= lo) & (cat < lo + 0.005)] = np.uint16(bits)
    # 1 % NaN: exponent field all ones, non-zero mantissa payload, random sign
    sel = (cat >= 0.070) & (cat < 0.080)
    out[sel] = sign[sel] | np.uint16(0x7F80) | mant[sel]
    return out


def paged_kv_block(index: int, block=16, heads=8, head_dim=128) -> np.ndarray:
    r = _rng(5, index)
    s = np.float32(np.exp(r.uniform(np.log(0.01), np.log(10.0))))
    return f32_to_bf16_bits(r.standard_normal(block * heads * head_dim, dtype=np.float32) * s)


def paged_kv(count=8192, block=16, heads=8, head_dim=128) -> list[np.ndarray]:
    """``count`` independent blocks; generated in one draw per block."""
    return [paged_kv_block(i, block, heads, head_dim) for i in range(count)]


def paged_kv_flat(count=8192, block=16, heads=8, head_dim=128) -> np.ndarray:
    """The same blocks as ``paged_kv``, concatenated (block i at i * block*heads*head_dim)."""
    per = block * heads * head_dim
    out = np.empty(count * per, dtype=np.uint16)
    for i in range(count):
        out[i * per:(i + 1) * per] = paged_kv_block(i, block, heads, head_dim)
    return out


def sweep_sizes(lo_bytes=1 << 20, hi_bytes=4 << 30) -> list[int]:
    """Element counts of the size sweep: 1 MiB .. 4 GiB of BF16, doubling."""
    out, b = [], lo_bytes
    while b <= hi_bytes:
        out.append(b // 2)
        b *= 2
    return out


def sweep_tensor(n: int) -> np.ndarray:
    return _blocks(n, (6, n), lambda r, k: f32_to_bf16_bits(r.standard_normal(k, dtype=np.float32)))
