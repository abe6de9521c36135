// Split + pack of one 1024-element chunk by one warp, shared by the encode
// kernel and the fused calibrate + encode kernel.  A Stage holds the staged
// tile: x[8192] (its BF16 patterns), enc_lut[256] (the tensor's codebook),
// lt (tile index within the tensor), n_tile (elements present), payload and
// off_sm (where pk and sm go).
#pragma once

#include "sz_device.cuh"

namespace sz {

// A chunk with more escapes than this is not staged: staging costs 4 bytes
// written and read per escape, more than reading the chunk's 2 KiB of input
// again, so the placement pass regenerates such a chunk's escapes from the
// input instead (enc_place).  Chunks of partial tiles may still be staged;
// the placement pass ignores the staging of every chunk above the limit.
constexpr uint32_t kStageMax = 256;

// Bounded mbarrier wait agreed by the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity));
}

__device__ __forceinline__ uint32_t sm_pair(uint32_t w) {
  // two BF16 patterns in w -> sm bytes at byte 0 and byte 2
  return (w & 0x007F007Fu) | ((w >> 8) & 0x00800080u);
}

// enc_lut codes of the 4 elements held in v (element k in bits 16k..16k+15 of
// v.x, v.y), one per byte (element k in byte k).  Shifting a word left by one
// puts the exponent bytes of its two elements at bytes 1 and 3.
__device__ __forceinline__ uint32_t codes4(const uint8_t* lut, uint2 v) {
  const uint32_t ax = v.x << 1, ay = v.y << 1;
  const uint32_t c0 = lut[__byte_perm(ax, 0, 0x4441)];
  const uint32_t c1 = lut[__byte_perm(ax, 0, 0x4443)];
  const uint32_t c2 = lut[__byte_perm(ay, 0, 0x4441)];
  const uint32_t c3 = lut[__byte_perm(ay, 0, 0x4443)];
  return c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
}

// Split + pack of chunk `warp` of the tile in `st`, with its escapes compacted
// in element order into the staging slot `slot`.  Each lane handles 4 consecutive
// elements per row of 128.  Escape handling is byte-parallel: an enc_lut value
// >= 16 (a non-zero high nibble) marks an escape, stored in pk as code 0.
// Returns the chunk's escape count.  FULL_TILE: all 8192 elements exist.
template <bool FULL_TILE, class Stage>
__device__ __forceinline__ uint32_t encode_chunk(const Stage& st, uint32_t warp, uint32_t lane, uint32_t* slot) {
  const uint8_t* lut = st.enc_lut;
  const uint32_t nt = st.n_tile;
  const uint64_t g = uint64_t(st.lt) * kTile;
  const uint32_t e0 = warp * kChunk + lane * 4u;  // element of this lane in row 0
  const uint16_t* xw = st.x + e0;
  uint8_t* pkw = st.payload + (g >> 1) + (e0 >> 1);
  uint8_t* smw = st.payload + st.off_sm + g + e0;
  const uint32_t lane_lt = (1u << lane) - 1u;
  uint32_t run = 0;  // escapes of this chunk so far (warp-uniform)
#pragma unroll
  for (int row = 0; row < 8; ++row) {
    const uint2 v = *reinterpret_cast<const uint2*>(xw + row * 128);
    uint32_t packed = codes4(lut, v);
    uint32_t nvalid = 4;
    if (!FULL_TILE) {
      const uint32_t il = e0 + uint32_t(row) * 128u;
      nvalid = (il < nt) ? ((nt - il) < 4u ? nt - il : 4u) : 0u;
      if (nvalid < 4) packed &= (1u << (8 * nvalid)) - 1u;  // absent elements: code 0, no escape
    }
    const uint32_t hi = packed & 0xF0F0F0F0u;
    uint32_t clean = packed & 0x0F0F0F0Fu;
    uint32_t m = 0;
    if (hi) {
      m = ((hi >> 4) + 0x7F7F7F7Fu) & 0x80808080u;  // bit 7 of each escape byte
      clean &= ~((m >> 7) * 0xFFu);
    }
    const uint32_t t = clean | (clean >> 4);  // byte 0 = c0 | c1 << 4, byte 2 = c2 | c3 << 4
    const uint32_t pk16 = __byte_perm(t, 0, 0x4420);
    const uint32_t sm4 = __byte_perm(sm_pair(v.x), sm_pair(v.y), 0x6420);
    if (FULL_TILE || nvalid == 4) {
      *reinterpret_cast<uint16_t*>(pkw + row * 64) = uint16_t(pk16);
      *reinterpret_cast<uint32_t*>(smw + row * 128) = sm4;
    } else if (nvalid > 0) {
      pkw[row * 64] = uint8_t(pk16);
      if (nvalid > 2) pkw[row * 64 + 1] = uint8_t(pk16 >> 8);
      for (uint32_t k = 0; k < nvalid; ++k) smw[row * 128 + k] = uint8_t(sm4 >> (8 * k));
    }
    if (__ballot_sync(0xFFFFFFFFu, m != 0)) {
      const uint32_t escm = ((m >> 7) & 1u) | ((m >> 14) & 2u) | ((m >> 21) & 4u) | ((m >> 28) & 8u);
      const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, escm & 1u), b1 = __ballot_sync(0xFFFFFFFFu, escm & 2u);
      const uint32_t b2 = __ballot_sync(0xFFFFFFFFu, escm & 4u), b3 = __ballot_sync(0xFFFFFFFFu, escm & 8u);
      uint32_t pos = run + __popc(b0 & lane_lt) + __popc(b1 & lane_lt) + __popc(b2 & lane_lt) +
                     __popc(b3 & lane_lt);
      const uint32_t ex[4] = {(v.x >> 7) & 0xFFu, (v.x >> 23) & 0xFFu, (v.y >> 7) & 0xFFu, (v.y >> 23) & 0xFFu};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if ((escm >> k) & 1u) {
          slot[pos] = uint32_t(row * 128 + lane * 4 + k) | (ex[k] << 16);
          ++pos;
        }
      }
      run += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
    }
  }
  return run;
}

// sm bytes of the four BF16 patterns in (a, b) (element 2k in the low half of
// a or b), element j in byte j: the low byte of each pattern with bit 7
// replaced by the pattern's sign.  One permute gathers the low bytes, one
// permute in sign-replicating mode (selector msb set) turns each pattern's
// high byte into 0x00 or 0xFF, one bit-select merges them.
__device__ __forceinline__ uint32_t sm_quad(uint32_t a, uint32_t b) {
  uint32_t lows, signs;
  asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(lows) : "r"(a), "r"(b));
  asm("prmt.b32 %0, %1, %2, 0xFDB9;" : "=r"(signs) : "r"(a), "r"(b));
  return (lows & 0x7F7F7F7Fu) | (signs & 0x80808080u);
}

// Exclusive warp prefix of per-lane counts `c` (0..8) and the warp total.
// Most rows hold at most one escape per lane: then two ballots suffice.
__device__ __forceinline__ uint32_t warp_prefix(uint32_t c, uint32_t lane, uint32_t* total) {
  const uint32_t lane_lt = (1u << lane) - 1u;
  const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, c >= 1);
  const uint32_t b2 = __ballot_sync(0xFFFFFFFFu, c >= 2);
  if (b2 == 0) {
    *total = __popc(b1);
    return __popc(b1 & lane_lt);
  }
  uint32_t incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= uint32_t(d)) incl += o;
  }
  *total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  return incl - c;
}

// Full tile, 8 elements per lane per row of 256 (4 rows per chunk).
// Same output as encode_chunk<true>: pk/sm of the chunk, its escapes in
// element order in `slot`; returns the escape count.
template <class Stage>
__device__ __forceinline__ uint32_t encode_chunk8(const Stage& st, uint32_t warp, uint32_t lane, uint32_t* slot) {
  const uint8_t* lut = st.enc_lut;
  const uint64_t g = uint64_t(st.lt) * kTile;
  const uint32_t e0 = warp * kChunk + lane * 8u;
  const uint16_t* xw = st.x + e0;
  uint8_t* pkw = st.payload + (g >> 1) + (e0 >> 1);
  uint8_t* smw = st.payload + st.off_sm + g + e0;
  const bool sm8 = ((st.off_sm & 7u) == 0);
  // Escape flags of this lane's 8 elements in the 4 rows: element b (< 4) of
  // row r at bit 8b + 2r, element 4 + b at bit 8b + 2r + 1.  enc_lut values are
  // 0..15 or SZ_ESCAPE_CODE (16): bit 4 of a code marks an escape, whose low
  // nibble, the code packed into pk, is already 0.
  uint32_t lane_esc = 0;
#pragma unroll
  for (int row = 0; row < 4; ++row) {
    const uint4 v = *reinterpret_cast<const uint4*>(xw + row * 256);
    const uint32_t a0 = v.x << 1, a1 = v.y << 1, a2 = v.z << 1, a3 = v.w << 1;
    const uint32_t lo = uint32_t(lut[__byte_perm(a0, 0, 0x4441)]) | (uint32_t(lut[__byte_perm(a0, 0, 0x4443)]) << 8) |
                        (uint32_t(lut[__byte_perm(a1, 0, 0x4441)]) << 16) |
                        (uint32_t(lut[__byte_perm(a1, 0, 0x4443)]) << 24);
    const uint32_t hi = uint32_t(lut[__byte_perm(a2, 0, 0x4441)]) | (uint32_t(lut[__byte_perm(a2, 0, 0x4443)]) << 8) |
                        (uint32_t(lut[__byte_perm(a3, 0, 0x4441)]) << 16) |
                        (uint32_t(lut[__byte_perm(a3, 0, 0x4443)]) << 24);
    lane_esc |= (((lo >> 4) & 0x01010101u) | ((hi >> 3) & 0x02020202u)) << (2 * row);
    const uint32_t clo = lo & 0x0F0F0F0Fu, chi = hi & 0x0F0F0F0Fu;
    const uint32_t tlo = clo | (clo >> 4), thi = chi | (chi >> 4);
    *reinterpret_cast<uint32_t*>(pkw + row * 128) = __byte_perm(tlo, thi, 0x6420);
    const uint32_t s01 = sm_quad(v.x, v.y);
    const uint32_t s23 = sm_quad(v.z, v.w);
    if (sm8) {
      *reinterpret_cast<uint2*>(smw + row * 256) = make_uint2(s01, s23);
    } else {
      *reinterpret_cast<uint32_t*>(smw + row * 256) = s01;
      *reinterpret_cast<uint32_t*>(smw + row * 256 + 4) = s23;
    }
  }
  // Escapes of the chunk, in element order (row, lane, k): one pass per chunk.
  if (__ballot_sync(0xFFFFFFFFu, lane_esc != 0) == 0) return 0;
  const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, uint32_t(__popc(lane_esc)));
  if (total > kStageMax) return total;  // regenerated from the input by the placement pass
  const uint32_t lane_lt = (1u << lane) - 1u;
  const uint16_t* xc = st.x + warp * kChunk;
  uint32_t multi = 0;  // non-zero if this lane has two or more escapes in a row
#pragma unroll
  for (int row = 0; row < 4; ++row) {
    const uint32_t m = (lane_esc >> (2 * row)) & 0x03030303u;
    multi |= m & (m - 1u);
  }
  uint32_t run = 0;
  if (!__any_sync(0xFFFFFFFFu, multi != 0)) {
    // at most one escape per lane and row: a ballot per row places them
#pragma unroll
    for (int row = 0; row < 4; ++row) {
      const uint32_t m = (lane_esc >> (2 * row)) & 0x03030303u;
      const uint32_t b = __ballot_sync(0xFFFFFFFFu, m != 0);
      if (m) {
        const uint32_t p = uint32_t(__ffs(m) - 1);  // 8 (k & 3) + (k >> 2)
        const uint32_t elem = uint32_t(row) * 256u + lane * 8u + (p >> 3) + ((p & 1u) << 2);  // chunk-local
        slot[run + __popc(b & lane_lt)] = elem | ((uint32_t(xc[elem]) << 9) & 0x00FF0000u);
      }
      run += __popc(b);
    }
    return run;
  }
  // Some lane has several escapes in a row: each row's flags as a byte, bit k
  // for element k (bits 0, 8, 16, 24 gathered to 0..3 by one multiply).
  uint32_t bytes[4], before[4];
#pragma unroll
  for (int row = 0; row < 4; ++row) {
    const uint32_t m = lane_esc >> (2 * row);
    const uint32_t m0 = m & 0x01010101u, m1 = (m >> 1) & 0x01010101u;
    bytes[row] = (((m0 * 0x00204081u) >> 21) & 0xFu) | ((((m1 * 0x00204081u) >> 21) & 0xFu) << 4);
    uint32_t total;
    before[row] = run + warp_prefix(__popc(bytes[row]), lane, &total);
    run += total;
  }
#pragma unroll
  for (int row = 0; row < 4; ++row) {
    uint32_t pos = before[row];
    for (uint32_t m = bytes[row]; m; m &= m - 1) {
      const uint32_t elem = uint32_t(row) * 256u + lane * 8u + uint32_t(__ffs(m) - 1);  // chunk-local
      slot[pos] = elem | ((uint32_t(xc[elem]) << 9) & 0x00FF0000u);  // position | exponent << 16
      ++pos;
    }
  }
  return run;
}

// Pad bytes of item `it` (pk -> sm, sm -> chunk_id, local_pos -> esc_val:
// each < 4 bytes), written by threads r = 0..11 of the caller.
__device__ __forceinline__ void finish_pads(const sz_item& it, const Layout& l, uint64_t n, uint32_t e, uint32_t flags,
                                            uint32_t r) {
  if (!flags && r < 12) {
    uint8_t* p = it.payload;
    if (r < 4 && l.n_pairs + r < l.off_sm) p[l.n_pairs + r] = 0;
    if (r >= 4 && r < 8 && l.off_sm + n + (r - 4) < l.off_cid) p[l.off_sm + n + (r - 4)] = 0;
    if (r >= 8 && l.off_lpos + 2ull * e + (r - 8) < l.off_ev) p[l.off_lpos + 2ull * e + (r - 8)] = 0;
  }
}

// The meta of item `it` (coverage: its codebook's), its line of the build
// report of a gated call, and its status bits in the header; one thread.  A
// gated item's meta holds n, its coverage and status SZ_META_GATED only.
__device__ inline void finish_meta(const EncWs& ws, const sz_item& it, const Layout& l, uint64_t n, uint32_t e,
                                   uint32_t flags, double coverage) {
  const bool gated = flags == SZ_META_GATED;
  if (flags && !gated) set_flag(ws.hdr, flags);
  if (it.meta != nullptr && (reinterpret_cast<uintptr_t>(it.meta) & 15) == 0) {
    sz_meta m;
    m.n = n;
    m.n_pairs = gated ? 0 : l.n_pairs;
    m.n_esc = gated ? 0 : e;
    m.comp_bytes = gated ? 0 : l.comp_bytes;
    m.off_pk = 0;
    m.off_sm = gated ? 0 : l.off_sm;
    m.off_cid = gated ? 0 : l.off_cid;
    m.off_lpos = gated ? 0 : l.off_lpos;
    m.off_ev = gated ? 0 : l.off_ev;
    m.chunk_size = kChunk;
    m.status = flags;
    m.coverage = coverage;
    m.reserved1 = 0;
    *it.meta = m;
  }
  if (ws.report != nullptr) {
    sz_gate_report* rep = ws.report;
    if (!flags) {
      atomicAdd(reinterpret_cast<unsigned long long*>(&rep->tensors_encoded), 1ull);
      atomicAdd(reinterpret_cast<unsigned long long*>(&rep->raw_bytes_encoded), 2ull * n);
      atomicAdd(reinterpret_cast<unsigned long long*>(&rep->payload_bytes), l.comp_bytes);
      if (l.comp_bytes > 2ull * n) atomicAdd(reinterpret_cast<unsigned long long*>(&rep->tensors_expanded), 1ull);
      atomicAdd(reinterpret_cast<unsigned long long*>(&rep->escapes), uint64_t(e));
    } else if (gated) {
      atomicAdd(reinterpret_cast<unsigned long long*>(&rep->tensors_gated), 1ull);
      atomicAdd(reinterpret_cast<unsigned long long*>(&rep->raw_bytes_gated), 2ull * n);
    } else {
      atomicAdd(reinterpret_cast<unsigned long long*>(&rep->tensors_failed), 1ull);
    }
  }
}

// The coverage an item's meta records: its codebook's (0 without a usable codebook).
__device__ __forceinline__ double codebook_coverage(const sz_item& it) {
  return (it.codebook && !(reinterpret_cast<uintptr_t>(it.codebook) & 15)) ? it.codebook->coverage : 0.0;
}

// Pads (threads r = 0..11), then meta and report (thread r == 0) of item `it`.
__device__ inline void finish_item(const EncWs& ws, const sz_item& it, const Layout& l, uint64_t n, uint32_t e,
                                   uint32_t flags, uint32_t r) {
  finish_pads(it, l, n, e, flags, r);
  if (r == 0) finish_meta(ws, it, l, n, e, flags, codebook_coverage(it));
}

}  // namespace sz
