// Decode ("splitzip_codec.py" decode_torch): dense reconstruction
// x = ((sm & 0x80) << 8) | (dec_lut[code] << 7) | (sm & 0x7F), then every
// escape overwrites its element with the stored exponent -- here fused into
// one pass that writes each output byte once.
//
// Launches per call (after a 256-byte header memset):
//   dec_prepare  validates each item's meta against the wire layout and the
//                readable payload size, and finds each tile's escape range
//                [k0, k1) by binary search of the sorted chunk_id stream
//                (chunks 8*lt .. 8*lt+7 belong to tile lt);
//   dec_main     persistent CTAs own a contiguous run of tiles.  A producer
//                warp streams pk, sm and the tile's chunk_id/local_pos/esc_val
//                slices into a 4-stage shared-memory ring: TMA bulk copies for
//                the 16-byte-aligned body of each slice and one zero-filling
//                16-byte cp.async for its ragged end, so nothing outside the
//                payload is read.  8 consumer warps decode 8 elements per
//                thread step with the 16-entry dec_lut held in registers
//                (byte permutes), apply the tile's escapes in shared memory and
//                hand the finished 16 KiB tile to a TMA bulk store.
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kDecStages = 4;
constexpr int kDecConsumerWarps = 8;
constexpr int kDecConsumers = kDecConsumerWarps * 32;
constexpr int kDecThreads = kDecConsumers + 32;
constexpr int kDecCtasPerSm = 2;
constexpr uint32_t kEcap = 1024;  // escapes per tile staged in shared memory
constexpr uint32_t kRangeInvalid = 0xFFFFFFFFu;
constexpr uint32_t kStageEnd = 1u, kStageInvalid = 2u, kStageSpill = 4u;

struct __align__(128) DecStage {
  uint8_t pk[kTile / 2 + 16];
  uint8_t sm[kTile + 32];
  uint32_t cid[kEcap + 8];
  uint16_t lpos[kEcap + 16];
  uint8_t ev[kEcap + 32];
  uint4 dec_lut;
  uint16_t* out;
  const uint8_t* payload;  // for tiles whose escapes spill past kEcap
  uint64_t off_cid, off_lpos, off_ev;
  uint32_t k0, m, lt, n_tile, flags;
  uint32_t sm_shift, cid_shift, lpos_shift, ev_shift;
};

struct DecShared {
  DecStage st[kDecStages];
  alignas(128) uint16_t out[2][kTile];
  uint64_t full[kDecStages];
  uint64_t empty[kDecStages];
};

__device__ bool meta_ok(const sz_item& it, uint64_t n_esc_limit) {
  const sz_meta* mp = it.meta;
  if (mp == nullptr || (reinterpret_cast<uintptr_t>(mp) & 15)) return false;
  const sz_meta m = *mp;
  if (m.n != it.n || m.chunk_size != kChunk || m.n_esc > m.n || m.n_esc > n_esc_limit) return false;
  const Layout l = layout_of(m.n, m.n_esc);
  return m.n_pairs == l.n_pairs && m.off_pk == 0 && m.off_sm == l.off_sm && m.off_cid == l.off_cid &&
         m.off_lpos == l.off_lpos && m.off_ev == l.off_ev && m.comp_bytes == l.comp_bytes &&
         l.comp_bytes <= it.capacity;
}

__device__ uint32_t item_problems(const Items& items, uint32_t i) {
  const sz_item& it = item_at(items, i);
  uint32_t bad = 0;
  if (it.n > SZ_MAX_ELEMS) return SZ_FLAG_SIZE;
  if (it.codebook == nullptr || (reinterpret_cast<uintptr_t>(it.codebook) & 15)) bad |= SZ_FLAG_ALIGN;
  if (it.n > 0 && (it.out == nullptr || (reinterpret_cast<uintptr_t>(it.out) & 15))) bad |= SZ_FLAG_ALIGN;
  if (it.n > 0 && (it.payload == nullptr || (reinterpret_cast<uintptr_t>(it.payload) & 15))) bad |= SZ_FLAG_ALIGN;
  if (!meta_ok(it, SZ_MAX_ELEMS)) bad |= SZ_FLAG_META;
  if (items.table) {
    const uint64_t expect = (i == 0) ? 0 : items.table[i - 1].tile_begin + tiles_of(items.table[i - 1].n);
    if (it.tile_begin != expect) bad |= SZ_FLAG_ITEMS;
    if (i + 1 == items.count && it.tile_begin + tiles_of(it.n) != items.total_tiles) bad |= SZ_FLAG_ITEMS;
  }
  return bad;
}

// First k in [0, e) with cid[k] >= target (e if none), found by the 16 lanes
// of a half warp (hl = lane within the half, half_mask = its lanes): each
// round probes 16 evenly spaced positions, so the search takes
// ceil(log16(e)) + 1 dependent loads instead of log2(e).
__device__ uint32_t lower_bound_cid16(const int32_t* cid, uint32_t e, uint32_t target, uint32_t hl,
                                      uint32_t half_mask) {
  uint32_t lo = 0, hi = e;  // the answer lies in [lo, hi]
  while (hi - lo > 16) {
    const uint32_t step = (hi - lo + 15) / 16;
    uint32_t p = lo + (hl + 1) * step - 1;
    if (p > hi - 1) p = hi - 1;
    const uint32_t c = __popc(__ballot_sync(half_mask, uint32_t(__ldg(cid + p)) < target));
    if (c == 0) {
      hi = lo + step - 1;  // the first probe already holds cid >= target
    } else {
      uint32_t last_less = lo + c * step - 1;
      if (last_less > hi - 1) last_less = hi - 1;
      if (c < 16) {
        uint32_t first_ge = lo + (c + 1) * step - 1;
        if (first_ge < hi) hi = first_ge;
      }
      lo = last_less + 1;
    }
  }
  const uint32_t p = lo + hl;
  const bool less = (p < hi) && uint32_t(__ldg(cid + p)) < target;
  return lo + __popc(__ballot_sync(half_mask, less));
}

constexpr int kPrepWarps = 8;

// Escape ranges per tile.  blockIdx.y = item; each warp owns a group of 32
// consecutive tiles of that item (lane l <-> tile ta + l).  The two half
// warps bracket the group's escapes with 16-ary searches for the first
// escape of tile ta and of tile ta + 32; the warp then reads the bracketed
// chunk_id slice once, coalesced, counting escapes per tile in shared
// memory, and a warp scan of the counts gives every tile's [k0, k1).
__global__ void __launch_bounds__(kPrepWarps * 32) dec_prepare(const __grid_constant__ Items items, DecWs ws) {
  __shared__ uint32_t s_bad;
  __shared__ uint32_t counts[kPrepWarps][32];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  for (uint32_t i = blockIdx.y; i < items.count; i += gridDim.y) {
    const sz_item& it = item_at(items, i);
    __syncthreads();
    if (threadIdx.x == 0) {
      s_bad = item_problems(items, i);
      if (blockIdx.x == 0) {
        ws.item_flags[i] = s_bad;
        if (s_bad) set_flag(ws.hdr, s_bad);
      }
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    const uint64_t tiles = (it.n > SZ_MAX_ELEMS) ? 0 : tiles_of(it.n);
    const uint32_t e = bad ? 0u : uint32_t(it.meta->n_esc);
    const int32_t* cid = bad ? nullptr : reinterpret_cast<const int32_t*>(it.payload + it.meta->off_cid);
    const uint32_t half_mask = lane < 16 ? 0x0000FFFFu : 0xFFFF0000u;
    for (uint64_t ta = (uint64_t(blockIdx.x) * kPrepWarps + warp) * 32; ta < tiles;
         ta += uint64_t(gridDim.x) * kPrepWarps * 32) {
      const uint32_t ng = (tiles - ta < 32) ? uint32_t(tiles - ta) : 32u;
      uint2 r = make_uint2(kRangeInvalid, 0);
      if (!bad) {
        const uint32_t target = uint32_t(ta) * kChunksPerTile + (lane < 16 ? 0u : 32u * kChunksPerTile);
        const uint32_t k = lower_bound_cid16(cid, e, target, lane & 15u, half_mask);
        const uint32_t k_lo = __shfl_sync(0xFFFFFFFFu, k, 0);
        const uint32_t k_hi = __shfl_sync(0xFFFFFFFFu, k, 16);
        counts[warp][lane] = 0;
        __syncwarp();
        // 8 independent loads per lane per round, then the shared-memory counts
        for (uint32_t kb = k_lo; kb < k_hi; kb += 32 * 8) {
          uint32_t c8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t kk = kb + lane + 32u * u;
            c8[u] = kk < k_hi ? uint32_t(__ldg(cid + kk)) : 0xFFFFFFFFu;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t rel = (c8[u] >> 3) - uint32_t(ta);  // tile within the group
            if (c8[u] != 0xFFFFFFFFu && rel < 32u) atomicAdd(&counts[warp][rel], 1u);
          }
        }
        __syncwarp();
        const uint32_t c = counts[warp][lane];
        uint32_t incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
          if (lane >= uint32_t(d)) incl += o;
        }
        r = make_uint2(k_lo + incl - c, k_lo + incl);
      }
      if (lane < ng) ws.ranges[it.tile_begin + ta + lane] = r;
    }
  }
}

// Decodes 4 elements: c16 holds their 4-bit codes (element j in nibble j),
// s4 their sm bytes (element j in byte j); d0..d3 = dec_lut bytes 0..15.
// Returns the 4 BF16 patterns as two words (element 2j in the low half).
__device__ __forceinline__ uint2 decode4(uint32_t c16, uint32_t s4, uint32_t d0, uint32_t d1, uint32_t d2,
                                         uint32_t d3) {
  const uint32_t sel = c16 & 0x7777u;
  const uint32_t lo = __byte_perm(d0, d1, sel);   // dec_lut[c] for c < 8
  const uint32_t hi = __byte_perm(d2, d3, sel);   // dec_lut[c] for c >= 8
  const uint32_t e4 = __byte_perm(lo, hi, ((c16 >> 1) & 0x4444u) | 0x3210u);
  const uint32_t y0 = __byte_perm(s4, e4, 0x5140u);  // sm0 e0 sm1 e1
  const uint32_t y1 = __byte_perm(s4, e4, 0x7362u);  // sm2 e2 sm3 e3
  uint2 r;
  r.x = ((y0 >> 1) & 0x7F807F80u) | (y0 & 0x007F007Fu) | ((y0 << 8) & 0x80008000u);
  r.y = ((y1 >> 1) & 0x7F807F80u) | (y1 & 0x007F007Fu) | ((y1 << 8) & 0x80008000u);
  return r;
}

__device__ __forceinline__ uint16_t merge_one(uint32_t sm, uint32_t exp) {
  return uint16_t(((sm & 0x80u) << 8) | ((exp & 0xFFu) << 7) | (sm & 0x7Fu));
}

// One slice copy into shared memory: the aligned body by TMA (issued by the
// caller's lane 0), the ragged end by a zero-filling cp.async.  Returns the
// shift of the slice start inside the staged bytes.
struct Slice {
  uint64_t a0, a1, end;  // a0 = floor16(start), a1 = floor16(end)
};
__device__ __forceinline__ Slice slice_of(uint64_t start, uint64_t bytes) {
  Slice s;
  s.a0 = start & ~uint64_t(15);
  s.end = start + bytes;
  s.a1 = s.end & ~uint64_t(15);
  if (s.a1 < s.a0) s.a1 = s.a0;
  return s;
}

__global__ void __launch_bounds__(kDecThreads, kDecCtasPerSm)
    dec_main(const __grid_constant__ Items items, DecWs ws) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  DecShared& sh = *reinterpret_cast<DecShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // an inconsistent item table (flagged by dec_prepare) is never walked
  if (ws.hdr->flags & SZ_FLAG_ITEMS) return;

  const uint64_t T = items.total_tiles;
  const uint64_t per = (T + gridDim.x - 1) / gridDim.x;
  const uint64_t t0 = uint64_t(blockIdx.x) * per;
  const uint64_t t1 = (t0 + per < T) ? t0 + per : T;

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&sh.full[s], 1 + 32);
      mbar_init(&sh.empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDecConsumerWarps) {
    // ---------------------------------------------------------------- producer warp
    uint32_t cur = 0xFFFFFFFFu;
    uint64_t cur_begin = 0, cur_end = 0;
    uint4 dlut = make_uint4(0, 0, 0, 0);
    uint2 rec = make_uint2(0, 0);
    for (uint64_t t = t0, it = 0;; ++t, ++it) {
      const int s = int(it % kDecStages);
      if (it >= uint64_t(kDecStages)) {
        if (!mbar_wait(&sh.empty[s], uint32_t((it / kDecStages) - 1) & 1)) {
          if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
          return;
        }
      }
      DecStage& st = sh.st[s];
      if (t >= t1) {
        if (lane == 0) {
          st.flags = kStageEnd;
          mbar_arrive(&sh.full[s]);
        }
        cp_async_mbar_arrive_noinc(&sh.full[s]);
        return;
      }
      // escape ranges of the next 32 tiles, one per lane
      if (((t - t0) & 31) == 0) {
        const uint64_t mine = t + lane;
        rec = (mine < t1) ? ws.ranges[mine] : make_uint2(kRangeInvalid, 0);
      }
      const uint32_t src_lane = uint32_t((t - t0) & 31);
      const uint32_t k0 = __shfl_sync(0xFFFFFFFFu, rec.x, src_lane);
      const uint32_t k1 = __shfl_sync(0xFFFFFFFFu, rec.y, src_lane);
      if (t >= cur_end) {
        cur = find_item(items, t);
        cur_begin = item_at(items, cur).tile_begin;
        cur_end = cur_begin + tiles_of(item_at(items, cur).n);
        if (ws.item_flags[cur] == 0) dlut = *reinterpret_cast<const uint4*>(item_at(items, cur).codebook->dec_lut);
      }
      const sz_item& itm = item_at(items, cur);
      const uint32_t lt = uint32_t(t - cur_begin);
      const uint64_t g = uint64_t(lt) * kTile;
      const bool invalid = (k0 == kRangeInvalid) || ws.item_flags[cur] != 0 || g >= itm.n;
      const uint32_t nt = invalid ? 0u : ((itm.n - g < kTile) ? uint32_t(itm.n - g) : kTile);
      if (invalid) {
        if (lane == 0) {
          st.flags = kStageInvalid;
          mbar_arrive(&sh.full[s]);
        }
        cp_async_mbar_arrive_noinc(&sh.full[s]);
        continue;
      }
      const sz_meta* mp = itm.meta;
      const uint64_t off_sm = mp->off_sm, off_cid = mp->off_cid, off_lpos = mp->off_lpos, off_ev = mp->off_ev;
      const uint8_t* base = itm.payload;
      const uint32_t m = (k1 > k0) ? k1 - k0 : 0u;
      const bool spill = m > kEcap;
      const Slice spk = slice_of(g >> 1, (nt + 1) >> 1);
      const Slice ssm = slice_of(off_sm + g, nt);
      Slice scid = slice_of(off_cid + 4ull * k0, 4ull * m);
      Slice slp = slice_of(off_lpos + 2ull * k0, 2ull * m);
      Slice sev = slice_of(off_ev + k0, m);
      const bool esc_smem = (m > 0) && !spill;
      const uint32_t tx = uint32_t(spk.a1 - spk.a0) + uint32_t(ssm.a1 - ssm.a0) +
                          (esc_smem ? uint32_t(scid.a1 - scid.a0) + uint32_t(slp.a1 - slp.a0) +
                                          uint32_t(sev.a1 - sev.a0)
                                    : 0u);
      if (lane == 0) {
        st.dec_lut = dlut;
        st.out = itm.out + g;
        st.payload = base;
        st.off_cid = off_cid;
        st.off_lpos = off_lpos;
        st.off_ev = off_ev;
        st.k0 = k0;
        st.m = m;
        st.lt = lt;
        st.n_tile = nt;
        st.flags = spill ? kStageSpill : 0u;
        st.sm_shift = uint32_t(off_sm + g - ssm.a0);
        st.cid_shift = uint32_t(off_cid + 4ull * k0 - scid.a0);
        st.lpos_shift = uint32_t(off_lpos + 2ull * k0 - slp.a0);
        st.ev_shift = uint32_t(off_ev + k0 - sev.a0);
        mbar_arrive_expect_tx(&sh.full[s], tx);
        if (spk.a1 > spk.a0) bulk_g2s(st.pk, base + spk.a0, uint32_t(spk.a1 - spk.a0), &sh.full[s]);
        if (ssm.a1 > ssm.a0) bulk_g2s(st.sm, base + ssm.a0, uint32_t(ssm.a1 - ssm.a0), &sh.full[s]);
        if (esc_smem) {
          if (scid.a1 > scid.a0) bulk_g2s(st.cid, base + scid.a0, uint32_t(scid.a1 - scid.a0), &sh.full[s]);
          if (slp.a1 > slp.a0) bulk_g2s(st.lpos, base + slp.a0, uint32_t(slp.a1 - slp.a0), &sh.full[s]);
          if (sev.a1 > sev.a0) bulk_g2s(st.ev, base + sev.a0, uint32_t(sev.a1 - sev.a0), &sh.full[s]);
        }
      } else if (lane == 1 && spk.end > spk.a1) {
        cp_async16_zfill(st.pk + (spk.a1 - spk.a0), base + spk.a1, uint32_t(spk.end - spk.a1));
      } else if (lane == 2 && ssm.end > ssm.a1) {
        cp_async16_zfill(st.sm + (ssm.a1 - ssm.a0), base + ssm.a1, uint32_t(ssm.end - ssm.a1));
      } else if (esc_smem && lane == 3 && scid.end > scid.a1) {
        cp_async16_zfill(reinterpret_cast<uint8_t*>(st.cid) + (scid.a1 - scid.a0), base + scid.a1,
                         uint32_t(scid.end - scid.a1));
      } else if (esc_smem && lane == 4 && slp.end > slp.a1) {
        cp_async16_zfill(reinterpret_cast<uint8_t*>(st.lpos) + (slp.a1 - slp.a0), base + slp.a1,
                         uint32_t(slp.end - slp.a1));
      } else if (esc_smem && lane == 5 && sev.end > sev.a1) {
        cp_async16_zfill(st.ev + (sev.a1 - sev.a0), base + sev.a1, uint32_t(sev.end - sev.a1));
      }
      cp_async_mbar_arrive_noinc(&sh.full[s]);
    }
  }

  // ------------------------------------------------------------------ consumer warps
  uint32_t bad_escape = 0;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kDecStages);
    const int ob = int(it & 1);
    if (tid == 0) bulk_wait_read<1>();  // the store that last used out[ob] has read it
    const bool ok = mbar_wait(&sh.full[s], (it / kDecStages) & 1);
    const DecStage& st = sh.st[s];
    // read before the vote: after it, an invalid tile's stage is released
    const uint32_t flags = ok ? st.flags : 0u;
    if (named_bar_red_or(1, kDecConsumers, !ok)) {
      if (tid == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      break;
    }
    if (flags & kStageEnd) break;
    if (flags & kStageInvalid) {
      if (tid == 0) mbar_arrive(&sh.empty[s]);
      continue;
    }
    const uint32_t nt = st.n_tile;
    uint16_t* const outs = sh.out[ob];
    {
      const uint4 dl = st.dec_lut;
      const uint32_t shift = st.sm_shift;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t grp = uint32_t(tid) + uint32_t(j) * kDecConsumers;  // 8 elements
        if (grp * 8u < nt) {
          const uint32_t c8 = *reinterpret_cast<const uint32_t*>(st.pk + grp * 4u);
          const uint32_t s_lo = *reinterpret_cast<const uint32_t*>(st.sm + shift + grp * 8u);
          const uint32_t s_hi = *reinterpret_cast<const uint32_t*>(st.sm + shift + grp * 8u + 4u);
          const uint2 a = decode4(c8 & 0xFFFFu, s_lo, dl.x, dl.y, dl.z, dl.w);
          const uint2 b = decode4(c8 >> 16, s_hi, dl.x, dl.y, dl.z, dl.w);
          *reinterpret_cast<uint4*>(outs + grp * 8u) = make_uint4(a.x, a.y, b.x, b.y);
        }
      }
    }
    const uint32_t m = st.m;
    if (m) {
      named_bar_sync(1, kDecConsumers);
      const bool spill = flags & kStageSpill;
      const uint32_t chunk0 = st.lt * kChunksPerTile;
      for (uint32_t k = uint32_t(tid); k < m; k += kDecConsumers) {
        uint32_t c, p, ev;
        if (!spill) {
          c = st.cid[(st.cid_shift >> 2) + k];
          p = st.lpos[(st.lpos_shift >> 1) + k];
          ev = st.ev[st.ev_shift + k];
        } else {
          const uint64_t kk = uint64_t(st.k0) + k;
          c = *reinterpret_cast<const uint32_t*>(st.payload + st.off_cid + 4 * kk);
          p = *reinterpret_cast<const uint16_t*>(st.payload + st.off_lpos + 2 * kk);
          ev = st.payload[st.off_ev + kk];
        }
        const uint32_t rel = c - chunk0;
        const uint32_t pos = rel * kChunk + p;
        if (rel < kChunksPerTile && p < kChunk && pos < nt) {
          outs[pos] = merge_one(st.sm[st.sm_shift + pos], ev);
        } else {
          bad_escape = 1;
        }
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, kDecConsumers);
    if (tid == 0) {
      uint16_t* const outp = st.out;  // the stage may be refilled once released
      mbar_arrive(&sh.empty[s]);
      const uint32_t body = (nt * 2u) & ~15u;
      if (body) bulk_s2g(outp, outs, body);
      bulk_commit();
      for (uint32_t k = body / 2u; k < nt; ++k) outp[k] = outs[k];
    }
  }
  if (bad_escape) set_flag(ws.hdr, SZ_FLAG_ESCAPE);
  if (tid == 0) bulk_wait_all<0>();
}

}  // namespace

cudaError_t launch_decode(const Items& items, void* ws_base, cudaStream_t stream, const DeviceInfo& dev) {
  DecWs ws = dec_ws(ws_base, items.count, items.total_tiles);
  cudaError_t err = cudaMemsetAsync(ws_base, 0, sizeof(WsHeader), stream);
  if (err != cudaSuccess) return err;
  {
    // blockIdx.y = item; x covers the average item's 32-tile groups (8 per block)
    const uint64_t per_item = items.count ? (items.total_tiles + items.count - 1) / items.count : 0;
    uint64_t gx = (per_item + 32 * kPrepWarps - 1) / (32 * kPrepWarps);
    if (gx < 1) gx = 1;
    if (gx > 1024) gx = 1024;
    const unsigned gy = items.count < 65535u ? items.count : 65535u;
    dec_prepare<<<dim3(unsigned(gx), gy), kPrepWarps * 32, 0, stream>>>(items, ws);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (items.total_tiles == 0) return cudaSuccess;
  static thread_local int configured_device = -1;
  const size_t smem = sizeof(DecShared);
  if (configured_device != dev.device) {
    err = cudaFuncSetAttribute(dec_main, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    configured_device = dev.device;
  }
  const uint64_t cap = uint64_t(dev.num_sms) * kDecCtasPerSm;
  const unsigned grid = unsigned(items.total_tiles < cap ? items.total_tiles : cap);
  if (g_timing.before) cudaEventRecord(g_timing.before, stream);
  dec_main<<<grid, kDecThreads, smem, stream>>>(items, ws);
  err = cudaGetLastError();
  if (g_timing.after) cudaEventRecord(g_timing.after, stream);
  return err;
}

}  // namespace sz
