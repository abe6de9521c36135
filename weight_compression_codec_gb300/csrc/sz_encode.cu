// Encode ("splitzip_codec.py" encode_torch + assemble_payload), one pass over
// the input with in-order escape compaction.
//
// Launches per call (after a 256-byte header memset):
//   enc_prepare  validates the item table and zeroes the tile status words;
//   enc_main     persistent CTAs take 8192-element tiles from a device-wide
//                ticket (so tiles start in ascending order), stream them in
//                with TMA bulk copies through a 4-stage shared-memory ring and
//                write pk and sm with coalesced stores.  Warp w of the 8
//                consumer warps owns chunk w of the tile, so its ballot/popc
//                escape count is the chunk's; a block scan gives the tile's
//                count, and a decoupled lookback over the tile status words
//                gives the tile's first global escape index.  chunk_id is then
//                written in place (its offset depends on n only); local_pos
//                and esc_val go to a per-item staging area because their
//                offsets depend on the total escape count;
//   enc_tail     moves local_pos/esc_val to their final offsets, zeroes every
//                pad byte and writes the meta.
//
// Lookback status word per tile (64 bits): flag in the high half (1 = tile
// aggregate, 2 = inclusive prefix), escape count in the low half.  Every wait
// is bounded (kWaitTimeoutNs); on timeout SZ_FLAG_TIMEOUT is raised.
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kEncStages = 4;
constexpr int kEncConsumerWarps = kChunksPerTile;  // one warp per chunk
constexpr int kEncConsumers = kEncConsumerWarps * 32;
constexpr int kEncThreads = kEncConsumers + 32;    // + producer warp
constexpr int kEncCtasPerSm = 2;
constexpr uint32_t kStageEnd = 1u, kStageInvalid = 2u;
constexpr unsigned long long kAgg = 1ull << 32, kIncl = 2ull << 32;

struct __align__(128) EncStage {
  uint16_t x[kTile];      // the tile's BF16 bit patterns
  uint8_t enc_lut[256];   // the item's codebook enc_lut
  unsigned long long ticket;
  uint8_t* payload;
  uint16_t* lpos_stage;
  uint8_t* ev_stage;
  uint64_t off_sm, off_cid, capacity;
  uint32_t lt, n_tile, flags, item;
};

struct EncShared {
  EncStage st[kEncStages];
  uint64_t full[kEncStages];
  uint64_t empty[kEncStages];
  uint32_t warp_cnt[kEncConsumerWarps];
  uint32_t warp_off[kEncConsumerWarps];
  uint32_t tile_base;
};

__global__ void enc_prepare(const __grid_constant__ Items items, EncWs ws) {
  const uint64_t nthreads = uint64_t(gridDim.x) * blockDim.x;
  const uint64_t gtid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (uint64_t t = gtid; t < items.total_tiles; t += nthreads) ws.status[t] = 0ull;
  for (uint64_t i = gtid; i < items.count; i += nthreads) {
    const sz_item& it = item_at(items, uint32_t(i));
    uint32_t bad = 0;
    if (it.n > SZ_MAX_ELEMS) bad |= SZ_FLAG_SIZE;
    if (it.codebook == nullptr || (reinterpret_cast<uintptr_t>(it.codebook) & 15)) bad |= SZ_FLAG_ALIGN;
    if (it.meta == nullptr || (reinterpret_cast<uintptr_t>(it.meta) & 15)) bad |= SZ_FLAG_ALIGN;
    if (it.n > 0 && (it.x == nullptr || (reinterpret_cast<uintptr_t>(it.x) & 15))) bad |= SZ_FLAG_ALIGN;
    if (it.n > 0 && (it.payload == nullptr || (reinterpret_cast<uintptr_t>(it.payload) & 15))) bad |= SZ_FLAG_ALIGN;
    if (!(bad & SZ_FLAG_SIZE) && layout_of(it.n, 0).off_cid > it.capacity) bad |= SZ_FLAG_CAPACITY;
    if (items.table) {
      const uint64_t expect = (i == 0) ? 0 : items.table[i - 1].tile_begin + tiles_of(items.table[i - 1].n);
      if (it.tile_begin != expect) bad |= SZ_FLAG_ITEMS;
      if (i + 1 == items.count && it.tile_begin + tiles_of(it.n) != items.total_tiles) bad |= SZ_FLAG_ITEMS;
    }
    ws.item_flags[i] = bad;
    if (bad) set_flag(ws.hdr, bad);
  }
}

// Walks back from tile j (inclusive) accumulating aggregates until an
// inclusive prefix is found.  Returns the exclusive prefix of tile j + 1.
__device__ uint32_t lookback(const unsigned long long* status, uint64_t j, bool* timed_out) {
  uint32_t excl = 0;
  uint64_t t0 = 0;
  uint32_t spins = 0;
  for (;;) {
    const unsigned long long v = ld_acquire_u64(status + j);
    const unsigned long long flag = v & ~0xFFFFFFFFull;
    if (flag == 0) {
      if ((++spins & 31) == 0) {
        const uint64_t now = global_timer_ns();
        if (t0 == 0) t0 = now;
        else if (now - t0 > kWaitTimeoutNs) {
          *timed_out = true;
          return excl;
        }
      }
      continue;
    }
    excl += uint32_t(v);
    if (flag == kIncl) return excl;
    --j;
  }
}

__device__ __forceinline__ uint32_t sm_pair(uint32_t w) {
  // two BF16 patterns in w -> sm bytes at byte 0 and byte 2
  return (w & 0x007F007Fu) | ((w >> 8) & 0x00800080u);
}

__global__ void __launch_bounds__(kEncThreads, kEncCtasPerSm)
    enc_main(const __grid_constant__ Items items, EncWs ws) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  EncShared& sh = *reinterpret_cast<EncShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // an inconsistent item table (flagged by enc_prepare) is never walked
  if (ws.hdr->flags & SZ_FLAG_ITEMS) return;

  if (tid == 0) {
    for (int s = 0; s < kEncStages; ++s) {
      mbar_init(&sh.full[s], 1 + 32);
      mbar_init(&sh.empty[s], kEncConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kEncConsumerWarps) {
    // ---------------------------------------------------------------- producer warp
    unsigned long long ticket = 0;
    if (lane == 0) ticket = atomicAdd(&ws.hdr->ticket, 1ull);
    uint32_t cur = 0xFFFFFFFFu;
    uint64_t cur_begin = 0;
    for (uint32_t it = 0;; ++it) {
      const int s = int(it % kEncStages);
      if (it >= uint32_t(kEncStages)) {
        if (!mbar_wait(&sh.empty[s], ((it / kEncStages) - 1) & 1)) {
          if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
          return;
        }
      }
      ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
      EncStage& st = sh.st[s];
      if (ticket >= items.total_tiles) {
        if (lane == 0) {
          st.flags = kStageEnd;
          mbar_arrive(&sh.full[s]);
        }
        cp_async_mbar_arrive_noinc(&sh.full[s]);
        return;
      }
      if (cur == 0xFFFFFFFFu || ticket < cur_begin || ticket >= cur_begin + tiles_of(item_at(items, cur).n)) {
        cur = find_item(items, ticket);
        cur_begin = item_at(items, cur).tile_begin;
      }
      const sz_item& itm = item_at(items, cur);
      const uint32_t lt = uint32_t(ticket - cur_begin);
      const uint64_t g = uint64_t(lt) * kTile;
      const bool invalid = ws.item_flags[cur] != 0 || g >= itm.n;
      const uint32_t nt = invalid ? 0u : ((itm.n - g < kTile) ? uint32_t(itm.n - g) : kTile);
      const uint32_t bulk = invalid ? 0u : ((nt * 2u) & ~15u);
      const uint32_t tail = invalid ? 0u : (nt * 2u - bulk);
      if (lane == 0) {
        st.ticket = ticket;
        st.item = cur;
        st.lt = lt;
        st.n_tile = nt;
        st.flags = invalid ? kStageInvalid : 0u;
        if (!invalid) {
          const Layout l = layout_of(itm.n, 0);
          st.payload = itm.payload;
          st.off_sm = l.off_sm;
          st.off_cid = l.off_cid;
          st.capacity = itm.capacity;
          st.lpos_stage = ws.lpos + cur_begin * kTile;
          st.ev_stage = ws.ev + cur_begin * kTile;
        }
        if (invalid) {
          mbar_arrive(&sh.full[s]);
        } else {
          mbar_arrive_expect_tx(&sh.full[s], bulk + 256u);
          if (bulk) bulk_g2s(st.x, itm.x + g, bulk, &sh.full[s]);
          bulk_g2s(st.enc_lut, itm.codebook->enc_lut, 256u, &sh.full[s]);
        }
      } else if (lane == 1 && tail) {
        cp_async16_zfill(reinterpret_cast<uint8_t*>(st.x) + bulk,
                         reinterpret_cast<const uint8_t*>(itm.x + g) + bulk, tail);
      }
      cp_async_mbar_arrive_noinc(&sh.full[s]);
      if (lane == 0) ticket = atomicAdd(&ws.hdr->ticket, 1ull);
    }
  }

  // ------------------------------------------------------------------ consumer warps
  const unsigned FULL = 0xFFFFFFFFu;
  const uint32_t lane_lt = (1u << lane) - 1u;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    // every consumer thread waits (bounded); the vote keeps all warps on the
    // same path so no named barrier below can be left short of threads
    const bool ok = mbar_wait(&sh.full[s], (it / kEncStages) & 1);
    if (named_bar_red_or(1, kEncConsumers, !ok)) {
      if (tid == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      break;
    }
    const EncStage& st = sh.st[s];
    const uint32_t flags = st.flags;
    if (flags & kStageEnd) break;
    const bool valid = !(flags & kStageInvalid);
    const uint32_t nt = st.n_tile;
    const uint32_t lt = st.lt;
    const uint64_t g = uint64_t(lt) * kTile;
    uint32_t wcnt = 0, esc_rows = 0;

    if (valid) {
      uint8_t* const pk = st.payload + (g >> 1);
      uint8_t* const smp = st.payload + st.off_sm + g;
#pragma unroll 2
      for (int row = 0; row < 8; ++row) {
        const uint32_t il = uint32_t(warp) * kChunk + uint32_t(row) * 128u + uint32_t(lane) * 4u;
        const uint2 v = *reinterpret_cast<const uint2*>(st.x + il);
        const uint32_t e0 = (v.x >> 7) & 0xFFu, e1 = (v.x >> 23) & 0xFFu;
        const uint32_t e2 = (v.y >> 7) & 0xFFu, e3 = (v.y >> 23) & 0xFFu;
        uint32_t c0 = st.enc_lut[e0], c1 = st.enc_lut[e1], c2 = st.enc_lut[e2], c3 = st.enc_lut[e3];
        const uint32_t nvalid = (il < nt) ? ((nt - il) < 4u ? nt - il : 4u) : 0u;
        if (nvalid < 4) {
          if (nvalid < 4) c3 = 0;
          if (nvalid < 3) c2 = 0;
          if (nvalid < 2) c1 = 0;
          if (nvalid < 1) c0 = 0;
        }
        // any enc_lut value >= 16 marks an escape, stored as code 0
        const uint32_t escm = uint32_t(c0 > 15u) | (uint32_t(c1 > 15u) << 1) | (uint32_t(c2 > 15u) << 2) |
                              (uint32_t(c3 > 15u) << 3);
        c0 = c0 > 15u ? 0u : c0;
        c1 = c1 > 15u ? 0u : c1;
        c2 = c2 > 15u ? 0u : c2;
        c3 = c3 > 15u ? 0u : c3;
        const uint32_t pk16 = c0 | (c1 << 4) | (c2 << 8) | (c3 << 12);
        const uint32_t sm4 = __byte_perm(sm_pair(v.x), sm_pair(v.y), 0x6420);
        if (nvalid == 4) {
          *reinterpret_cast<uint16_t*>(pk + (il >> 1)) = uint16_t(pk16);
          *reinterpret_cast<uint32_t*>(smp + il) = sm4;
        } else if (nvalid > 0) {
          pk[il >> 1] = uint8_t(pk16);
          if (nvalid > 2) pk[(il >> 1) + 1] = uint8_t(pk16 >> 8);
          for (uint32_t k = 0; k < nvalid; ++k) smp[il + k] = uint8_t(sm4 >> (8 * k));
        }
        const uint32_t rowcnt = __reduce_add_sync(FULL, __popc(escm));
        if (rowcnt) {
          esc_rows |= 1u << row;
          wcnt += rowcnt;
        }
      }
    }
    if (lane == 0) sh.warp_cnt[warp] = wcnt;
    named_bar_sync(1, kEncConsumers);
    if (tid == 0) {
      uint32_t agg = 0;
      for (int w = 0; w < kEncConsumerWarps; ++w) {
        sh.warp_off[w] = agg;
        agg += sh.warp_cnt[w];
      }
      unsigned long long* status = ws.status;
      const unsigned long long ticket = st.ticket;
      uint32_t base = 0;
      if (!valid || lt == 0) {
        st_release_u64(status + ticket, kIncl | agg);
      } else {
        st_release_u64(status + ticket, kAgg | agg);
        bool timed_out = false;
        base = lookback(status, ticket - 1, &timed_out);
        if (timed_out) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        st_release_u64(status + ticket, kIncl | (base + agg));
      }
      sh.tile_base = base;
    }
    named_bar_sync(1, kEncConsumers);
    if (esc_rows) {
      uint32_t e_idx = sh.tile_base + sh.warp_off[warp];
      const uint32_t chunk_id = lt * kChunksPerTile + uint32_t(warp);
      uint8_t* const cidp = st.payload + st.off_cid;
      const uint64_t cap = st.capacity;
      uint16_t* const lps = st.lpos_stage;
      uint8_t* const evs = st.ev_stage;
      for (int row = 0; row < 8; ++row) {
        if (!((esc_rows >> row) & 1u)) continue;
        const uint32_t il = uint32_t(warp) * kChunk + uint32_t(row) * 128u + uint32_t(lane) * 4u;
        const uint2 v = *reinterpret_cast<const uint2*>(st.x + il);
        uint32_t e[4] = {(v.x >> 7) & 0xFFu, (v.x >> 23) & 0xFFu, (v.y >> 7) & 0xFFu, (v.y >> 23) & 0xFFu};
        uint32_t escm = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (il + k < nt && st.enc_lut[e[k]] > 15u) escm |= 1u << k;
        const uint32_t b0 = __ballot_sync(FULL, escm & 1u), b1 = __ballot_sync(FULL, escm & 2u);
        const uint32_t b2 = __ballot_sync(FULL, escm & 4u), b3 = __ballot_sync(FULL, escm & 8u);
        uint32_t pos = e_idx + __popc(b0 & lane_lt) + __popc(b1 & lane_lt) + __popc(b2 & lane_lt) +
                       __popc(b3 & lane_lt);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if ((escm >> k) & 1u) {
            const uint64_t cid_off = st.off_cid + 4ull * pos;
            if (cid_off + 4 <= cap) *reinterpret_cast<uint32_t*>(cidp + 4ull * pos) = chunk_id;
            lps[pos] = uint16_t(row * 128 + lane * 4 + k);
            evs[pos] = uint8_t(e[k]);
            ++pos;
          }
        }
        e_idx += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
  }
}

// One CTA row (blockIdx.y) per item; blockIdx.x strides over its escapes.
__global__ void enc_tail(const __grid_constant__ Items items, EncWs ws) {
  for (uint32_t i = blockIdx.y; i < items.count; i += gridDim.y) {
    const sz_item& it = item_at(items, i);
    uint32_t flags = ws.item_flags[i];
    const uint64_t tiles = tiles_of(it.n);
    uint64_t e = 0;
    if (!flags && tiles) {
      const unsigned long long v = ws.status[it.tile_begin + tiles - 1];
      if ((v & ~0xFFFFFFFFull) != kIncl) flags |= SZ_FLAG_TIMEOUT;
      e = uint32_t(v);
    }
    const Layout l = layout_of(it.n, e);
    if (!flags && l.comp_bytes > it.capacity) flags |= SZ_FLAG_CAPACITY;
    if (!flags) {
      uint8_t* p = it.payload;
      const uint16_t* lps = ws.lpos + it.tile_begin * kTile;
      const uint8_t* evs = ws.ev + it.tile_begin * kTile;
      const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
      for (uint64_t k = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < e; k += stride) {
        *reinterpret_cast<uint16_t*>(p + l.off_lpos + 2 * k) = lps[k];
        p[l.off_ev + k] = evs[k];
      }
      if (blockIdx.x == 0 && threadIdx.x < 16) {
        // pad bytes: pk -> sm, sm -> chunk_id, local_pos -> esc_val (each < 4 bytes)
        const uint32_t t = threadIdx.x;
        if (t < 4 && l.n_pairs + t < l.off_sm) p[l.n_pairs + t] = 0;
        if (t >= 4 && t < 8 && l.off_sm + it.n + (t - 4) < l.off_cid) p[l.off_sm + it.n + (t - 4)] = 0;
        if (t >= 8 && t < 12 && l.off_lpos + 2 * e + (t - 8) < l.off_ev) p[l.off_lpos + 2 * e + (t - 8)] = 0;
      }
    }
    if (flags) {
      if (blockIdx.x == 0 && threadIdx.x == 0) set_flag(ws.hdr, flags);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && it.meta != nullptr &&
        (reinterpret_cast<uintptr_t>(it.meta) & 15) == 0) {
      sz_meta m;
      m.n = it.n;
      m.n_pairs = l.n_pairs;
      m.n_esc = e;
      m.comp_bytes = l.comp_bytes;
      m.off_pk = 0;
      m.off_sm = l.off_sm;
      m.off_cid = l.off_cid;
      m.off_lpos = l.off_lpos;
      m.off_ev = l.off_ev;
      m.chunk_size = kChunk;
      m.status = flags;
      m.coverage = (it.codebook && !(reinterpret_cast<uintptr_t>(it.codebook) & 15)) ? it.codebook->coverage : 0.0;
      m.reserved1 = 0;
      *it.meta = m;
    }
  }
}

}  // namespace

cudaError_t launch_encode(const Items& items, void* ws_base, cudaStream_t stream, const DeviceInfo& dev) {
  EncWs ws = enc_ws(ws_base, items.count, items.total_tiles);
  cudaError_t err = cudaMemsetAsync(ws_base, 0, sizeof(WsHeader), stream);
  if (err != cudaSuccess) return err;
  {
    const uint64_t work = items.total_tiles > items.count ? items.total_tiles : items.count;
    const uint64_t blocks = (work + 255) / 256;
    const unsigned grid = unsigned(blocks < 2048 ? (blocks ? blocks : 1) : 2048);
    enc_prepare<<<grid, 256, 0, stream>>>(items, ws);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (items.total_tiles > 0) {
    static thread_local int configured_device = -1;
    const size_t smem = sizeof(EncShared);
    if (configured_device != dev.device) {
      err = cudaFuncSetAttribute(enc_main, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (err != cudaSuccess) return err;
      configured_device = dev.device;
    }
    const uint64_t cap = uint64_t(dev.num_sms) * kEncCtasPerSm;
    const unsigned grid = unsigned(items.total_tiles < cap ? items.total_tiles : cap);
    if (g_timing.before) cudaEventRecord(g_timing.before, stream);
    enc_main<<<grid, kEncThreads, smem, stream>>>(items, ws);
    err = cudaGetLastError();
    if (g_timing.after) cudaEventRecord(g_timing.after, stream);
    if (err != cudaSuccess) return err;
  }
  {
    uint64_t per_item = items.count ? items.total_tiles / items.count : 0;
    uint64_t gx = per_item / 8;
    const uint64_t gx_cap = uint64_t(dev.num_sms) * 2;
    if (gx < 1) gx = 1;
    if (gx > gx_cap) gx = gx_cap;
    const unsigned gy = items.count < 65535u ? items.count : 65535u;
    enc_tail<<<dim3(unsigned(gx), gy), 256, 0, stream>>>(items, ws);
    err = cudaGetLastError();
  }
  return err;
}

}  // namespace sz
