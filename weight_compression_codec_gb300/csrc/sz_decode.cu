// Decode ("splitzip_codec.py" decode_torch): dense reconstruction
// x = ((sm & 0x80) << 8) | (dec_lut[code] << 7) | (sm & 0x7F), then every
// escape overwrites its element with the stored exponent -- here fused into
// one pass that writes each output byte once.
//
// Launches per call (after a 256-byte header memset):
//   dec_prepare  validates each item's meta against the wire layout and the
//                readable payload size, finds each tile's escape range
//                [k0, k1) by searching the sorted chunk_id stream (chunks
//                8*lt .. 8*lt+7 belong to tile lt), and (tables of several
//                items) writes the tile -> item map; items of up to 32 tiles
//                take one warp each;
//   dec_main     persistent CTAs own a contiguous run of tiles.  A producer
//                warp (which resolves 32 tiles at a time, one per lane)
//                streams pk, sm and the tile's chunk_id/local_pos/esc_val
//                slices into a 4-stage shared-memory ring: TMA bulk copies for
//                the 16-byte-aligned body of each slice and one zero-filling
//                16-byte cp.async for its ragged end, so nothing outside the
//                payload is read.  A tile with more than 1024 escapes takes
//                further stages carrying only its next escapes.  8 consumer
//                warps decode 8 elements per thread step with the 16-entry
//                dec_lut held in registers (byte permutes), patch the tile's
//                escapes in shared memory and hand the finished 16 KiB tile
//                to a TMA bulk store.
//
// In-place slot decode (the payload in the leading comp_bytes of the
// tensor's own 2n-byte output, "splitzip_codec.py" GpuSplitZipDecoder): the
// same prepare pass, which also copies the escape streams to a stash; then
// dip_stash copies the pk bytes of phase C there (about n / 8 bytes; the
// pages' decoder copies the whole payload), and dec_main<true> decodes each
// tensor's tiles in an order that reads everything else in place (three
// phases, see ip_phases), each tile storing once the tiles whose payload
// bytes lie under it have read them.
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kDecStages = 4;
constexpr int kDecConsumerWarps = 8;
constexpr int kDecConsumers = kDecConsumerWarps * 32;
constexpr int kDecProducerWarp = kDecConsumerWarps;
constexpr int kDecStorerWarp = kDecConsumerWarps + 1;
constexpr int kDecThreads = kDecConsumers + 64;  // + producer warp + storer warp
constexpr int kDecCtasPerSm = 2;
constexpr uint32_t kEcap = 1024;  // escapes per stage; a tile with more is sent as several stages
constexpr uint32_t kRangeInvalid = 0xFFFFFFFFu;
// kStageCont: escapes only, continuing the previous stage's tile;
// kStageMore: further escape stages of this tile follow.
constexpr uint32_t kStageEnd = 1u, kStageInvalid = 2u, kStageCont = 4u, kStageMore = 8u;

struct __align__(128) DecStage {
  uint8_t pk[kTile / 2 + 16];
  uint8_t sm[kTile + 32];
  uint32_t cid[kEcap + 8];
  uint16_t lpos[kEcap + 16];
  uint8_t ev[kEcap + 32];
  uint4 dec_lut;
  uint16_t* out;
  uint32_t m, lt, n_tile, flags;
  uint32_t sm_shift, cid_shift, lpos_shift, ev_shift;
  uint64_t tile;  // flat tile index (in-place decode: its read_done word)
  uint4 dep;      // in-place decode: tiles (local indices) [x, y] and [z, w] to wait for ...
  uint2 dep2;     // ... and [x, y]
};

// What the producer needs of one tile, resolved by one lane of the producer
// warp when a window of tiles starts (kept in shared memory, not registers,
// so the producer's loop stays light on registers).
constexpr uint32_t kWin = 16;
struct WinEntry {
  const uint8_t* base;  // payload
  uint16_t* out;        // the tile's first output element
  uint64_t off_sm, off_cid, off_lpos, off_ev;
  uint64_t pkv, escv;   // address of payload byte 0 in the pk / escape source (in place: maybe the stash)
  uint64_t tile;        // flat tile index (in place: kNoTile for a hole past a tensor's end)
  uint4 dec_lut;
  uint4 dep;            // in place: tiles to wait for (as DecStage::dep, dep2)
  uint2 dep2;
  uint32_t k0, k1, lt, nt;
  uint32_t ok;
};

// A finished output tile handed from the consumer warps to the storer warp.
struct StoreSlot {
  uint16_t* out;  // the tile's first output element
  uint64_t tile;  // flat tile index
  uint4 dep;      // in place: tiles to wait for (as DecStage::dep, dep2)
  uint2 dep2;
  uint32_t nt, lt, end;  // end: no more tiles
};

struct DecShared {
  DecStage st[kDecStages];
  alignas(128) uint16_t out[2][kTile];
  WinEntry win[kWin];
  StoreSlot sto[2];
  uint64_t full[kDecStages];
  uint64_t empty[kDecStages];
  uint64_t out_full[2];   // out[b] holds a finished tile (sto[b] describes it)
  uint64_t out_empty[2];  // the store of out[b] has read it
};

__device__ bool meta_ok(const sz_item& it, uint64_t n_esc_limit, uint64_t capacity) {
  const sz_meta* mp = it.meta;
  if (mp == nullptr || (reinterpret_cast<uintptr_t>(mp) & 15)) return false;
  const sz_meta m = *mp;
  if (m.n != it.n || m.chunk_size != kChunk || m.n_esc > m.n || m.n_esc > n_esc_limit) return false;
  const Layout l = layout_of(m.n, m.n_esc);
  return m.n_pairs == l.n_pairs && m.off_pk == 0 && m.off_sm == l.off_sm && m.off_cid == l.off_cid &&
         m.off_lpos == l.off_lpos && m.off_ev == l.off_ev && m.comp_bytes == l.comp_bytes &&
         l.comp_bytes <= capacity;
}

// Internal item flag (never in the header word): a tensor kept raw by the
// coverage gate (meta status SZ_META_GATED), skipped without an error.
constexpr uint32_t kItemGated = 0x80000000u;

// In-place decode (the payload in the leading bytes of the item's own output,
// its 2n-byte slot): payload must equal out and the payload must fit in 2n
// bytes (SZ_FLAG_META otherwise).
__device__ uint32_t item_problems(const Items& items, uint32_t i, bool inplace) {
  const sz_item& it = item_at(items, i);
  uint32_t bad = 0;
  if (it.n > SZ_MAX_ELEMS) return SZ_FLAG_SIZE;
  if (items.table) {
    const uint64_t expect = (i == 0) ? 0 : items.table[i - 1].tile_begin + tiles_of(items.table[i - 1].n);
    if (it.tile_begin != expect) bad |= SZ_FLAG_ITEMS;
    if (i + 1 == items.count && it.tile_begin + tiles_of(it.n) != items.total_tiles) bad |= SZ_FLAG_ITEMS;
  }
  const sz_meta* mp = it.meta;
  if (mp != nullptr && !(reinterpret_cast<uintptr_t>(mp) & 15) && (mp->status & SZ_META_GATED))
    return bad | kItemGated;  // nothing stored, nothing to write
  if (it.codebook == nullptr || (reinterpret_cast<uintptr_t>(it.codebook) & 15)) bad |= SZ_FLAG_ALIGN;
  if (it.n > 0 && (it.out == nullptr || (reinterpret_cast<uintptr_t>(it.out) & 15))) bad |= SZ_FLAG_ALIGN;
  if (it.n > 0 && (it.payload == nullptr || (reinterpret_cast<uintptr_t>(it.payload) & 15))) bad |= SZ_FLAG_ALIGN;
  uint64_t capacity = it.capacity;
  if (inplace) {
    if (it.n > 0 && it.payload != reinterpret_cast<const uint8_t*>(it.out)) bad |= SZ_FLAG_META;
    if (capacity > 2 * it.n) capacity = 2 * it.n;
  }
  if (!meta_ok(it, SZ_MAX_ELEMS, capacity)) bad |= SZ_FLAG_META;
  return bad;
}

// First k in [0, e) with cid[k] >= target (e if none), found by the 32 lanes
// of a warp: each round probes 32 evenly spaced positions, so the search
// takes ceil(log32(e)) + 1 dependent loads instead of log2(e).
__device__ uint32_t lower_bound_cid32(const int32_t* cid, uint32_t e, uint32_t target, uint32_t lane) {
  uint32_t lo = 0, hi = e;  // the answer lies in [lo, hi]
  while (hi - lo > 32) {
    const uint32_t step = (hi - lo + 31) / 32;
    uint32_t p = lo + (lane + 1) * step - 1;
    if (p > hi - 1) p = hi - 1;
    const uint32_t c = __popc(__ballot_sync(0xFFFFFFFFu, uint32_t(__ldg(cid + p)) < target));
    if (c == 0) {
      hi = lo + step - 1;  // the first probe already holds cid >= target
    } else {
      uint32_t last_less = lo + c * step - 1;
      if (last_less > hi - 1) last_less = hi - 1;
      if (c < 32) {
        uint32_t first_ge = lo + (c + 1) * step - 1;
        if (first_ge < hi) hi = first_ge;
      }
      lo = last_less + 1;
    }
  }
  const uint32_t p = lo + lane;
  const bool less = (p < hi) && uint32_t(__ldg(cid + p)) < target;
  return lo + __popc(__ballot_sync(0xFFFFFFFFu, less));
}

// Copies payload bytes [a, b) to dst_v + a .. dst_v + b (dst_v: the stash
// address of payload byte 0, congruent to src mod 16; b - a <= 16400) with
// one warp: each lane issues 8 16-byte loads before its stores.
__device__ __noinline__ void stash_copy_warp(uint64_t dst_v, const uint8_t* src, uint64_t a, uint64_t b, uint32_t lane) {
  const uint64_t a16 = (a + 15) & ~uint64_t(15), b16 = b & ~uint64_t(15);
  if (a16 >= b16) {
    for (uint64_t x = a + lane; x < b; x += 32) *reinterpret_cast<uint8_t*>(dst_v + x) = src[x];
    return;
  }
  if (lane < a16 - a) *reinterpret_cast<uint8_t*>(dst_v + a + lane) = src[a + lane];
  if (lane < b - b16) *reinterpret_cast<uint8_t*>(dst_v + b16 + lane) = src[b16 + lane];
  const uint4* s4 = reinterpret_cast<const uint4*>(src) + a16 / 16;
  uint4* d4 = reinterpret_cast<uint4*>(dst_v + a16);
  const uint32_t nv = uint32_t((b16 - a16) / 16);  // at most 1025
  for (uint32_t v0 = lane; v0 < nv; v0 += 8 * 32) {
    uint4 r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (v0 + 32u * j < nv) r[j] = s4[v0 + 32u * j];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (v0 + 32u * j < nv) d4[v0 + 32u * j] = r[j];
  }
}

constexpr int kPrepWarps = 8;
constexpr uint64_t kSmallTiles = 32;  // items of at most one 32-tile group are prepared by one warp
constexpr uint32_t kDenseGroup = 4096;  // escapes in a 32-tile group above which tiles are searched, not counted

// Escape ranges of the 32-tile group of item i starting at its tile ta (lane
// l <-> tile ta + l), and the group's tile -> item map entries.  A 32-ary
// warp search finds the group's first escape; then, unless the group holds
// more than kDenseGroup escapes, the warp reads the chunk_id stream from
// there, 512 entries per round, counting escapes per tile in shared memory
// until it reaches the next group, and a warp scan of the counts gives every
// tile's [k0, k1).  A denser group is not read whole: a second search finds
// its end and each lane binary-searches its own tile's first escape.  Writes
// outside the table's tiles are dropped.
__device__ void prepare_group(const Items& items, const DecWs& ws, uint32_t i, const sz_item& it, uint64_t tiles,
                              bool bad, uint64_t ta, uint32_t lane, uint32_t* counts) {
  const uint32_t ng = (tiles - ta < 32) ? uint32_t(tiles - ta) : 32u;
  uint2 r = make_uint2(kRangeInvalid, 0);
  if (!bad) {
    const uint32_t e = uint32_t(it.meta->n_esc);
    const int32_t* cid = reinterpret_cast<const int32_t*>(it.payload + it.meta->off_cid);
    const uint32_t first = uint32_t(ta) * kChunksPerTile;   // first chunk of the group
    const uint32_t limit = first + 32u * kChunksPerTile;    // first chunk of the next group
    const uint32_t k_lo = lower_bound_cid32(cid, e, first, lane);
    const bool dense = k_lo + kDenseGroup < e && uint32_t(__ldg(cid + k_lo + kDenseGroup)) < limit;
    if (dense) {
      const uint32_t k_hi = lower_bound_cid32(cid, e, limit, lane);
      const uint32_t target_l = first + lane * kChunksPerTile;
      uint32_t lo = k_lo, len = k_hi - k_lo;
      while (len > 0) {
        const uint32_t half = len >> 1;
        if (uint32_t(__ldg(cid + lo + half)) < target_l) {
          lo += half + 1;
          len -= half + 1;
        } else {
          len = half;
        }
      }
      const uint32_t next = __shfl_down_sync(0xFFFFFFFFu, lo, 1);
      r = make_uint2(lo, lane == 31 ? k_hi : next);
    } else {
      counts[lane] = 0;
      __syncwarp();
      for (uint32_t kb = k_lo; kb < e; kb += 32 * 16) {
        uint32_t c16[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const uint32_t kk = kb + lane + 32u * u;
          c16[u] = kk < e ? uint32_t(__ldg(cid + kk)) : 0xFFFFFFFFu;
        }
        bool past = false;  // this lane read a chunk_id of a later group (or the stream's end)
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const uint32_t rel = (c16[u] >> 3) - uint32_t(ta);  // tile within the group
          if (c16[u] != 0xFFFFFFFFu && rel < 32u) atomicAdd(&counts[rel], 1u);
          past |= c16[u] >= limit;
        }
        if (__any_sync(0xFFFFFFFFu, past)) break;
      }
      __syncwarp();
      const uint32_t c = counts[lane];
      uint32_t incl = c;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= uint32_t(d)) incl += o;
      }
      r = make_uint2(k_lo + incl - c, k_lo + incl);
      __syncwarp();  // counts is reused by the warp's next group
    }
  }
  const uint64_t tt = it.tile_begin + ta + lane;
  if (lane < ng && tt < items.total_tiles) {
    ws.ranges[tt] = r;
    if (ws.tile_item) ws.tile_item[tt] = i;
    if (ws.read_done) ws.read_done[tt] = 0;
  }
  if (ws.stash && !bad) {
    // in place: this group's share of the escape streams into the stash
    const sz_meta* mp = it.meta;
    const IpStash st = ip_stash(it.n, mp->n_esc, mp->off_sm, mp->off_cid, mp->comp_bytes);
    const uint64_t len = st.esc_to - st.esc_from;
    if (len) {
      const uint64_t groups = (tiles + 31) / 32;
      const uint64_t per = ((len + groups - 1) / groups + 15) & ~uint64_t(15);
      const uint64_t ea = st.esc_from + (ta / 32) * per;
      const uint64_t eb = (ea + per < st.esc_to) ? ea + per : st.esc_to;
      const uint64_t base = reinterpret_cast<uint64_t>(ws.stash) + ip_stash_at(it.tile_begin, i);
      if (ea < eb) stash_copy_warp(base + st.esc_off - st.esc_from, it.payload, ea, eb, lane);
    }
  }
}

// In-place decode: records in the header whether this item's tile count
// differs from item 0's (the schedule interleaves tensors of equal counts).
__device__ void note_tile_count(const Items& items, const DecWs& ws, const sz_item& it) {
  const uint64_t n0 = item_at(items, 0).n;
  if (it.n > SZ_MAX_ELEMS || n0 > SZ_MAX_ELEMS || tiles_of(it.n) != tiles_of(n0)) atomicOr(&ws.hdr->tiles_differ, 1u);
}

// Validation and escape ranges per item.  Rows of the grid (blockIdx.y) take
// groups of kPrepWarps consecutive items: items of at most 32 tiles are
// prepared by one warp of the row's first block, larger ones by the row's
// blocks dealt round-robin over them (warp per 32-tile group, each warp
// validating the item for itself).
__global__ void __launch_bounds__(kPrepWarps * 32) dec_prepare(const __grid_constant__ Items items, DecWs ws,
                                                                bool inplace) {
  __shared__ uint32_t counts[kPrepWarps][32];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t groups = (items.count + kPrepWarps - 1) / kPrepWarps;
  for (uint32_t grp = blockIdx.y; grp < groups; grp += gridDim.y) {
    {
      const uint32_t i = grp * kPrepWarps + warp;
      if (blockIdx.x == 0 && i < items.count) {
        const sz_item& it = item_at(items, i);
        if (it.n <= kSmallTiles * kTile) {
          uint32_t bad = 0;
          if (lane == 0) {
            bad = item_problems(items, i, inplace);
            ws.item_flags[i] = bad;
            if (bad & ~kItemGated) set_flag(ws.hdr, bad & ~kItemGated);
            if (inplace) note_tile_count(items, ws, it);
          }
          bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
          const uint64_t tiles = tiles_of(it.n);
          if (!(bad & SZ_FLAG_ITEMS) && tiles > 0) prepare_group(items, ws, i, it, tiles, bad != 0, 0, lane, counts[warp]);
        }
      }
    }
    // larger items: the row's blocks are dealt round-robin over its items,
    // blocks_per_item of them to each
    const uint32_t in_row = min(uint32_t(kPrepWarps), items.count - grp * kPrepWarps);
    const uint32_t R = min(in_row, gridDim.x);
    const uint32_t blocks_per_item = gridDim.x / R;
    const uint32_t rank = blockIdx.x / R;
    if (rank >= blocks_per_item) continue;
    for (uint32_t q = blockIdx.x % R; q < in_row; q += R) {
      const uint32_t i = grp * kPrepWarps + q;
      const sz_item& it = item_at(items, i);
      if (it.n <= kSmallTiles * kTile) continue;
      // every warp validates the item itself (no block barrier); the item's
      // first block publishes the result
      uint32_t bad = 0;
      if (lane == 0) {
        bad = item_problems(items, i, inplace);
        if (rank == 0 && warp == 0) {
          ws.item_flags[i] = bad;
          if (bad & ~kItemGated) set_flag(ws.hdr, bad & ~kItemGated);
          if (inplace) note_tile_count(items, ws, it);
        }
      }
      bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
      if (bad & SZ_FLAG_ITEMS) continue;
      const uint64_t tiles = (it.n > SZ_MAX_ELEMS) ? 0 : tiles_of(it.n);
      for (uint64_t ta = (uint64_t(rank) * kPrepWarps + warp) * 32; ta < tiles;
           ta += uint64_t(blocks_per_item) * kPrepWarps * 32)
        prepare_group(items, ws, i, it, tiles, bad != 0, ta, lane, counts[warp]);
    }
  }
}

constexpr int kStashWarps = 8;
constexpr uint64_t kStashTiles = 2;  // consecutive tiles per warp (2: 202 us, 4: 204 us, 8: 212 us per KV-cache call)

// In-place decode, before the main pass: each warp takes kStashTiles
// consecutive tiles and copies the pk bytes of those of them in phase C
// (but tile 0) into the stash; the tensor is resolved once per run of tiles
// in the same tensor.  (dec_prepare has cleared the read_done words and
// copied the escape streams.)
__global__ void __launch_bounds__(kStashWarps * 32, 4) dip_stash(const __grid_constant__ Items items, DecWs ws) {
  if (ws.hdr->flags & SZ_FLAG_ITEMS) return;
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t T = items.total_tiles;
  for (uint64_t t0 = (uint64_t(blockIdx.x) * kStashWarps + (threadIdx.x >> 5)) * kStashTiles; t0 < T;
       t0 += uint64_t(gridDim.x) * kStashWarps * kStashTiles) {
    const uint64_t t1 = (t0 + kStashTiles < T) ? t0 + kStashTiles : T;
    for (uint64_t tt = t0; tt < t1;) {
      // the run of tiles [tt, te) in one tensor
      const uint32_t idx = ws.tile_item ? ws.tile_item[tt] : 0u;
      if (idx >= items.count) {
        ++tt;
        continue;
      }
      const sz_item& it = item_at(items, idx);
      const uint64_t tb = it.tile_begin;
      const uint64_t tiles = (it.n > SZ_MAX_ELEMS) ? 0 : tiles_of(it.n);
      if (tt < tb || tt - tb >= tiles) {
        ++tt;
        continue;
      }
      const uint64_t te = (tb + tiles < t1) ? tb + tiles : t1;
      if (ws.item_flags[idx] == 0) {
        const sz_meta* mp = it.meta;
        const IpStash st = ip_stash(it.n, mp->n_esc, mp->off_sm, mp->off_cid, mp->comp_bytes);
        uint64_t pa = (tt - tb) * (kTile / 2), pb = (te - tb) * (kTile / 2);  // the run's pk bytes
        if (pa < st.pk_from) pa = st.pk_from;
        if (pb > st.pk_to) pb = st.pk_to;
        if (pa < pb) {
          const uint64_t base = reinterpret_cast<uint64_t>(ws.stash) + ip_stash_at(tb, idx);
          stash_copy_warp(base - st.pk_from, it.payload, pa, pb, lane);
        }
      }
      tt = te;
    }
  }
}

// Diagnostic (sz_check_bounded_waits): each kind of bounded wait the kernels
// use, on something that never completes -- warp 0 an mbarrier phase that
// gets one of its two arrivals, warp 1 a word polled by one thread, warp 2
// words polled by a warp.  Each gives up, sets SZ_FLAG_TIMEOUT and writes 1
// to gave_up[warp].
__global__ void __launch_bounds__(96) wait_selftest(DecWs ws, const uint32_t* never, uint32_t* gave_up);

// The read_done word lane `lane` of a warp watches for the store of flat tile
// `tile` (local index lt in its tensor): one tile of the local ranges
// [dep.x, dep.y], [dep.z, dep.w], [dep2.x, dep2.y] other than the tile
// itself (at most 4 + 3), or nullptr.
__device__ __forceinline__ const uint32_t* dep_word(const DecWs& ws, uint64_t tile, uint32_t lt, uint4 dep,
                                                    uint2 dep2, uint32_t lane) {
  const uint32_t lo[3] = {dep.x, dep.z, dep2.x}, hi[3] = {dep.y, dep.w, dep2.y};
  uint32_t k = lane;
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const uint32_t cnt = hi[r] >= lo[r] ? hi[r] - lo[r] + 1 : 0;
    if (k < cnt) {
      const uint32_t t = lo[r] + k;
      return t == lt ? nullptr : ws.read_done + (tile - lt + t);
    }
    k -= cnt;
  }
  return nullptr;
}

// One thread waits (bounded) until word p is set, with acquire ordering;
// gives up after kWaitTimeoutNs, or at once when another CTA has already given
// up (SZ_FLAG_TIMEOUT).
__device__ bool wait_word(const DecWs& ws, const uint32_t* p) {
  if (ld_acquire_u32(p)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire_u32(p)) return true;
    if ((i & 63) == 0 &&
        (global_timer_ns() - t0 > kWaitTimeoutNs || (ld_acquire_u32(&ws.hdr->flags) & SZ_FLAG_TIMEOUT)))
      return false;
  }
}

// One warp waits (bounded) until every lane's word p is set; v is a value of
// it read earlier (the load is issued when the tile's first stage lands, so
// its latency hides behind the decode, and the schedule makes the words
// usually set by then).  Relaxed loads: a word is set only after its tile's
// copies have read their bytes, and the store that follows is issued only
// after the word is seen.  Gives up after kWaitTimeoutNs, or at once when
// another CTA has already given up (SZ_FLAG_TIMEOUT).
__device__ bool wait_words_warp(const DecWs& ws, const uint32_t* p, uint32_t v, uint32_t lane) {
  bool ok = p == nullptr || v != 0;
  if (__all_sync(0xFFFFFFFFu, ok)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (!ok) ok = ld_relaxed_u32(p) != 0;
    if (__all_sync(0xFFFFFFFFu, ok)) return true;
    if ((i & 63) == 0 && __any_sync(0xFFFFFFFFu, lane == 0 && (global_timer_ns() - t0 > kWaitTimeoutNs ||
                                                              (ld_acquire_u32(&ws.hdr->flags) & SZ_FLAG_TIMEOUT))))
      return false;
  }
}

__global__ void __launch_bounds__(96) wait_selftest(DecWs ws, const uint32_t* never, uint32_t* gave_up) {
  __shared__ uint64_t bar;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 2);
    fence_mbar_init();
  }
  __syncthreads();
  bool ok;
  if (warp == 0) {
    if (lane == 0) mbar_arrive(&bar);  // one arrival of two: the phase never completes
    ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar, 0));
  } else if (warp == 1) {
    ok = true;
    if (lane == 0) ok = wait_word(ws, never);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  } else {
    ok = wait_words_warp(ws, lane < 4 ? never : nullptr, 0u, lane);
  }
  if (!ok && lane == 0) {
    set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
    gave_up[warp] = 1;
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

// In-place decode schedule.  Each tensor's tiles are decoded in its phase
// order (ip_rank: A from the top down, then B from the top down, then C
// from the bottom up), and a tile only waits for tiles earlier in that
// order.  Work is handed out in chunks of up to kIpChunk consecutive
// positions of one tensor's order.  When all K tensors have Tu tiles, chunk
// ticket q is chunk q / K of tensor q % K (rank-major: a tile d chunks
// further in its tensor's order comes d K tickets later); otherwise the
// tensors are taken from the last to the first, each in its order, and cut
// into chunks.  CTA b of the R CTAs (a cooperative launch, so all are
// resident) takes chunks b, b + R, b + 2R, ... and the positions of each
// chunk in order.  Every CTA meets its tiles in increasing (chunk ticket,
// position) order and a tile only waits for tiles earlier in that order,
// which are read before it by induction.  Chunks keep a CTA on consecutive
// tiles (measured on the 64-tensor KV cache: 203 us with single tiles, 186 us
// with chunks of 4); longer chunks leave too few chunks per CTA to balance (8:
// 192 us, 16: 200 us, 32: 231 us).  The cyclic order over chunks keeps the
// CTAs advancing together, so waits are short.
constexpr uint64_t kIpChunk = 4;
constexpr uint64_t kNoTile = ~0ull;

// chunk size, and number of chunk tickets
__device__ __forceinline__ uint64_t ip_chunk_size(uint64_t Tu) {
  return (Tu != 0 && Tu < kIpChunk) ? Tu : kIpChunk;
}
__device__ __forceinline__ uint64_t ip_chunks(uint64_t T, uint32_t K, uint64_t Tu, uint64_t C) {
  return Tu == 0 ? (T + C - 1) / C : uint64_t(K) * ((Tu + C - 1) / C);
}
// the phases of a tensor of n elements (off_sm from n alone: the meta of a
// valid item agrees with it)
__device__ __forceinline__ IpPhases ip_phases_of(uint64_t n) {
  return ip_phases(n, ((n + 1) / 2 + 3) & ~uint64_t(3));
}
// flat tile at position j of chunk ticket q, or kNoTile past a tensor's end
__device__ uint64_t ip_tile_of(const Items& items, const DecWs& ws, uint64_t q, uint64_t j, uint64_t T,
                               uint64_t Tu, uint64_t C) {
  if (Tu == 0) {
    const uint64_t d = q * C + j;
    if (d >= T) return kNoTile;
    const uint64_t p = T - 1 - d;  // the tensors from the last down, each in its own order
    const uint32_t i = ws.tile_item ? ws.tile_item[p] : 0u;
    if (i >= items.count) return p;
    const sz_item& it = item_at(items, i);
    const uint64_t tb = it.tile_begin;
    if (it.n > SZ_MAX_ELEMS || p < tb || p - tb >= tiles_of(it.n)) return p;  // not a valid tensor tile
    return tb + ip_tile_at(ip_phases_of(it.n), tb + tiles_of(it.n) - 1 - p);
  }
  const uint64_t r = q / items.count, i = q - r * items.count, d = r * C + j;
  if (d >= Tu) return kNoTile;
  const uint64_t n = item_at(items, uint32_t(i)).n;
  if (n > SZ_MAX_ELEMS || tiles_of(n) != Tu) return i * Tu + (Tu - 1 - d);
  return i * Tu + ip_tile_at(ip_phases_of(n), d);
}

// INPLACE = false: sz_decode(_many); persistent CTAs own contiguous tile
// ranges.  INPLACE = true: in-place slot decode; CTAs take tiles in the
// cyclic descending order above, read the stashed sm and escape bytes from
// the stash, mark each tile's read_done once its stage has landed and store
// a tile only after the tiles whose in-place bytes lie under its output have
// been read.
template <bool INPLACE>
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

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&sh.full[s], 1 + 32);
      mbar_init(&sh.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.out_full[b], 1);
      mbar_init(&sh.out_empty[b], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDecStorerWarp) {
    // ---------------------------------------------------------------- storer warp
    // Takes each finished output tile from the consumer warps and stores it
    // (TMA bulk store of its 16-byte body, plain stores for the ragged end);
    // in place, first waits until the tiles whose payload bytes lie under it
    // have read them.  Waiting here keeps the consumers decoding the next
    // tile into the other output buffer.
    for (uint32_t k = 0;; ++k) {
      const int b = int(k & 1u);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sh.out_full[b], (k >> 1) & 1u))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        break;
      }
      const StoreSlot so = sh.sto[b];
      if (so.end) break;
      bool go = true;
      if constexpr (INPLACE) {
        const uint32_t* p = dep_word(ws, so.tile, so.lt, so.dep, so.dep2, uint32_t(lane));
        go = wait_words_warp(ws, p, p ? ld_relaxed_u32(p) : 1u, uint32_t(lane));
        if (lane == 0) {
          if (go) {
            fence_proxy_async_global();
          } else {
            set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
          }
        }
      }
      const uint32_t body = (so.nt * 2u) & ~15u;
      if (lane == 0) {
        if (go && body) bulk_s2g(so.out, sh.out[b], body);
        bulk_commit();
      }
      if (go)
        for (uint32_t e = body / 2u + uint32_t(lane); e < so.nt; e += 32) so.out[e] = sh.out[b][e];
      if (lane == 0) bulk_wait_read<0>();  // the bulk store has read out[b]
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.out_empty[b]);
    }
    if (lane == 0) bulk_wait_all<0>();
    return;
  }

  if (warp == kDecProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    // When a window of kWin tiles starts, lane l resolves tile l of it in
    // parallel (escape range, item through the tile -> item map, payload,
    // output, dec_lut, section offsets; in place also the sm and escape
    // sources and the tiles to wait for) into sh.win[l]; then the tiles are
    // issued one by one from that table.
    uint64_t it = 0;  // stages handed out
    // next free stage of the ring (bounded wait agreed by the warp)
    auto acquire = [&](int& s) -> bool {
      s = int(it % kDecStages);
      if (it >= uint64_t(kDecStages) &&
          !__all_sync(0xFFFFFFFFu, mbar_wait(&sh.empty[s], uint32_t((it / kDecStages) - 1) & 1))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return false;
      }
      return true;
    };
    // next / t1: the CTA's range of tiles, or (in place) of its positions k
    // (k <-> position k % C of chunk ticket blockIdx.x + (k / C) R)
    uint64_t next = 0, t1 = 0;
    const uint64_t R = gridDim.x;
    uint64_t Tu = 0, C = 1;  // in place: every tensor's tile count when they are all equal; chunk size
    if constexpr (INPLACE) {
      if (ws.hdr->tiles_differ == 0 && items.count > 0 && T % items.count == 0) Tu = T / items.count;
      C = ip_chunk_size(Tu);
      const uint64_t Q = ip_chunks(T, items.count, Tu, C);
      t1 = blockIdx.x < Q ? (Q - blockIdx.x + R - 1) / R * C : 0;
    } else {
      const uint64_t per = (T + R - 1) / R;
      next = uint64_t(blockIdx.x) * per;
      t1 = (next + per < T) ? next + per : T;
    }
    uint32_t win_len = 0, win_pos = 0;
    for (;;) {
      if (win_pos == win_len) {
        const uint64_t first = next;
        win_len = next < t1 ? uint32_t((t1 - next < kWin) ? t1 - next : kWin) : 0u;
        next += win_len;
        win_pos = 0;
        if (win_len == 0) {
          int s;
          if (!acquire(s)) return;
          if (lane == 0) {
            sh.st[s].flags = kStageEnd;
            mbar_arrive(&sh.full[s]);
          }
          cp_async_mbar_arrive_noinc(&sh.full[s]);
          return;
        }
        __syncwarp();  // every lane is done with the previous window's entries
        if (uint32_t(lane) < win_len) {
          const uint64_t k = first + lane;
          const uint64_t mine =
              INPLACE ? ip_tile_of(items, ws, blockIdx.x + (k / C) * R, k % C, T, Tu, C) : k;
          WinEntry& w = sh.win[lane];
          w.tile = mine;
          uint32_t ok = 0;
          if (mine != kNoTile) {
            const uint2 rec = ws.ranges[mine];
            const uint32_t idx = ws.tile_item ? ws.tile_item[mine] : 0u;
            if (idx < items.count && rec.x != kRangeInvalid && ws.item_flags[idx] == 0) {
              const sz_item& itm = item_at(items, idx);
              const uint64_t tb = itm.tile_begin;
              if (mine >= tb && mine - tb < tiles_of(itm.n)) {
                const uint32_t lt = uint32_t(mine - tb);
                const uint64_t g = uint64_t(lt) * kTile;
                const sz_meta* mp = itm.meta;
                w.k0 = rec.x;
                w.k1 = rec.y;
                w.lt = lt;
                w.nt = (itm.n - g < kTile) ? uint32_t(itm.n - g) : kTile;
                w.base = itm.payload;
                w.out = itm.out + g;
                w.off_sm = mp->off_sm;
                w.off_cid = mp->off_cid;
                w.off_lpos = mp->off_lpos;
                w.off_ev = mp->off_ev;
                w.dec_lut = *reinterpret_cast<const uint4*>(itm.codebook->dec_lut);
                if constexpr (INPLACE) {
                  const IpStash sv = ip_stash(itm.n, mp->n_esc, w.off_sm, w.off_cid, mp->comp_bytes);
                  const IpPhases ph = ip_phases(itm.n, w.off_sm);
                  const uint64_t sb = reinterpret_cast<uint64_t>(ws.stash) + ip_stash_at(tb, idx);
                  // phase C reads its pk bytes from the stash (but tile 0, which
                  // reads its own before it stores over them)
                  w.pkv = (lt >= ph.tB && lt < ph.tA && lt > 0) ? sb - sv.pk_from
                                                               : reinterpret_cast<uint64_t>(itm.payload);
                  w.escv = sb + sv.esc_off - sv.esc_from;
                  const IpDeps d = ip_deps(itm.n, w.off_sm, lt);
                  w.dep = make_uint4(uint32_t(d.pk_lo), uint32_t(d.pk_hi), uint32_t(d.pk2_lo), uint32_t(d.pk2_hi));
                  w.dep2 = make_uint2(uint32_t(d.sm_lo), uint32_t(d.sm_hi));
                } else {
                  w.pkv = w.escv = reinterpret_cast<uint64_t>(itm.payload);
                }
                ok = 1;
              }
            }
          }
          w.ok = ok;
        }
        __syncwarp();
      }
      const WinEntry& w = sh.win[win_pos++];
      const uint64_t tile = w.tile;
      if (INPLACE && tile == kNoTile) continue;  // past the end of a tensor: no stage
      int s;
      if (!acquire(s)) return;
      if (!w.ok) {
        if (lane == 0) {
          sh.st[s].flags = kStageInvalid;
          sh.st[s].tile = tile;
          mbar_arrive(&sh.full[s]);
        }
        cp_async_mbar_arrive_noinc(&sh.full[s]);
        ++it;
        continue;
      }
      const uint32_t k0 = w.k0, k1 = w.k1, lt = w.lt, nt = w.nt;
      const uint64_t g = uint64_t(lt) * kTile;
      const uint64_t off_sm = w.off_sm, off_cid = w.off_cid, off_lpos = w.off_lpos, off_ev = w.off_ev;
      const uint8_t* base = w.base;
      const uint8_t* pk_src = reinterpret_cast<const uint8_t*>(w.pkv);    // payload byte 0 of the pk source
      const uint8_t* esc_src = reinterpret_cast<const uint8_t*>(w.escv);  // ... of the escape streams' source
      const uint32_t m = (k1 > k0) ? k1 - k0 : 0u;
      const uint32_t pieces = m ? (m + kEcap - 1) / kEcap : 1u;
      const Slice spk = slice_of(g >> 1, (nt + 1) >> 1);
      const Slice ssm = slice_of(off_sm + g, nt);
      // the tile: pk, sm and its first kEcap escapes, then one stage per
      // further kEcap escapes
      for (uint32_t pc = 0; pc < pieces; ++pc) {
        if (pc > 0 && !acquire(s)) return;
        DecStage& st = sh.st[s];
        const bool first = pc == 0;
        const uint32_t pk0 = k0 + pc * kEcap;
        const uint32_t pm = m ? ((m - pc * kEcap < kEcap) ? m - pc * kEcap : kEcap) : 0u;
        const Slice scid = slice_of(off_cid + 4ull * pk0, 4ull * pm);
        const Slice slp = slice_of(off_lpos + 2ull * pk0, 2ull * pm);
        const Slice sev = slice_of(off_ev + pk0, pm);
        const uint32_t tx = (first ? uint32_t(spk.a1 - spk.a0) + uint32_t(ssm.a1 - ssm.a0) : 0u) +
                            (pm ? uint32_t(scid.a1 - scid.a0) + uint32_t(slp.a1 - slp.a0) + uint32_t(sev.a1 - sev.a0)
                                : 0u);
        if (lane == 0) {
          st.dec_lut = w.dec_lut;
          st.out = w.out;
          st.m = pm;
          st.lt = lt;
          st.n_tile = nt;
          st.flags = (first ? 0u : kStageCont) | (pc + 1 < pieces ? kStageMore : 0u);
          st.tile = tile;
          if constexpr (INPLACE) {
            st.dep = w.dep;
            st.dep2 = w.dep2;
          }
          st.sm_shift = uint32_t(off_sm + g - ssm.a0);
          st.cid_shift = uint32_t(off_cid + 4ull * pk0 - scid.a0);
          st.lpos_shift = uint32_t(off_lpos + 2ull * pk0 - slp.a0);
          st.ev_shift = uint32_t(off_ev + pk0 - sev.a0);
          mbar_arrive_expect_tx(&sh.full[s], tx);
          if (first && spk.a1 > spk.a0) bulk_g2s(st.pk, pk_src + spk.a0, uint32_t(spk.a1 - spk.a0), &sh.full[s]);
          if (first && ssm.a1 > ssm.a0) bulk_g2s(st.sm, base + ssm.a0, uint32_t(ssm.a1 - ssm.a0), &sh.full[s]);
          if (pm && scid.a1 > scid.a0) bulk_g2s(st.cid, esc_src + scid.a0, uint32_t(scid.a1 - scid.a0), &sh.full[s]);
          if (pm && slp.a1 > slp.a0) bulk_g2s(st.lpos, esc_src + slp.a0, uint32_t(slp.a1 - slp.a0), &sh.full[s]);
          if (pm && sev.a1 > sev.a0) bulk_g2s(st.ev, esc_src + sev.a0, uint32_t(sev.a1 - sev.a0), &sh.full[s]);
        } else if (first && lane == 1 && spk.end > spk.a1) {
          cp_async16_zfill(st.pk + (spk.a1 - spk.a0), pk_src + spk.a1, uint32_t(spk.end - spk.a1));
        } else if (first && lane == 2 && ssm.end > ssm.a1) {
          cp_async16_zfill(st.sm + (ssm.a1 - ssm.a0), base + ssm.a1, uint32_t(ssm.end - ssm.a1));
        } else if (pm && lane == 3 && scid.end > scid.a1) {
          cp_async16_zfill(reinterpret_cast<uint8_t*>(st.cid) + (scid.a1 - scid.a0), esc_src + scid.a1,
                           uint32_t(scid.end - scid.a1));
        } else if (pm && lane == 4 && slp.end > slp.a1) {
          cp_async16_zfill(reinterpret_cast<uint8_t*>(st.lpos) + (slp.a1 - slp.a0), esc_src + slp.a1,
                           uint32_t(slp.end - slp.a1));
        } else if (pm && lane == 5 && sev.end > sev.a1) {
          cp_async16_zfill(st.ev + (sev.a1 - sev.a0), esc_src + sev.a1, uint32_t(sev.end - sev.a1));
        }
        cp_async_mbar_arrive_noinc(&sh.full[s]);
        ++it;
      }
    }
  }

  // ------------------------------------------------------------------ consumer warps
  uint32_t bad_escape = 0;
  uint32_t tiles_done = 0;  // tiles handed to the storer; the current tile goes to out[tiles_done & 1]
  bool in_tile = false;     // the previous stage left its tile open (more escape stages)
  // waits (bounded) until the storer has read out[tiles_done & 1]'s previous tile
  auto out_free = [&]() -> bool {
    return tiles_done < 2 || mbar_wait(&sh.out_empty[tiles_done & 1u], ((tiles_done >> 1) - 1) & 1u);
  };
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kDecStages);
    const int ob = int(tiles_done & 1u);
    bool ok = mbar_wait(&sh.full[s], (it / kDecStages) & 1);
    const DecStage& st = sh.st[s];
    // read before the vote: after it, an invalid tile's stage is released
    const uint32_t flags = ok ? st.flags : 0u;
    if constexpr (INPLACE) {
      // The tile's payload bytes are in shared memory now (or it reads
      // none): the phase completes only after the copies' reads of global
      // memory have returned, so no store issued after this flag is seen can
      // change what they read.  A relaxed store suffices (a release fence
      // here, on every tile, cost a quarter of the kernel's time).
      if (tid == 0 && ok && !(flags & (kStageCont | kStageEnd))) st_relaxed_u32(ws.read_done + st.tile, 1u);
    }
    // a tile's first stage writes out[ob]: its previous tile must have been read
    if (ok && !in_tile && !(flags & (kStageEnd | kStageInvalid))) ok = out_free();
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
    if (!(flags & kStageCont)) {
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
      // an escape's code is 0, so its decoded value already holds the right
      // sign and mantissa: the patch rewrites the exponent field only
      named_bar_sync(1, kDecConsumers);
      const uint32_t chunk0 = st.lt * kChunksPerTile;
      for (uint32_t k = uint32_t(tid); k < m; k += kDecConsumers) {
        const uint32_t c = st.cid[(st.cid_shift >> 2) + k];
        const uint32_t p = st.lpos[(st.lpos_shift >> 1) + k];
        const uint32_t ev = st.ev[st.ev_shift + k];
        const uint32_t rel = c - chunk0;
        const uint32_t pos = rel * kChunk + p;
        if (rel < kChunksPerTile && p < kChunk && pos < nt) {
          outs[pos] = uint16_t((outs[pos] & 0x807Fu) | (ev << 7));
        } else {
          bad_escape = 1;
        }
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, kDecConsumers);
    const bool more = (flags & kStageMore) != 0;
    if (tid == 0) {
      if (!more) {
        // hand the finished tile to the storer (what it needs is read from
        // the stage before the stage is released)
        StoreSlot& so = sh.sto[ob];
        so.out = st.out;
        so.tile = st.tile;
        so.lt = st.lt;
        so.nt = nt;
        if constexpr (INPLACE) {
          so.dep = st.dep;
          so.dep2 = st.dep2;
        }
        so.end = 0;
      }
      mbar_arrive(&sh.empty[s]);
      if (!more) mbar_arrive(&sh.out_full[ob]);
    }
    in_tile = more;
    if (!more) ++tiles_done;
  }
  if (bad_escape) set_flag(ws.hdr, SZ_FLAG_ESCAPE);
  // tell the storer there is nothing more (in the slot it reads next)
  if (tid == 0) {
    if (!out_free()) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
    sh.sto[tiles_done & 1u].end = 1;
    mbar_arrive(&sh.out_full[tiles_done & 1u]);
  }
}

}  // namespace

namespace {

cudaError_t launch_prepare(const Items& items, const DecWs& ws, cudaStream_t stream, bool inplace) {
  // blockIdx.y = group of kPrepWarps items; x covers the average item's
  // 32-tile groups (8 per block) times the items a row takes in turn (1 when
  // items are of one group or less: their warps need no other block)
  const uint64_t per_item = items.count ? (items.total_tiles + items.count - 1) / items.count : 0;
  const uint64_t per_row = items.count < uint32_t(kPrepWarps) ? items.count : uint64_t(kPrepWarps);
  uint64_t gx = per_item <= kSmallTiles ? 1 : (per_item + 32 * kPrepWarps - 1) / (32 * kPrepWarps) * per_row;
  if (gx < 1) gx = 1;
  if (gx > 1024) gx = 1024;
  const uint64_t groups = (uint64_t(items.count) + kPrepWarps - 1) / kPrepWarps;
  const unsigned gy = unsigned(groups < 65535u ? (groups ? groups : 1) : 65535u);
  dec_prepare<<<dim3(unsigned(gx), gy), kPrepWarps * 32, 0, stream>>>(items, ws, inplace);
  return cudaGetLastError();
}

template <bool INPLACE>
cudaError_t launch_main(const Items& items, const DecWs& ws, cudaStream_t stream, const DeviceInfo& dev) {
  static thread_local int configured_device = -1;
  static thread_local int ctas_per_sm = kDecCtasPerSm;
  const size_t smem = sizeof(DecShared);
  cudaError_t err;
  if (configured_device != dev.device) {
    err = cudaFuncSetAttribute(dec_main<INPLACE>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    int nb = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, dec_main<INPLACE>, kDecThreads, smem);
    if (err != cudaSuccess) return err;
    if (nb < 1) return cudaErrorInvalidConfiguration;
    ctas_per_sm = nb < kDecCtasPerSm ? nb : kDecCtasPerSm;
    configured_device = dev.device;
  }
  const uint64_t cap = uint64_t(dev.num_sms) * ctas_per_sm;
  const unsigned grid = unsigned(items.total_tiles < cap ? items.total_tiles : cap);
  if (g_timing.before) cudaEventRecord(g_timing.before, stream);
  if constexpr (INPLACE) {
    // tiles wait for tiles of other CTAs' runs: every CTA must be resident
    Items it = items;
    DecWs w = ws;
    void* args[] = {&it, &w};
    err = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(dec_main<true>), dim3(grid), dim3(kDecThreads),
                                      args, smem, stream);
  } else {
    dec_main<false><<<grid, kDecThreads, smem, stream>>>(items, ws);
    err = cudaGetLastError();
  }
  if (g_timing.after) cudaEventRecord(g_timing.after, stream);
  return err;
}

}  // namespace

cudaError_t launch_decode(const Items& items, void* ws_base, cudaStream_t stream, const DeviceInfo& dev) {
  const DecWs ws = dec_ws(ws_base, items.count, items.total_tiles);
  cudaError_t err = cudaMemsetAsync(ws_base, 0, sizeof(WsHeader), stream);
  if (err != cudaSuccess || (err = launch_prepare(items, ws, stream, false)) != cudaSuccess) return err;
  if (items.total_tiles == 0) return cudaSuccess;
  return launch_main<false>(items, ws, stream, dev);
}

cudaError_t launch_wait_selftest(void* ws_base, cudaStream_t stream) {
  // workspace: header | never (u32, zero) | gave_up[3] u32
  DecWs ws = dec_ws(ws_base, 1, 0);
  uint32_t* words = reinterpret_cast<uint32_t*>(static_cast<char*>(ws_base) + sizeof(WsHeader));
  cudaError_t err = cudaMemsetAsync(ws_base, 0, sizeof(WsHeader) + 16, stream);
  if (err != cudaSuccess) return err;
  wait_selftest<<<1, 96, 0, stream>>>(ws, words, words + 1);
  return cudaGetLastError();
}

cudaError_t launch_decode_inplace(const Items& items, void* ws_base, cudaStream_t stream, const DeviceInfo& dev) {
  const DecWs ws = ip_ws(ws_base, items.count, items.total_tiles);
  cudaError_t err = cudaMemsetAsync(ws_base, 0, sizeof(WsHeader), stream);
  if (err != cudaSuccess || (err = launch_prepare(items, ws, stream, true)) != cudaSuccess) return err;
  if (items.total_tiles == 0) return cudaSuccess;
  const uint64_t blocks = (items.total_tiles + kStashWarps * kStashTiles - 1) / (kStashWarps * kStashTiles);
  const uint64_t cap = uint64_t(dev.num_sms) * 32;  // four waves of 8 blocks per SM, then grid-stride
  dip_stash<<<unsigned(blocks < cap ? blocks : cap), kStashWarps * 32, 0, stream>>>(items, ws);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return launch_main<true>(items, ws, stream, dev);
}

}  // namespace sz
