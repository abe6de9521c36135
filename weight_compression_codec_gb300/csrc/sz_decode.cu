// Decode ("splitzip_codec.py" decode_torch): dense reconstruction
// x = ((sm & 0x80) << 8) | (dec_lut[code] << 7) | (sm & 0x7F), then every
// escape overwrites its element with the stored exponent -- here fused into
// one pass that writes each output byte once.
//
// Out of place, one kernel per call (after a 256-byte header memset):
//   dec_main     persistent CTAs own a contiguous run of tiles.  A producer
//                warp resolves 16 tiles at a time, one per lane: the tensor
//                (a 32-entry window of the item table in the lanes), its
//                meta checked against the wire layout and the readable
//                payload size, and the tile's escape range [k0, k1) in the
//                tensor's sorted chunk_id stream (chunks 8*lt .. 8*lt+7
//                belong to tile lt).  Ranges continue from the previous
//                window's end: a counting pass over the next chunk_id entries
//                gives them when escapes are sparse, per-lane 17-ary searches
//                otherwise.  It then streams pk, sm and the tile's
//                chunk_id/local_pos/esc_val slices into a 4-stage
//                shared-memory ring: TMA bulk copies for the 16-byte-aligned
//                body of each slice and one zero-filling 16-byte cp.async for
//                its ragged end, so nothing outside the payload is read.  A
//                tile with more than 1024 escapes takes further stages
//                carrying only its next escapes.  8 consumer warps decode 8
//                elements per thread step with the 16-entry dec_lut held in
//                registers (byte permutes), patch the tile's escapes in
//                shared memory and hand the finished 16 KiB tile to a storer
//                warp, which issues its TMA bulk store.
//
// In-place slot decode (the payload in the leading comp_bytes of the
// tensor's own 2n-byte output, "splitzip_codec.py" GpuSplitZipDecoder):
//   dec_prepare  validates each item's meta, finds each tile's escape range
//                by searching the chunk_id stream, writes the tile -> item
//                map, clears the read_done words and copies the escape
//                streams to a stash;
//   dip_stash    copies the pk bytes of phase C there (about n / 8 bytes; the
//                pages' decoder copies the whole payload);
//   dec_main<true> decodes each tensor's tiles in an order that reads
//                everything else in place (three phases, see ip_phases), each
//                tile storing once the tiles whose payload bytes lie under it
//                have read them.
#include <cstddef>

#include "sz_count.cuh"
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kDecStages = 4;
constexpr int kDecConsumerWarps = 8;
constexpr int kDecConsumers = kDecConsumerWarps * 32;
constexpr uint32_t kEcap = 1024;  // escapes in a tile's first stage; a tile with more is sent as several stages
constexpr uint32_t kRangeInvalid = 0xFFFFFFFFu;
// kStageCont: escapes only, continuing the previous stage's tile;
// kStageMore: further escape stages of this tile follow.
constexpr uint32_t kStageEnd = 1u, kStageInvalid = 2u, kStageCont = 4u, kStageMore = 8u;

// In-place decode (dec_inplace): two CTAs per SM, each one pipeline (8
// consumer warps, a producer warp, a storer warp).
constexpr int kIpProducerWarp = kDecConsumerWarps;
constexpr int kIpStorerWarp = kDecConsumerWarps + 1;
constexpr int kIpThreads = kDecConsumers + 64;
constexpr int kIpCtasPerSm = 2;

// Out-of-place decode (dec_flat): one CTA per SM with two pipelines (8
// consumer warps and a producer warp each) fed by one resolver warp.  The two
// pipelines take windows of tiles as they become free, so they finish
// together; two CTAs per SM, each with a fixed share of the tiles, did not
// (the SM's scheduler favours one of them, which finished 20 % earlier).
constexpr int kPipes = 2;
constexpr int kFlatProducerWarp = kPipes * kDecConsumerWarps;  // producers: warps 16, 17
constexpr int kFlatResolverWarp = kFlatProducerWarp + kPipes;  // 18
constexpr int kFlatThreads = (kFlatResolverWarp + 1) * 32;
constexpr uint32_t kPool = 3;  // window tables between the resolver and the producers

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

// A tile's further stages carry escapes only: their chunk_id, local_pos and
// esc_val slices fill the whole stage from pk on (kEcapCont of them, each
// array with 32 bytes of slack for the aligned copy and its ragged end), so a
// tile of 6,400 escapes takes three stages instead of seven.
constexpr uint32_t kEcapCont = 2688;
constexpr uint32_t kContLpos = (4u * kEcapCont + 32u + 15u) & ~15u;               // byte offset of local_pos
constexpr uint32_t kContEv = (kContLpos + 2u * kEcapCont + 32u + 15u) & ~15u;     // byte offset of esc_val
static_assert(offsetof(DecStage, pk) == 0, "continuation arrays start at the stage");
static_assert(kContEv + kEcapCont + 32u <= offsetof(DecStage, ev) + sizeof(DecStage::ev),
              "continuation arrays fit in pk .. ev");

// What the producer needs of one tile, resolved by one lane when a window of
// tiles starts (kept in shared memory, not registers, so the producer's loop
// stays light on registers).  In place the producer's lanes resolve windows
// of kWin tiles (WinEntry); out of place the resolver warp fills tables of
// up to kFlatWin compact WinOut ahead of the producers.
constexpr uint32_t kWin = 16;
constexpr uint32_t kFlatWin = 32;
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
struct WinOut {
  const uint8_t* base;  // payload
  uint16_t* out;        // the tile's first output element
  uint64_t off_sm, off_cid;
  uint4 dec_lut;
  uint64_t tile;        // flat tile index
  uint32_t k0, k1, lt, nt;
  uint32_t n_esc, ok;
};
static_assert(sizeof(WinOut) == 80, "compact window entry");

// A finished output tile handed from the consumer warps to the storer warp.
struct StoreSlot {
  uint16_t* out;  // the tile's first output element
  uint64_t tile;  // flat tile index
  uint4 dep;      // in place: tiles to wait for (as DecStage::dep, dep2)
  uint2 dep2;
  uint32_t nt, lt, end;  // end: no more tiles
};

struct IpShared {
  DecStage st[kDecStages];
  alignas(128) uint16_t out[2][kTile];
  WinEntry win[kWin];
  StoreSlot sto[2];
  uint64_t full[kDecStages];
  uint64_t empty[kDecStages];
  uint64_t out_full[2];   // out[b] holds a finished tile (sto[b] describes it)
  uint64_t out_empty[2];  // the store of out[b] has read it
};

// What the resolver keeps of the tensor of the last tile it resolved, so
// that a window that continues it needs no table, meta or codebook loads.
struct ItemCache {
  const uint8_t* payload;
  uint16_t* out;  // the tensor's first output element
  uint64_t n, off_sm, off_cid, tile_begin;
  uint4 dec_lut;
  uint32_t e, tiles;
};

struct FlatShared {
  DecStage st[kPipes][kDecStages];
  alignas(128) uint16_t out[kPipes][2][kTile];
  WinOut win[kPool][kFlatWin];
  uint32_t win_len[kPool];  // tiles in win[q]
  uint32_t issued[kPool];   // tiles of win[q] issued so far
  uint32_t next_tile;       // tiles of the CTA claimed by the producers
  ItemCache cache;          // the resolver's
  uint64_t full[kPipes][kDecStages];
  uint64_t empty[kPipes][kDecStages];
  uint64_t win_full[kPool];   // the resolver has filled win[q]
  uint64_t win_empty[kPool];  // a producer has issued every tile of win[q]
};
static_assert(sizeof(FlatShared) <= 227 * 1024, "one CTA per SM");

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
  if (it.tile_begin + tiles_of(it.n) > items.total_tiles) bad |= SZ_FLAG_ITEMS;
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
  pdl_trigger();
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

// ------------------------------------------------------------------ escape ranges inside the decode kernel

// First k in [lo, hi] with cid[k] >= target, where every k < lo holds
// cid[k] < target and hi is the stream's end or holds cid[hi] >= target.
// Each round the lane probes 16 evenly spaced positions at once (independent
// loads), so the search costs about log17(hi - lo) memory latencies.  The
// result stays in [lo, hi] whatever the stream holds.
__device__ uint32_t lower_bound_lane(const int32_t* cid, uint32_t lo, uint32_t hi, uint32_t target) {
  while (hi - lo > 16u) {
    const uint32_t step = (hi - lo + 16u) / 17u;
    uint32_t c = 0;
#pragma unroll
    for (uint32_t j = 1; j <= 16; ++j) {
      const uint64_t p = uint64_t(lo) + uint64_t(step) * j - 1u;
      if (p < hi && uint32_t(__ldg(cid + p)) < target) ++c;
    }
    const uint64_t first_ge = uint64_t(lo) + uint64_t(step) * (c + 1u) - 1u;  // probe c + 1, if it exists
    lo += step * c;
    if (c < 16u && first_ge < hi) hi = uint32_t(first_ge);
  }
  uint32_t c = 0;
#pragma unroll
  for (uint32_t j = 0; j < 16; ++j)
    if (uint64_t(lo) + j < hi && uint32_t(__ldg(cid + lo + j)) < target) ++c;
  return lo + c;
}

// One guided round, then lower_bound_lane: the first 16 probes are spaced
// `step` apart around `guess` (clipped to [lo, hi)), so a good guess leaves a
// bracket of `step` after one memory latency; a bad one costs that round.
__device__ uint32_t lower_bound_guess(const int32_t* cid, uint32_t lo, uint32_t hi, uint32_t target,
                                      uint64_t guess, uint32_t step) {
  if (hi - lo > 64u) {
    const int64_t p0 = int64_t(guess) - 8 * int64_t(step);
    uint32_t c = 0, first_ge = hi;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      int64_t p = p0 + int64_t(j) * step;
      p = p < int64_t(lo) ? int64_t(lo) : (p > int64_t(hi) - 1 ? int64_t(hi) - 1 : p);
      const bool less = uint32_t(__ldg(cid + p)) < target;
      c += less ? 1u : 0u;
      if (!less && uint32_t(p) < first_ge) first_ge = uint32_t(p);
    }
    // probes are non-decreasing: the c that are less come first
    if (c > 0) {
      int64_t pl = p0 + int64_t(c - 1) * step;
      pl = pl < int64_t(lo) ? int64_t(lo) : (pl > int64_t(hi) - 1 ? int64_t(hi) - 1 : pl);
      lo = uint32_t(pl) + 1u;
    }
    if (first_ge < hi && first_ge >= lo) hi = first_ge;
    if (lo > hi) lo = hi;
  }
  return lower_bound_lane(cid, lo, hi, target);
}

// Probe spacing of a guided search whose guess stands `dist` escapes from a
// known end of the bracket: escape counts of like tiles vary by about their
// square root, so 16 probes this far apart cover several deviations.
__device__ __forceinline__ uint32_t guess_step(uint64_t dist) {
  const uint32_t s = uint32_t(sqrtf(float(dist))) + 1u;
  return s < 4u ? 4u : s;
}

// The tile after the last one the resolver resolved: its tensor, its local
// index and its first escape (item == kNoItem: not known), and the escapes
// per tile of the last window (the guess for the next one).
constexpr uint32_t kNoItem = 0xFFFFFFFFu;
struct RangeCarry {
  uint32_t item, lt, k;
  float rho;
};

constexpr uint32_t kCountEntries = 1024;  // chunk_ids a sparse window's ends are searched among (32 per lane)

// The end of this lane's tile (the first k >= k_start with cid[k] >= target)
// when it lies among the kCountEntries entries from k_start: the warp first
// asks L1 for their lines (one 128-byte line per lane), then each lane
// binary-searches them, so the pass costs one memory latency and a few L1
// hits.  *exact is false when every entry read is below the target (and the
// stream goes on): the end lies further.
__device__ uint32_t bound_window(const int32_t* cid, uint32_t e, uint32_t k_start, uint32_t target, bool active,
                                 uint32_t lane, bool* exact) {
  const uint32_t k_end = (uint64_t(k_start) + kCountEntries < e) ? k_start + kCountEntries : e;
  if (uint64_t(k_start) + 32u * lane < k_end)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(cid + k_start + 32u * lane) : "memory");
  uint32_t lo = k_start, len = active ? k_end - k_start : 0u;
  while (len > 0) {
    const uint32_t half = len >> 1;
    if (uint32_t(__ldg(cid + lo + half)) < target) {
      lo += half + 1u;
      len -= half + 1u;
    } else {
      len = half;
    }
  }
  *exact = lo < k_end || k_end == e;
  return lo;
}

// Asks L2 for the chunk_ids the next window will count or probe (about
// `expect` of them from escape k, at least kCountEntries), one window ahead:
// whole 16-byte lines inside the stream.  The producers read these lines a
// window later, after more than L2 holds has streamed through it, so every
// prefetched line is read from DRAM twice; a window of more than
// kPrefetchMax escapes is not prefetched: its lanes' guided searches touch a
// few sectors each, and the lanes whose ends lie past a capped prefetch
// would wait on DRAM all the same.
constexpr uint32_t kPrefetchMax = 8192;
__device__ __forceinline__ void prefetch_count(const uint8_t* payload, uint64_t off_cid, uint32_t e, uint32_t k,
                                               uint32_t expect, uint32_t lane) {
  if (lane != 0 || k >= e || expect > kPrefetchMax) return;
  uint64_t cnt = expect < kCountEntries ? kCountEntries : expect;
  if (uint64_t(k) + cnt > e) cnt = e - k;
  const uint64_t a = (reinterpret_cast<uint64_t>(payload) + off_cid + 4ull * k) & ~uint64_t(15);
  const uint64_t b = (reinterpret_cast<uint64_t>(payload) + off_cid + 4ull * (k + cnt)) & ~uint64_t(15);
  if (b > a)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(uint32_t(b - a)) : "memory");
}

// Tensors dec_small decodes whole (their item checks passed): at most two
// tiles, and a payload that fits one of its buffers.
constexpr uint32_t kSdPay = 26624;  // payload bytes a dec_small buffer holds
__device__ __forceinline__ bool small_fits(const sz_item& it) {
  return it.n <= kSmallMax && it.meta->comp_bytes <= kSdPay;
}

// Out-of-place decode, resolver warp: lane l < len resolves tile first + l
// into win[l]; all 32 lanes take part.
//  * A window that continues the tensor of the last one (carry) takes the
//    tensor from `cache` and its first escape from carry.k; when the window
//    holds fewer than kCountEntries escapes, every tile's end is found among
//    those entries (bound_window: one L1 fill, then binary searches in L1).
//  * Otherwise each lane finds its tensor (a 32-entry window of the item
//    table from item `cur`), checks it (item_problems) and searches for its
//    tile's end (lower_bound_guess: at most 8192 escapes per tile bracket it,
//    the tensor's mean escape density gives the first guess).
//  * Windows denser than one counting pass search past what was read.
// A window's first tile either starts its tensor or follows the last
// resolved tile (prime_carry gives the carry of a CTA's first tile).
// Flags found are raised in the header; a tile of a bad or gated tensor gets
// ok = 0.
__device__ void resolve_window(const Items& items, const DecWs& ws, WinOut* win, uint64_t first, uint32_t len,
                               uint32_t lane, uint32_t& cur, RangeCarry& carry, ItemCache& cache) {
  constexpr unsigned kAll = 0xFFFFFFFFu;
  const bool act = lane < len;
  const uint64_t mine = first + (act ? lane : len - 1u);
  const bool cont = carry.item != kNoItem && first == cache.tile_begin + carry.lt &&
                    first + len <= cache.tile_begin + cache.tiles;
  uint32_t idx = carry.item, lt = 0, e = 0, tiles = 0, bad = 0;
  bool ok = act;
  const int32_t* cid = nullptr;
  const uint8_t* payload = nullptr;
  uint16_t* out0 = nullptr;
  uint64_t n = 0, off_sm = 0, off_cid = 0;
  uint4 dl = make_uint4(0, 0, 0, 0);
  if (cont) {
    lt = carry.lt + (act ? lane : 0u);
    e = cache.e;
    tiles = cache.tiles;
    payload = cache.payload;
    out0 = cache.out;
    n = cache.n;
    off_sm = cache.off_sm;
    off_cid = cache.off_cid;
    dl = cache.dec_lut;
    cid = reinterpret_cast<const int32_t*>(payload + off_cid);
  } else {
    idx = 0;
    if (items.table) {
      // lane j holds the first tile of item cur + j; the tile's item is the
      // last of them that starts at or before it
      const uint64_t tbj = (uint64_t(cur) + lane < items.count) ? items.table[cur + lane].tile_begin : ~0ull;
      uint32_t pos = 0;
#pragma unroll
      for (uint32_t st = 16; st > 0; st >>= 1) {
        const uint64_t v = __shfl_sync(kAll, tbj, int(pos + st - 1u));
        if (v <= mine) pos += st;
      }
      const uint64_t t31 = __shfl_sync(kAll, tbj, 31);
      if (pos == 31u && t31 <= mine) pos = 32u;
      if (pos == 32u && uint64_t(cur) + 32u < items.count) {
        idx = find_item(items, mine);  // more than 31 items start in the window (empty items)
      } else {
        idx = cur + (pos ? pos - 1u : 0u);
      }
    }
    const sz_item& it = item_at(items, idx);
    if (act) {
      // the codebook's dec_lut is loaded with the meta, not after the checks
      const sz_codebook* cb = it.codebook;
      if (cb != nullptr && !(reinterpret_cast<uintptr_t>(cb) & 15)) dl = *reinterpret_cast<const uint4*>(cb->dec_lut);
      bad = item_problems(items, idx, false);
      if (!(bad & SZ_FLAG_SIZE) && (mine < it.tile_begin || mine - it.tile_begin >= tiles_of(it.n))) bad |= SZ_FLAG_ITEMS;
    }
    ok = act && bad == 0;
    if (ok && ws.small_done && small_fits(it)) ok = false;  // dec_small decoded it
    if (ok) {
      const sz_meta* mp = it.meta;
      lt = uint32_t(mine - it.tile_begin);
      tiles = uint32_t(tiles_of(it.n));
      e = uint32_t(mp->n_esc);
      n = it.n;
      payload = it.payload;
      out0 = it.out;
      off_sm = mp->off_sm;
      off_cid = mp->off_cid;
      cid = reinterpret_cast<const int32_t*>(payload + off_cid);
    }
  }
  // lane 0's tensor, and whether the window continues the previous one
  const uint32_t idx0 = __shfl_sync(kAll, idx, 0);
  const uint32_t lt0 = __shfl_sync(kAll, lt, 0);
  const uint32_t e0 = __shfl_sync(kAll, e, 0);
  const uint32_t tiles0 = __shfl_sync(kAll, tiles, 0);
  const int32_t* cid0 = reinterpret_cast<const int32_t*>(
      __shfl_sync(kAll, reinterpret_cast<unsigned long long>(cid), 0));
  const bool ok0 = __shfl_sync(kAll, ok, 0);
  const bool k0_known = ok0 && (lt0 == 0 || (carry.item == idx0 && carry.lt == lt0));
  const uint32_t k_start = lt0 == 0 ? 0u : carry.k;  // first escape of tile lt0 when k0_known
  const uint32_t act_mask = len >= 32u ? kAll : ((1u << len) - 1u);
  const bool one_item = cont || __ballot_sync(kAll, ok && idx == idx0) == act_mask;
  const bool need_end = ok && lt + 1u < tiles;  // the last tile of a tensor ends at e
  uint32_t B = e;  // end of this lane's escape range
  uint64_t s_lo = 0, s_hi = 0, s_guess = 0;  // this lane's search bracket and first guess (search: it searches)
  uint32_t s_target = 8u * (lt + 1u);
  const int32_t* s_cid = cid;
  bool search = false;
  if (one_item && k0_known) {
    // expected escapes per tile: the last window's, or the tensor's mean
    const float rho = cont ? carry.rho : float(e0) / float(tiles0 ? tiles0 : 1u);
    if (rho * float(len) <= 0.75f * float(kCountEntries)) {
      bool exact = true;
      const uint32_t t = bound_window(cid0, e0, k_start, 8u * (lt + 1u), need_end, lane, &exact);
      // lanes below `n_exact` found their end among the entries read (the ends are monotone)
      const uint32_t n_exact = __popc(__ballot_sync(kAll, act && exact));
      if (need_end) {
        if (exact) {
          B = t;
        } else {
          // denser than expected: search past what was read, at the density read
          search = true;
          const float r = fmaxf(rho, float(kCountEntries) / float(n_exact + 1u));
          s_lo = uint64_t(k_start) + kCountEntries;
          s_hi = uint64_t(k_start) + kTile * uint64_t(lane + 1u);
          s_guess = uint64_t(k_start) + uint64_t(r * float(lane + 1u));
        }
      }
    } else if (need_end) {
      // dense: every end by a search guided by the density
      search = true;
      s_lo = k_start;
      s_hi = uint64_t(k_start) + kTile * uint64_t(lane + 1u);
      s_guess = uint64_t(k_start) + uint64_t(rho * float(lane + 1u));
    }
  } else if (need_end) {
    // at most 8192 escapes per tile bracket the end of tile lt
    search = true;
    const uint64_t after = uint64_t(kTile) * (tiles - lt - 1u);  // escapes the later tiles can hold
    s_lo = e > after ? e - after : 0;
    s_hi = uint64_t(kTile) * (lt + 1u);
    if (idx == idx0 && k0_known) {
      if (s_lo < k_start) s_lo = k_start;
      const uint64_t cap = uint64_t(k_start) + kTile * uint64_t(lane + 1u);
      if (s_hi > cap) s_hi = cap;
    }
    s_guess = uint64_t(e) * (lt + 1u) / tiles;  // the tensor's mean density
  }
  if (s_hi > e) s_hi = e;
  if (s_lo > s_hi) s_lo = s_hi;
  if (s_guess < s_lo) s_guess = s_lo;
  if (s_guess > s_hi) s_guess = s_hi;
  const uint32_t found =
      search ? lower_bound_guess(s_cid, uint32_t(s_lo), uint32_t(s_hi), s_target, s_guess, guess_step(s_guess - s_lo))
             : 0u;
  if (search) B = found;
  // each tile's first escape: the end of the tile before it in the same tensor
  const uint32_t prev_end = __shfl_up_sync(kAll, B, 1);
  const uint32_t prev_idx = __shfl_up_sync(kAll, idx, 1);
  const bool prev_ok = __shfl_up_sync(kAll, ok, 1);
  uint32_t k0 = 0, late = 0;
  if (ok) {
    if (lane == 0) {
      k0 = k_start;
      if (!k0_known) {
        ok = false;  // starts inside a tensor it does not continue: tiles of the table not consecutive
        late |= SZ_FLAG_ITEMS;
      }
    } else if (prev_ok && prev_idx == idx) {
      k0 = prev_end;
    } else if (lt != 0) {
      ok = false;  // a tile that neither starts its tensor nor follows the previous tile of it
      late |= SZ_FLAG_ITEMS;
    }
    if (ok && B < k0) {
      B = k0;  // chunk_id not sorted
      late |= SZ_FLAG_ESCAPE;
    }
  }
  const uint32_t err = __reduce_or_sync(kAll, (bad & ~kItemGated) | late);
  if (lane == 0 && err) set_flag(ws.hdr, err);
  if (act) {
    WinOut& w = win[lane];
    w.tile = mine;
    w.ok = ok;
    if (ok) {
      const uint64_t g = uint64_t(lt) * kTile;
      w.k0 = k0;
      w.k1 = B;
      w.lt = lt;
      w.nt = (n - g < kTile) ? uint32_t(n - g) : kTile;
      w.base = payload;
      w.out = out0 + g;
      w.off_sm = off_sm;
      w.off_cid = off_cid;
      w.n_esc = e;
      w.dec_lut = dl;
    }
  }
  // the last tile's tensor is kept for the next window, whose count is prefetched
  const uint32_t last = len - 1u;
  const bool ok_last = __shfl_sync(kAll, ok, int(last));
  const uint32_t idx_last = __shfl_sync(kAll, idx, int(last));
  const uint32_t lt_last = __shfl_sync(kAll, lt, int(last));
  const uint32_t k_last = __shfl_sync(kAll, B, int(last));
  if (!cont && ok_last) {
    const int src = int(last);
    cache.payload = reinterpret_cast<const uint8_t*>(
        __shfl_sync(kAll, reinterpret_cast<unsigned long long>(payload), src));
    cache.out = reinterpret_cast<uint16_t*>(__shfl_sync(kAll, reinterpret_cast<unsigned long long>(out0), src));
    cache.n = __shfl_sync(kAll, n, src);
    cache.off_sm = __shfl_sync(kAll, off_sm, src);
    cache.off_cid = __shfl_sync(kAll, off_cid, src);
    cache.tile_begin = mine - lt;  // (lane `last`'s values, as every lane computes them from its own)
    cache.tile_begin = __shfl_sync(kAll, cache.tile_begin, src);
    cache.dec_lut.x = __shfl_sync(kAll, dl.x, src);
    cache.dec_lut.y = __shfl_sync(kAll, dl.y, src);
    cache.dec_lut.z = __shfl_sync(kAll, dl.z, src);
    cache.dec_lut.w = __shfl_sync(kAll, dl.w, src);
    cache.e = __shfl_sync(kAll, e, src);
    cache.tiles = __shfl_sync(kAll, tiles, src);
  }
  // density of this window's tensor of its last tile (one-tensor windows: as measured)
  const uint32_t k_first = __shfl_sync(kAll, k0, 0);
  carry.rho = one_item && k0_known ? float(k_last - k_first) / float(len)
                                   : float(cache.e) / float(cache.tiles ? cache.tiles : 1u);
  carry.item = ok_last ? idx_last : kNoItem;
  carry.lt = lt_last + 1u;
  carry.k = k_last;
  if (!cont) cur = idx_last;
  if (ok_last && carry.lt < cache.tiles)
    prefetch_count(cache.payload, cache.off_cid, cache.e, carry.k, uint32_t(carry.rho * float(kFlatWin)) + 64u, lane);
}

constexpr int kStashWarps = 8;
constexpr uint64_t kStashTiles = 2;  // consecutive tiles per warp (2: 202 us, 4: 204 us, 8: 212 us per KV-cache call)

// In-place decode, before the main pass: each warp takes kStashTiles
// consecutive tiles and copies the pk bytes of those of them in phase C
// (but tile 0) into the stash; the tensor is resolved once per run of tiles
// in the same tensor.  (dec_prepare has cleared the read_done words and
// copied the escape streams.)
__global__ void __launch_bounds__(kStashWarps * 32, 4) dip_stash(const __grid_constant__ Items items, DecWs ws) {
  pdl_wait();  // dec_prepare's writes
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

// One tile as a producer issues it.
struct TileSrc {
  const uint8_t* base;     // payload (the sm bytes are read from it)
  const uint8_t* pk_src;   // address of payload byte 0 in the pk source
  const uint8_t* esc_src;  // ... in the escape streams' source
  uint16_t* out;           // the tile's first output element
  uint64_t off_sm, off_cid, off_lpos, off_ev, tile;
  uint4 dec_lut, dep;
  uint2 dep2;
  uint32_t k0, k1, lt, nt;
};

// A ring of kDecStages stages between one producer warp and its consumers.
struct Ring {
  DecStage* st;
  uint64_t* full;   // a stage's bytes have landed (1 + 32 arrivals + transaction bytes)
  uint64_t* empty;  // the consumers have released it
};

// Next free stage of the ring (bounded wait agreed by the warp); `it`
// counts the stages handed out.
__device__ __forceinline__ bool acquire_stage(const Ring& r, uint64_t it, int& s, WsHeader* hdr, uint32_t lane) {
  s = int(it % kDecStages);
  if (it >= uint64_t(kDecStages) &&
      !__all_sync(0xFFFFFFFFu, mbar_wait(&r.empty[s], uint32_t((it / kDecStages) - 1) & 1))) {
    if (lane == 0) set_flag(hdr, SZ_FLAG_TIMEOUT);
    return false;
  }
  return true;
}

// A stage that carries no bytes: kStageEnd or kStageInvalid (with the tile).
__device__ bool issue_marker(const Ring& r, uint64_t& it, uint32_t flags, uint64_t tile, WsHeader* hdr,
                             uint32_t lane) {
  int s;
  if (!acquire_stage(r, it, s, hdr, lane)) return false;
  if (lane == 0) {
    r.st[s].flags = flags;
    r.st[s].tile = tile;
    mbar_arrive(&r.full[s]);
  }
  cp_async_mbar_arrive_noinc(&r.full[s]);
  ++it;
  return true;
}

// The stages of one tile: pk, sm and its first kEcap escapes, then one stage
// per further kEcapCont escapes (laid out from pk on).  Each slice's 16-byte-aligned body goes by TMA
// (lane 0), its ragged end by a zero-filling cp.async (lanes 1-5), so nothing
// outside the payload is read.
template <bool INPLACE>
__device__ bool issue_tile(const Ring& r, uint64_t& it, const TileSrc& t, WsHeader* hdr, uint32_t lane) {
  const uint32_t m = (t.k1 > t.k0) ? t.k1 - t.k0 : 0u;
  const uint32_t pieces = m > kEcap ? 1u + (m - kEcap + kEcapCont - 1u) / kEcapCont : 1u;
  const uint64_t g = uint64_t(t.lt) * kTile;
  const Slice spk = slice_of(g >> 1, (t.nt + 1) >> 1);
  const Slice ssm = slice_of(t.off_sm + g, t.nt);
  for (uint32_t pc = 0; pc < pieces; ++pc) {
    int s;
    if (!acquire_stage(r, it, s, hdr, lane)) return false;
    DecStage& st = r.st[s];
    uint64_t* const full = &r.full[s];
    const bool first = pc == 0;
    const uint32_t before = first ? 0u : kEcap + (pc - 1u) * kEcapCont;  // escapes of the tile in earlier stages
    const uint32_t cap = first ? kEcap : kEcapCont;
    const uint32_t pk0 = t.k0 + before;
    const uint32_t pm = m > before ? ((m - before < cap) ? m - before : cap) : 0u;
    uint8_t* const dcid = first ? reinterpret_cast<uint8_t*>(st.cid) : st.pk;
    uint8_t* const dlpos = first ? reinterpret_cast<uint8_t*>(st.lpos) : st.pk + kContLpos;
    uint8_t* const dev = first ? st.ev : st.pk + kContEv;
    const Slice scid = slice_of(t.off_cid + 4ull * pk0, 4ull * pm);
    const Slice slp = slice_of(t.off_lpos + 2ull * pk0, 2ull * pm);
    const Slice sev = slice_of(t.off_ev + pk0, pm);
    const uint32_t tx = (first ? uint32_t(spk.a1 - spk.a0) + uint32_t(ssm.a1 - ssm.a0) : 0u) +
                        (pm ? uint32_t(scid.a1 - scid.a0) + uint32_t(slp.a1 - slp.a0) + uint32_t(sev.a1 - sev.a0)
                            : 0u);
    if (lane == 0) {
      st.dec_lut = t.dec_lut;
      st.out = t.out;
      st.m = pm;
      st.lt = t.lt;
      st.n_tile = t.nt;
      st.flags = (first ? 0u : kStageCont) | (pc + 1 < pieces ? kStageMore : 0u);
      st.tile = t.tile;
      if constexpr (INPLACE) {
        st.dep = t.dep;
        st.dep2 = t.dep2;
      }
      st.sm_shift = uint32_t(t.off_sm + g - ssm.a0);
      st.cid_shift = uint32_t(t.off_cid + 4ull * pk0 - scid.a0);
      st.lpos_shift = uint32_t(t.off_lpos + 2ull * pk0 - slp.a0);
      st.ev_shift = uint32_t(t.off_ev + pk0 - sev.a0);
      mbar_arrive_expect_tx(full, tx);
      if (first && spk.a1 > spk.a0) bulk_g2s(st.pk, t.pk_src + spk.a0, uint32_t(spk.a1 - spk.a0), full);
      if (first && ssm.a1 > ssm.a0) bulk_g2s(st.sm, t.base + ssm.a0, uint32_t(ssm.a1 - ssm.a0), full);
      if (pm && scid.a1 > scid.a0) bulk_g2s(dcid, t.esc_src + scid.a0, uint32_t(scid.a1 - scid.a0), full);
      if (pm && slp.a1 > slp.a0) bulk_g2s(dlpos, t.esc_src + slp.a0, uint32_t(slp.a1 - slp.a0), full);
      if (pm && sev.a1 > sev.a0) bulk_g2s(dev, t.esc_src + sev.a0, uint32_t(sev.a1 - sev.a0), full);
    } else if (first && lane == 1 && spk.end > spk.a1) {
      cp_async16_zfill(st.pk + (spk.a1 - spk.a0), t.pk_src + spk.a1, uint32_t(spk.end - spk.a1));
    } else if (first && lane == 2 && ssm.end > ssm.a1) {
      cp_async16_zfill(st.sm + (ssm.a1 - ssm.a0), t.base + ssm.a1, uint32_t(ssm.end - ssm.a1));
    } else if (pm && lane == 3 && scid.end > scid.a1) {
      cp_async16_zfill(dcid + (scid.a1 - scid.a0), t.esc_src + scid.a1, uint32_t(scid.end - scid.a1));
    } else if (pm && lane == 4 && slp.end > slp.a1) {
      cp_async16_zfill(dlpos + (slp.a1 - slp.a0), t.esc_src + slp.a1, uint32_t(slp.end - slp.a1));
    } else if (pm && lane == 5 && sev.end > sev.a1) {
      cp_async16_zfill(dev + (sev.a1 - sev.a0), t.esc_src + sev.a1, uint32_t(sev.end - sev.a1));
    }
    cp_async_mbar_arrive_noinc(full);
    ++it;
  }
  return true;
}

// The hand-off of finished tiles to the in-place decode's storer warp.
struct StoreHandoff {
  StoreSlot* sto;       // [2]
  uint64_t* out_full;   // [2]
  uint64_t* out_empty;  // [2]
};

// The 8 consumer warps of one pipeline (thread ctid of 256, named barrier
// `bar`): per stage a bounded wait and a vote, the dense decode of the tile
// with dec_lut in 4 registers (byte permutes), the escape patch in shared
// memory, then out[b] (b alternating per tile) goes to a TMA bulk store --
// issued here out of place, by the storer warp in place (INPLACE, which also
// marks each tile's read_done once its stage has landed).
template <bool INPLACE>
__device__ void consume(const Ring& r, uint16_t (*out)[kTile], uint32_t ctid, uint32_t bar, const DecWs& ws,
                        const StoreHandoff& ho) {
  uint32_t bad_escape = 0;
  uint32_t tiles_done = 0;  // finished tiles; the current tile goes to out[tiles_done & 1]
  bool in_tile = false;     // the previous stage left its tile open (more escape stages)
  // in place: waits (bounded) until the storer has read out[tiles_done & 1]'s previous tile
  auto out_free = [&]() -> bool {
    if constexpr (INPLACE) {
      return tiles_done < 2 || mbar_wait(&ho.out_empty[tiles_done & 1u], ((tiles_done >> 1) - 1) & 1u);
    } else {
      return true;
    }
  };
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kDecStages);
    const int ob = int(tiles_done & 1u);
    bool ok = mbar_wait(&r.full[s], (it / kDecStages) & 1);
    const DecStage& st = r.st[s];
    // read before the vote: after it, an invalid tile's stage is released
    const uint32_t flags = ok ? st.flags : 0u;
    const bool opens = ok && !in_tile && !(flags & (kStageEnd | kStageInvalid));  // writes out[ob] first
    if constexpr (INPLACE) {
      // The tile's payload bytes are in shared memory now (or it reads
      // none): the phase completes only after the copies' reads of global
      // memory have returned, so no store issued after this flag is seen can
      // change what they read.  A relaxed store suffices (a release fence
      // here, on every tile, cost a quarter of the kernel's time).
      if (ctid == 0 && ok && !(flags & (kStageCont | kStageEnd))) st_relaxed_u32(ws.read_done + st.tile, 1u);
      // a tile's first stage writes out[ob]: its previous tile must have been read
      if (opens) ok = out_free();
    } else {
      // the bulk store of out[ob]'s previous tile (two tiles back) must have read it
      if (opens && ctid == 0 && tiles_done >= 2) bulk_wait_read<1>();
    }
    if (named_bar_red_or(bar, kDecConsumers, !ok)) {
      if (ctid == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      break;
    }
    if (flags & kStageEnd) break;
    if (flags & kStageInvalid) {
      if (ctid == 0) mbar_arrive(&r.empty[s]);
      continue;
    }
    const uint32_t nt = st.n_tile;
    uint16_t* const outs = out[ob];
    if (!(flags & kStageCont)) {
      const uint4 dl = st.dec_lut;
      const uint32_t shift = st.sm_shift;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t grp = ctid + uint32_t(j) * kDecConsumers;  // 8 elements
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
      named_bar_sync(bar, kDecConsumers);
      const uint32_t chunk0 = st.lt * kChunksPerTile;
      // a tile's further stages hold their escapes from pk on (kEcapCont layout)
      const bool cont = (flags & kStageCont) != 0;
      const uint32_t* const cidb = cont ? reinterpret_cast<const uint32_t*>(st.pk) : st.cid;
      const uint16_t* const lposb = cont ? reinterpret_cast<const uint16_t*>(st.pk + kContLpos) : st.lpos;
      const uint8_t* const evb = cont ? st.pk + kContEv : st.ev;
      for (uint32_t k = ctid; k < m; k += kDecConsumers) {
        const uint32_t c = cidb[(st.cid_shift >> 2) + k];
        const uint32_t p = lposb[(st.lpos_shift >> 1) + k];
        const uint32_t ev = evb[st.ev_shift + k];
        const uint32_t rel = c - chunk0;
        const uint32_t pos = rel * kChunk + p;
        if (rel < kChunksPerTile && p < kChunk && pos < nt) {
          outs[pos] = uint16_t((outs[pos] & 0x807Fu) | (ev << 7));
        } else {
          bad_escape = 1;
        }
      }
    }
    const bool more = (flags & kStageMore) != 0;
    uint16_t* const gout = st.out;  // read before the stage is released
    fence_proxy_async_smem();
    named_bar_sync(bar, kDecConsumers);
    if (ctid == 0) {
      if (!more) {
        if constexpr (INPLACE) {
          // hand the finished tile to the storer (what it needs is read from
          // the stage before the stage is released)
          StoreSlot& so = ho.sto[ob];
          so.out = gout;
          so.tile = st.tile;
          so.lt = st.lt;
          so.nt = nt;
          so.dep = st.dep;
          so.dep2 = st.dep2;
          so.end = 0;
        } else {
          const uint32_t body = (nt * 2u) & ~15u;
          if (body) bulk_s2g(gout, outs, body);
          bulk_commit();
        }
      }
      mbar_arrive(&r.empty[s]);
      if constexpr (INPLACE) {
        if (!more) mbar_arrive(&ho.out_full[ob]);
      }
    }
    if constexpr (!INPLACE) {
      if (!more)  // the ragged end of the tile (under 8 elements) by plain stores
        for (uint32_t e = ((nt * 2u) & ~15u) / 2u + ctid; e < nt; e += kDecConsumers) gout[e] = outs[e];
    }
    in_tile = more;
    if (!more) ++tiles_done;
  }
  if (bad_escape) set_flag(ws.hdr, SZ_FLAG_ESCAPE);
  if constexpr (INPLACE) {
    // tell the storer there is nothing more (in the slot it reads next)
    if (ctid == 0) {
      if (!out_free()) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      ho.sto[tiles_done & 1u].end = 1;
      mbar_arrive(&ho.out_full[tiles_done & 1u]);
    }
  } else {
    if (ctid == 0) bulk_wait_all<0>();  // the tile stores have completed
  }
}

// In-place slot decode.  CTAs take tiles in the cyclic order above; the
// producer's lanes resolve each window from dec_prepare's ranges and tile ->
// item map, the pk bytes of phase C and the escape bytes come from the stash,
// each tile's read_done is set once its stage has landed, and the storer warp
// stores a tile only after the tiles whose in-place bytes lie under its
// output have been read.
__global__ void __launch_bounds__(kIpThreads, kIpCtasPerSm)
    dec_inplace(const __grid_constant__ Items items, DecWs ws) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  IpShared& sh = *reinterpret_cast<IpShared*>(smem_raw);
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
  const Ring ring{sh.st, sh.full, sh.empty};

  if (warp == kIpStorerWarp) {
    // ---------------------------------------------------------------- storer warp
    // Takes each finished output tile from the consumer warps and stores it
    // (TMA bulk store of its 16-byte body, plain stores for the ragged end),
    // once the tiles whose payload bytes lie under it have read them.
    // Waiting here keeps the consumers decoding the next tile into the other
    // output buffer.
    for (uint32_t k = 0;; ++k) {
      const int b = int(k & 1u);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sh.out_full[b], (k >> 1) & 1u))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        break;
      }
      const StoreSlot so = sh.sto[b];
      if (so.end) break;
      const uint32_t* p = dep_word(ws, so.tile, so.lt, so.dep, so.dep2, uint32_t(lane));
      const bool go = wait_words_warp(ws, p, p ? ld_relaxed_u32(p) : 1u, uint32_t(lane));
      if (lane == 0) {
        if (go) {
          fence_proxy_async_global();
        } else {
          set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
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

  if (warp == kIpProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    // When a window of kWin tiles starts, lane l resolves tile l of it in
    // parallel (escape range, item through the tile -> item map, payload,
    // output, dec_lut, section offsets, the sm and escape sources and the
    // tiles to wait for) into sh.win[l]; then the tiles are issued one by one
    // from that table.  Positions k of the CTA: k <-> position k % C of chunk
    // ticket blockIdx.x + (k / C) R.
    uint64_t it = 0;  // stages handed out
    const uint64_t R = gridDim.x;
    uint64_t Tu = 0;  // every tensor's tile count when they are all equal
    if (ws.hdr->tiles_differ == 0 && items.count > 0 && T % items.count == 0) Tu = T / items.count;
    const uint64_t C = ip_chunk_size(Tu);
    const uint64_t Q = ip_chunks(T, items.count, Tu, C);
    const uint64_t kend = blockIdx.x < Q ? (Q - blockIdx.x + R - 1) / R * C : 0;
    uint64_t next = 0;
    uint32_t win_len = 0, win_pos = 0;
    for (;;) {
      if (win_pos == win_len) {
        const uint64_t first = next;
        win_len = next < kend ? uint32_t((kend - next < kWin) ? kend - next : kWin) : 0u;
        next += win_len;
        win_pos = 0;
        if (win_len == 0) {
          issue_marker(ring, it, kStageEnd, 0, ws.hdr, uint32_t(lane));
          return;
        }
        __syncwarp();  // every lane is done with the previous window's entries
        if (uint32_t(lane) < win_len) {
          const uint64_t k = first + lane;
          const uint64_t mine = ip_tile_of(items, ws, blockIdx.x + (k / C) * R, k % C, T, Tu, C);
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
                ok = 1;
              }
            }
          }
          w.ok = ok;
        }
        __syncwarp();
      }
      const WinEntry& w = sh.win[win_pos++];
      if (w.tile == kNoTile) continue;  // past the end of a tensor: no stage
      if (!w.ok) {
        if (!issue_marker(ring, it, kStageInvalid, w.tile, ws.hdr, uint32_t(lane))) return;
        continue;
      }
      TileSrc t;
      t.base = w.base;
      t.pk_src = reinterpret_cast<const uint8_t*>(w.pkv);
      t.esc_src = reinterpret_cast<const uint8_t*>(w.escv);
      t.out = w.out;
      t.off_sm = w.off_sm;
      t.off_cid = w.off_cid;
      t.off_lpos = w.off_lpos;
      t.off_ev = w.off_ev;
      t.tile = w.tile;
      t.dec_lut = w.dec_lut;
      t.dep = w.dep;
      t.dep2 = w.dep2;
      t.k0 = w.k0;
      t.k1 = w.k1;
      t.lt = w.lt;
      t.nt = w.nt;
      if (!issue_tile<true>(ring, it, t, ws.hdr, uint32_t(lane))) return;
    }
  }

  consume<true>(ring, sh.out, uint32_t(tid), 1u, ws, StoreHandoff{sh.sto, sh.out_full, sh.out_empty});
}

// The carry of a CTA's first tile t0 in item `cur` (as found by
// find_item_warp): the tensor, checked, in `cache`, and the first escape of
// tile t0 by a 32-lane search (one round guided by the tensor's mean
// density, then 32-ary rounds, lower_bound_cid32).  A bad or gated tensor
// leaves the carry unknown: its tiles are rejected by the window resolution.
__device__ void prime_carry(const Items& items, uint64_t t0, uint32_t cur, uint32_t lane, RangeCarry& carry,
                            ItemCache& cache) {
  constexpr unsigned kAll = 0xFFFFFFFFu;
  carry = RangeCarry{kNoItem, 0u, 0u, 0.0f};
  const sz_item& it = item_at(items, cur);
  if (item_problems(items, cur, false) != 0) return;
  if (t0 < it.tile_begin || t0 - it.tile_begin >= tiles_of(it.n)) return;
  const sz_meta* mp = it.meta;
  const uint32_t lt0 = uint32_t(t0 - it.tile_begin);
  const uint32_t tiles = uint32_t(tiles_of(it.n));
  const uint32_t e = uint32_t(mp->n_esc);
  const int32_t* cid = reinterpret_cast<const int32_t*>(it.payload + mp->off_cid);
  uint32_t k = 0;
  if (lt0 > 0) {
    // the answer lies in [lo, hi]: at most 8192 escapes per tile before and after
    const uint64_t after = uint64_t(kTile) * (tiles - lt0);
    uint32_t lo = uint32_t(e > after ? e - after : 0);
    uint32_t hi = uint32_t(uint64_t(kTile) * lt0 < e ? uint64_t(kTile) * lt0 : e);
    const uint32_t target = 8u * lt0;
    if (hi - lo > 32u) {
      // one round around the mean-density guess, 32 probes `step` apart
      const uint64_t guess = uint64_t(e) * lt0 / tiles;
      const uint32_t step = guess_step(guess > lo ? guess - lo : 0) / 2u + 1u;
      int64_t p = int64_t(guess) + (int64_t(lane) - 16) * int64_t(step);
      p = p < int64_t(lo) ? int64_t(lo) : (p > int64_t(hi) - 1 ? int64_t(hi) - 1 : p);
      const uint32_t less = __ballot_sync(kAll, uint32_t(__ldg(cid + p)) < target);
      const uint32_t c = __popc(less);  // probes are non-decreasing: the less ones come first
      const uint32_t p_last_less = __shfl_sync(kAll, uint32_t(p), int(c ? c - 1u : 0u));
      const uint32_t p_first_ge = __shfl_sync(kAll, uint32_t(p), int(c < 32u ? c : 31u));
      if (c > 0) lo = p_last_less + 1u;
      if (c < 32u && p_first_ge >= lo) hi = p_first_ge;
      if (lo > hi) lo = hi;
    }
    // lower_bound_cid32 searches [0, e); here only [lo, hi) is open
    k = lo + lower_bound_cid32(cid + lo, hi - lo, target, lane);
  }
  carry = RangeCarry{cur, lt0, k, float(e) / float(tiles)};
  cache.payload = it.payload;
  cache.out = it.out;
  cache.n = it.n;
  cache.off_sm = mp->off_sm;
  cache.off_cid = mp->off_cid;
  cache.tile_begin = it.tile_begin;
  cache.dec_lut = *reinterpret_cast<const uint4*>(it.codebook->dec_lut);
  cache.e = e;
  cache.tiles = tiles;
}

// find_item_warp with 8 probes a lane (256 a round), for the resolver's first
// search, which lies on the path to the CTA's first tile: 8192 tensors take
// two dependent rounds of loads instead of three.
__device__ uint32_t find_item_wide(const Items& items, uint64_t tile, uint32_t lane) {
  constexpr unsigned kAll = 0xFFFFFFFFu;
  if (items.table == nullptr) return 0;
  uint32_t lo = 0, hi = items.count;  // table[lo].tile_begin <= tile; the answer is in [lo, hi)
  while (hi - lo > 32) {
    const uint32_t step = (hi - lo + 255) / 256;
    uint32_t c = 0;  // this lane's probes at or before `tile` (a prefix of them: the probes ascend)
#pragma unroll
    for (uint32_t k = 0; k < 8; ++k) {
      const uint64_t p = uint64_t(lo) + uint64_t(lane * 8u + k) * step;
      c += (p < hi && items.table[p].tile_begin <= tile) ? 1u : 0u;
    }
    const uint32_t total = __reduce_add_sync(kAll, c);  // probes 0 .. total-1 are at or before it
    if (total) lo += (total - 1u) * step;                // probe 0 is lo itself unless the table is not consecutive
    if (lo + step < hi) hi = lo + step;
  }
  const uint32_t p = lo + lane;
  const uint32_t m = __ballot_sync(kAll, p < hi && items.table[p].tile_begin <= tile);
  return m ? lo + (31u - __clz(m)) : lo;
}

// Out-of-place decode (sz_decode(_many)).  One CTA per SM owns a contiguous
// range of tiles, cut into windows of kFlatWin tiles.  The resolver warp
// resolves the windows in order (prime_carry for the first tile, then
// resolve_window: tensors, checks, escape ranges continued from window to
// window) into a pool of kPool tables; window w goes to table w % kPool,
// refilled once every tile of its previous window has been issued.  The two
// producer warps claim the CTA's tiles one at a time from a shared counter
// (tile i: window i / kFlatWin, entry i % kFlatWin), so the two pipelines
// stay within a tile of each other; each issues its tiles into its own ring,
// and each pipeline's 8 consumer warps decode, patch and store.
__global__ void __launch_bounds__(kFlatThreads, 1) dec_flat(const __grid_constant__ Items items, DecWs ws) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  FlatShared& sh = *reinterpret_cast<FlatShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  if (tid == 0) {
    for (int p = 0; p < kPipes; ++p)
      for (int s = 0; s < kDecStages; ++s) {
        mbar_init(&sh.full[p][s], 1 + 32);
        mbar_init(&sh.empty[p][s], 1);
      }
    for (uint32_t q = 0; q < kPool; ++q) {
      mbar_init(&sh.win_full[q], 1);
      mbar_init(&sh.win_empty[q], 1);
      sh.issued[q] = 0;
    }
    sh.next_tile = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t T = items.total_tiles;
  const uint64_t per = (T + gridDim.x - 1) / gridDim.x;
  uint64_t t1 = uint64_t(blockIdx.x + 1) * per;
  if (t1 > T) t1 = T;
  uint64_t t0 = uint64_t(blockIdx.x) * per;
  if (t0 > t1) t0 = t1;
  if (ws.small_done) {
    pdl_wait();  // dec_small's header bits
    if (!ws.hdr->large) return;  // dec_small decoded every tensor
  }

  if (warp == kFlatResolverWarp) {
    // ---------------------------------------------------------------- resolver warp
    if (t0 >= t1) return;
    RangeCarry carry;
    ItemCache& cache = sh.cache;
    uint32_t cur = find_item_wide(items, t0, uint32_t(lane));
    // a CTA whose first tile starts its tensor needs no carry: the first
    // window finds its tensors and escape ranges itself
    const bool kept = !ws.small_done || item_problems(items, cur, false) != 0 || !small_fits(item_at(items, cur));
    if (t0 != item_at(items, cur).tile_begin && kept) {
      prime_carry(items, t0, cur, uint32_t(lane), carry, cache);
    } else {
      carry = RangeCarry{kNoItem, 0u, 0u, 0.0f};
      if (lane == 0) cache = ItemCache{};
    }
    __syncwarp();
    for (uint32_t w = 0;; ++w) {
      const uint64_t first = t0 + uint64_t(w) * kFlatWin;
      if (first >= t1) return;
      const uint32_t len = uint32_t((t1 - first < kFlatWin) ? t1 - first : kFlatWin);
      const uint32_t q = w % kPool;
      if (w >= kPool && !__all_sync(0xFFFFFFFFu, mbar_wait(&sh.win_empty[q], ((w / kPool) - 1) & 1u))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return;
      }
      resolve_window(items, ws, sh.win[q], first, len, uint32_t(lane), cur, carry, cache);
      if (lane == 0) sh.win_len[q] = len;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.win_full[q]);  // releases the table's writes to the producers
    }
  }

  if (warp >= kFlatProducerWarp) {
    // ---------------------------------------------------------------- producer warps
    const int p = warp - kFlatProducerWarp;
    const Ring ring{sh.st[p], sh.full[p], sh.empty[p]};
    uint64_t it = 0;  // stages handed out
    for (;;) {
      uint32_t i = 0;
      if (lane == 0) i = atomicAdd(&sh.next_tile, 1u);
      i = __shfl_sync(0xFFFFFFFFu, i, 0);
      if (t0 + i >= t1) {
        issue_marker(ring, it, kStageEnd, 0, ws.hdr, uint32_t(lane));
        return;
      }
      const uint32_t w = i / kFlatWin;
      const uint32_t q = w % kPool;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sh.win_full[q], (w / kPool) & 1u))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return;
      }
      const WinOut& e = sh.win[q][i % kFlatWin];
      if (!e.ok) {
        if (!issue_marker(ring, it, kStageInvalid, e.tile, ws.hdr, uint32_t(lane))) return;
      } else {
        TileSrc t;
        t.base = e.base;
        t.pk_src = t.esc_src = e.base;
        t.out = e.out;
        t.off_sm = e.off_sm;
        t.off_cid = e.off_cid;
        t.off_lpos = e.off_cid + 4ull * e.n_esc;
        t.off_ev = round_up4(t.off_lpos + 2ull * e.n_esc);
        t.tile = e.tile;
        t.dec_lut = e.dec_lut;
        t.k0 = e.k0;
        t.k1 = e.k1;
        t.lt = e.lt;
        t.nt = e.nt;
        if (!issue_tile<false>(ring, it, t, ws.hdr, uint32_t(lane))) return;
      }
      // the last of a window's tiles to be issued frees its table
      __syncwarp();  // every lane has read the entry
      if (lane == 0 && atomicAdd(&sh.issued[q], 1u) + 1u == sh.win_len[q]) {
        sh.issued[q] = 0;
        mbar_arrive(&sh.win_empty[q]);
      }
    }
  }

  // ------------------------------------------------------------------ consumer warps
  const int p = warp / kDecConsumerWarps;
  consume<false>(Ring{sh.st[p], sh.full[p], sh.empty[p]}, sh.out[p], uint32_t(tid - p * kDecConsumers),
                 1u + uint32_t(p), ws, StoreHandoff{nullptr, nullptr, nullptr});
}

// ---------------------------------------------------------------- small tensors
// Out-of-place decode of tables of small tensors (sz_decode_many over
// tensors of at most two tiles on average, e.g. the blocks of a paged KV
// cache; the pages' decode_torch, tensor by tensor).  dec_flat's first tile
// waits for a chain of dependent loads (tensor search, meta, chunk_id search)
// before its first copy; here a tensor's whole payload (at most kSdPay
// bytes) is copied into shared memory after one table read and one meta read,
// and one group of 8 warps decodes it straight to HBM:
//   * an evaluation warp checks the CTA's tensors 32 at a time (one lane
//     each: item checks, meta, dec_lut) into a double-buffered table;
//   * a copy warp copies each payload by TMA into a ring of kSdBufs buffers;
//   * groups of 8 warps take the tensors in turn: each thread decodes 8
//     elements per step (dec_lut in 4 registers) and stores 16 bytes; after a
//     group barrier the escapes are written over their elements (sign and
//     mantissa from the sm byte, exponent from esc_val), which is all an
//     escape changes.
// A tensor with more elements, or a larger payload, is left to dec_flat:
// the header's `large` bit tells it to run.
constexpr uint32_t kSdGroups = 3;
constexpr uint32_t kSdGroupThreads = 256;
constexpr uint32_t kSdEvalWarp = kSdGroups * 8;     // 24
constexpr uint32_t kSdCopyWarp = kSdEvalWarp + 1;   // 25
constexpr uint32_t kSdThreads = (kSdCopyWarp + 1) * 32;  // 832
constexpr uint32_t kSdBufs = 8;
constexpr uint32_t kSdBatch = 32;  // tensors per evaluation batch
constexpr uint32_t kSdDecode = 0u, kSdSkip = 1u;

struct SdInfo {  // one tensor, as the evaluation warp leaves it
  const uint8_t* payload;
  uint16_t* out;
  uint32_t n, e, comp, off_sm, off_cid, off_lpos, off_ev;
  uint32_t status;  // kSdDecode, or kSdSkip (bad, gated, empty, or left to dec_flat)
  uint4 dec_lut;
};
static_assert(sizeof(SdInfo) == 64, "64 bytes");

struct SdShared {
  alignas(128) uint8_t pay[kSdBufs][kSdPay + 128];  // a tensor's payload (+ slack for over-reads of its last group)
  SdInfo info[2][kSdBatch];
  SdInfo slot[kSdBufs];   // the tensor of pay[b]
  uint32_t slot_item[kSdBufs];
  uint64_t full[kSdBufs], empty[kSdBufs];
  uint64_t info_full[2], info_empty[2];
};
static_assert(sizeof(SdShared) <= 227u * 1024u, "one CTA per SM");

__global__ void __launch_bounds__(kSdThreads, 1) dec_small(const __grid_constant__ Items items, DecWs ws) {
  constexpr unsigned FULL = 0xFFFFFFFFu;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SdShared& sh = *reinterpret_cast<SdShared*>(smem_raw);
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
  pdl_trigger();  // dec_flat, launched after, waits for this grid before it reads the header
  if (tid == 0) {
    for (uint32_t b = 0; b < kSdBufs; ++b) {
      mbar_init(&sh.full[b], 1 + 32);
      mbar_init(&sh.empty[b], 8);
    }
    for (uint32_t h = 0; h < 2; ++h) {
      mbar_init(&sh.info_full[h], 1);
      mbar_init(&sh.info_empty[h], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t G = gridDim.x;
  const uint32_t K = blockIdx.x < items.count ? (items.count - 1u - blockIdx.x) / G + 1u : 0u;  // the CTA's tensors

  if (warp == kSdEvalWarp) {
    // ---------------------------------------------------------------- evaluation warp
    for (uint32_t bt = 0; bt * kSdBatch < K; ++bt) {
      const uint32_t h = bt & 1u;
      if (bt >= 2 && !__all_sync(FULL, mbar_wait(&sh.info_empty[h], ((bt >> 1) - 1) & 1u))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return;
      }
      const uint32_t k = bt * kSdBatch + lane;
      SdInfo inf{};
      inf.status = kSdSkip;
      if (k < K) {
        const uint32_t i = blockIdx.x + k * G;
        const uint32_t bad = item_problems(items, i, false);
        const sz_item& it = item_at(items, i);
        if (bad & ~kItemGated) {
          set_flag(ws.hdr, bad & ~kItemGated);
        } else if (!bad && it.n > 0) {
          if (!small_fits(it)) {
            atomicOr(&ws.hdr->large, 1u);  // dec_flat decodes it
          } else {
            const sz_meta* mp = it.meta;
            inf.payload = it.payload;
            inf.out = it.out;
            inf.n = uint32_t(it.n);
            inf.e = uint32_t(mp->n_esc);
            inf.comp = uint32_t(mp->comp_bytes);
            inf.off_sm = uint32_t(mp->off_sm);
            inf.off_cid = uint32_t(mp->off_cid);
            inf.off_lpos = uint32_t(mp->off_lpos);
            inf.off_ev = uint32_t(mp->off_ev);
            inf.dec_lut = *reinterpret_cast<const uint4*>(it.codebook->dec_lut);
            inf.status = kSdDecode;
          }
        }
      }
      sh.info[h][lane] = inf;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.info_full[h]);
    }
    return;
  }

  if (warp == kSdCopyWarp) {
    // ---------------------------------------------------------------- copy warp
    // Tensor k into buffer k % kSdBufs once the group done with tensor
    // k - kSdBufs has released it; after the K tensors, one end slot per group.
    for (uint32_t k = 0; k < K + kSdGroups; ++k) {
      const uint32_t b = k % kSdBufs;
      if (k >= kSdBufs && !__all_sync(FULL, mbar_wait(&sh.empty[b], ((k / kSdBufs) - 1) & 1u))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return;
      }
      uint32_t bytes = 0;
      const uint8_t* src = nullptr;
      if (k < K) {
        const uint32_t bt = k / kSdBatch, h = bt & 1u, j = k % kSdBatch;
        if (j == 0 && !__all_sync(FULL, mbar_wait(&sh.info_full[h], (bt >> 1) & 1u))) {
          if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
          return;
        }
        const SdInfo& inf = sh.info[h][j];
        if (lane < 16) reinterpret_cast<uint32_t*>(&sh.slot[b])[lane] = reinterpret_cast<const uint32_t*>(&inf)[lane];
        if (inf.status == kSdDecode) {
          bytes = inf.comp;
          src = inf.payload;
        }
        __syncwarp();
        if (lane == 0 && (j + 1 == kSdBatch || k + 1 == K)) mbar_arrive(&sh.info_empty[h]);  // the batch is copied out
      }
      if (lane == 0) sh.slot_item[b] = k < K ? k : kNoItem;
      __syncwarp();  // the slot is written before the barrier's arrivals
      const uint32_t bulk = bytes & ~15u;
      if (lane == 0) {
        mbar_arrive_expect_tx(&sh.full[b], bulk);
        if (bulk) bulk_g2s(sh.pay[b], src, bulk, &sh.full[b]);
      } else if (lane == 1 && bytes > bulk) {
        cp_async16_zfill(sh.pay[b] + bulk, src + bulk, bytes - bulk);
      }
      cp_async_mbar_arrive_noinc(&sh.full[b]);
    }
    return;
  }

  // ------------------------------------------------------------------ decoding groups
  const uint32_t g = warp / 8u, gt = tid % kSdGroupThreads, bar_id = 1u + g;
  bool bad_escape = false;
  for (uint32_t k = g;; k += kSdGroups) {
    const uint32_t b = k % kSdBufs;
    const bool ok = mbar_wait(&sh.full[b], (k / kSdBufs) & 1u);
    if (named_bar_red_or(bar_id, kSdGroupThreads, !ok)) {
      if (gt == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      break;
    }
    if (sh.slot_item[b] == kNoItem) break;
    const SdInfo& sl = sh.slot[b];
    if (sl.status == kSdDecode) {
      const uint8_t* const pay = sh.pay[b];
      const uint32_t n = sl.n, e = sl.e, off_sm = sl.off_sm;
      uint16_t* const out = sl.out;
      const uint4 dl = sl.dec_lut;
      // dense decode, 8 elements a thread per step (the last group may read
      // past the payload's end into the buffer's slack: those lanes' values
      // beyond n are not stored)
      for (uint32_t q = gt; 8u * q < n; q += kSdGroupThreads) {
        const uint32_t c8 = *reinterpret_cast<const uint32_t*>(pay + 4u * q);
        const uint32_t s_lo = *reinterpret_cast<const uint32_t*>(pay + off_sm + 8u * q);
        const uint32_t s_hi = *reinterpret_cast<const uint32_t*>(pay + off_sm + 8u * q + 4u);
        const uint2 lo = decode4(c8 & 0xFFFFu, s_lo, dl.x, dl.y, dl.z, dl.w);
        const uint2 hi = decode4(c8 >> 16, s_hi, dl.x, dl.y, dl.z, dl.w);
        if (8u * q + 8u <= n) {
          *reinterpret_cast<uint4*>(out + 8u * q) = make_uint4(lo.x, lo.y, hi.x, hi.y);
        } else {
          for (uint32_t r = 0; 8u * q + r < n; ++r) {
            const uint32_t w = r < 2u ? lo.x : (r < 4u ? lo.y : (r < 6u ? hi.x : hi.y));
            out[8u * q + r] = uint16_t(w >> (16u * (r & 1u)));
          }
        }
      }
      // the escapes over their elements (after every dense store of the group)
      named_bar_sync(bar_id, kSdGroupThreads);
      const uint32_t chunks = (n + kChunk - 1u) / kChunk;
      for (uint32_t j = gt; j < e; j += kSdGroupThreads) {
        const uint32_t c = *reinterpret_cast<const uint32_t*>(pay + sl.off_cid + 4u * j);
        const uint32_t lp = *reinterpret_cast<const uint16_t*>(pay + sl.off_lpos + 2u * j);
        const uint32_t ev = pay[sl.off_ev + j];
        const uint32_t pos = c * kChunk + lp;
        if (c < chunks && lp < kChunk && pos < n) {
          const uint32_t sm = pay[off_sm + pos];
          out[pos] = uint16_t(((sm & 0x80u) << 8) | (ev << 7) | (sm & 0x7Fu));
        } else {
          bad_escape = true;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[b]);  // this warp is done with pay[b] and slot[b]
  }
  if (__any_sync(FULL, bad_escape) && lane == 0) set_flag(ws.hdr, SZ_FLAG_ESCAPE);
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

// Opts a kernel into its dynamic shared memory once per device and host
// thread; returns its resident CTAs per SM.
cudaError_t configure(const void* fn, size_t smem, int threads, int device, int* configured_device, int* per_sm) {
  if (*configured_device == device) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (err != cudaSuccess) return err;
  int nb = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem);
  if (err != cudaSuccess) return err;
  if (nb < 1) return cudaErrorInvalidConfiguration;
  *per_sm = nb;
  *configured_device = device;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_decode(const Items& items, void* ws_base, cudaStream_t stream, const DeviceInfo& dev,
                          bool clear_header) {
  cudaError_t err = clear_header ? cudaMemsetAsync(ws_base, 0, sizeof(WsHeader), stream) : cudaSuccess;
  if (err != cudaSuccess || items.total_tiles == 0) return err;
  static thread_local int configured_device = -1, per_sm = 1;
  const size_t smem = sizeof(FlatShared);
  err = configure(reinterpret_cast<const void*>(dec_flat), smem, kFlatThreads, dev.device, &configured_device,
                  &per_sm);
  if (err != cudaSuccess) return err;
  const uint64_t cap = uint64_t(dev.num_sms);  // one CTA per SM: its two pipelines share the SM's tiles
  const unsigned grid = unsigned(items.total_tiles < cap ? items.total_tiles : cap);
  if (small_route(items)) {
    // tables of small tensors: dec_small decodes what fits it, then dec_flat
    // (programmatic dependent launch) returns at once unless it left a tensor
    static thread_local int configured_small = -1, per_sm_small = 1;
    err = configure(reinterpret_cast<const void*>(dec_small), sizeof(SdShared), kSdThreads, dev.device,
                    &configured_small, &per_sm_small);
    if (err != cudaSuccess) return err;
    DecWs ws = dec_ws(ws_base);
    if (!clear_header && (err = cudaMemsetAsync(&ws.hdr->large, 0, sizeof(uint32_t), stream)) != cudaSuccess)
      return err;
    const unsigned sgrid = unsigned(items.count < cap ? items.count : cap);
    if (g_timing.before) cudaEventRecord(g_timing.before, stream);
    dec_small<<<sgrid, kSdThreads, sizeof(SdShared), stream>>>(items, ws);
    err = cudaGetLastError();
    if (g_timing.after) cudaEventRecord(g_timing.after, stream);
    if (err != cudaSuccess) return err;
    ws.small_done = true;
    return launch_pdl(dec_flat, dim3(grid), dim3(kFlatThreads), smem, stream, items, ws);
  }
  if (g_timing.before) cudaEventRecord(g_timing.before, stream);
  dec_flat<<<grid, kFlatThreads, smem, stream>>>(items, dec_ws(ws_base));
  err = cudaGetLastError();
  if (g_timing.after) cudaEventRecord(g_timing.after, stream);
  return err;
}

cudaError_t launch_wait_selftest(void* ws_base, cudaStream_t stream) {
  // workspace: header | never (u32, zero) | gave_up[3] u32
  DecWs ws = dec_ws(ws_base);
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
  err = launch_pdl(dip_stash, dim3(unsigned(blocks < cap ? blocks : cap)), dim3(kStashWarps * 32), 0, stream, items, ws);
  if (err != cudaSuccess) return err;
  static thread_local int configured_device = -1, per_sm = kIpCtasPerSm;
  const size_t smem = sizeof(IpShared);
  err = configure(reinterpret_cast<const void*>(dec_inplace), smem, kIpThreads, dev.device, &configured_device,
                  &per_sm);
  if (err != cudaSuccess) return err;
  const uint64_t cap_ip = uint64_t(dev.num_sms) * (per_sm < kIpCtasPerSm ? per_sm : kIpCtasPerSm);
  const unsigned grid = unsigned(items.total_tiles < cap_ip ? items.total_tiles : cap_ip);
  if (g_timing.before) cudaEventRecord(g_timing.before, stream);
  // tiles wait for tiles of other CTAs' runs: every CTA must be resident
  Items it = items;
  DecWs w = ws;
  void* args[] = {&it, &w};
  err = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(dec_inplace), dim3(grid), dim3(kIpThreads), args,
                                    smem, stream);
  if (g_timing.after) cudaEventRecord(g_timing.after, stream);
  return err;
}

}  // namespace sz
