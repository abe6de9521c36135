// Encode ("splitzip_codec.py" encode_torch + assemble_payload): one streaming
// pass over the input, then the in-order placement of the escape stream.
//
// Launches per call (after a 256-byte header memset):
//   enc_prepare  validates the item table, zeroes per-tensor escape totals,
//                segment tickets and segment status words;
//   enc_main     persistent CTAs own contiguous runs of 8192-element tiles.
//                A producer warp streams each tile (and the tensor's enc_lut)
//                into a 4-stage shared-memory ring with TMA bulk copies; 8
//                chunk warps -- warp w owns chunk w (1024 elements) -- split
//                and pack with coalesced pk/sm stores, and compact the chunk's
//                escapes with ballot/popc in element order into the chunk's
//                staging slot.  The chunk counts and each tensor's escape
//                total are recorded.  No warp ever waits on another CTA.
//   enc_place    per tensor, segments of 256 chunks (claimed by ticket, so
//                segments start in order): a block scan of the chunk counts
//                and a decoupled lookback across the tensor's segments give
//                each escape its global index; chunk_id, local_pos and
//                esc_val are then written once, in order, at their final
//                offsets (the tensor's total is already known, so every
//                offset is).  The segment holding chunk 0 also zeroes the pad
//                bytes and writes the meta.
// Every wait is bounded (kWaitTimeoutNs); on timeout SZ_FLAG_TIMEOUT is raised.
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kEncStages = 4;
constexpr int kEncChunkWarps = kChunksPerTile;  // one warp per chunk
constexpr int kProducerWarp = kEncChunkWarps;
constexpr int kEncThreads = (kEncChunkWarps + 1) * 32;
constexpr int kEncCtasPerSm = 2;
constexpr uint32_t kStageEnd = 1u, kStageInvalid = 2u;
constexpr unsigned FULL = 0xFFFFFFFFu;
constexpr uint32_t kSegChunks = 256;                     // chunks per placement segment
constexpr uint32_t kSegTiles = kSegChunks / kChunksPerTile;  // 32
constexpr unsigned long long kAgg = 1ull << 32, kIncl = 2ull << 32;

struct __align__(128) EncStage {
  uint16_t x[kTile];     // the tile's BF16 bit patterns
  uint8_t enc_lut[256];  // the tensor's codebook enc_lut
  unsigned long long tile;  // global tile index
  uint8_t* payload;
  uint64_t off_sm;
  uint32_t lt, n_tile, flags, item;
};

constexpr uint32_t kRun = 4;  // tiles per ticket

// What the producer needs of an item; cached in shared memory for tables of
// up to kCachedItems items, so mapping a ticket to its item costs no global
// round trip.
constexpr uint32_t kCachedItems = 128;
struct ItemLite {
  uint64_t tile_begin, n;
  const uint16_t* x;
  uint8_t* payload;
  const uint8_t* enc_lut;
  uint32_t flags, pad;
};

__device__ __forceinline__ ItemLite item_lite(const Items& items, const EncWs& ws, uint32_t i) {
  const sz_item& it = item_at(items, i);
  ItemLite l;
  l.tile_begin = it.tile_begin;
  l.n = it.n;
  l.x = it.x;
  l.payload = it.payload;
  l.flags = ws.item_flags[i];
  l.enc_lut = l.flags ? nullptr : it.codebook->enc_lut;
  l.pad = 0;
  return l;
}

struct EncShared {
  ItemLite item[kCachedItems];
  EncStage st[kEncStages];
  uint64_t full[kEncStages];
  uint64_t empty[kEncStages];
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
    ws.item_esc[i] = 0;
    ws.seg_ticket[i] = 0;
    if (bad) set_flag(ws.hdr, bad);
  }
}

__device__ __forceinline__ uint32_t sm_pair(uint32_t w) {
  // two BF16 patterns in w -> sm bytes at byte 0 and byte 2
  return (w & 0x007F007Fu) | ((w >> 8) & 0x00800080u);
}

// Bounded mbarrier wait agreed by the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(FULL, mbar_wait(bar, parity));
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
// in element order into (lslot, eslot).  Each lane handles 4 consecutive
// elements per row of 128.  Escape handling is byte-parallel: an enc_lut value
// >= 16 (a non-zero high nibble) marks an escape, stored in pk as code 0.
// Returns the chunk's escape count.  FULL_TILE: all 8192 elements exist.
template <bool FULL_TILE>
__device__ __forceinline__ uint32_t encode_chunk(const EncStage& st, uint32_t warp, uint32_t lane, uint16_t* lslot,
                                                 uint8_t* eslot) {
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
    if (__ballot_sync(FULL, m != 0)) {
      const uint32_t escm = ((m >> 7) & 1u) | ((m >> 14) & 2u) | ((m >> 21) & 4u) | ((m >> 28) & 8u);
      const uint32_t b0 = __ballot_sync(FULL, escm & 1u), b1 = __ballot_sync(FULL, escm & 2u);
      const uint32_t b2 = __ballot_sync(FULL, escm & 4u), b3 = __ballot_sync(FULL, escm & 8u);
      uint32_t pos = run + __popc(b0 & lane_lt) + __popc(b1 & lane_lt) + __popc(b2 & lane_lt) +
                     __popc(b3 & lane_lt);
      const uint32_t ex[4] = {(v.x >> 7) & 0xFFu, (v.x >> 23) & 0xFFu, (v.y >> 7) & 0xFFu, (v.y >> 23) & 0xFFu};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if ((escm >> k) & 1u) {
          lslot[pos] = uint16_t(row * 128 + lane * 4 + k);
          eslot[pos] = uint8_t(ex[k]);
          ++pos;
        }
      }
      run += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
    }
  }
  return run;
}

// sm bytes of the two BF16 patterns of w at bytes 0 and 2 (bytes 1 and 3 are
// don't-care): bit 7 of each comes from bit 15 of its pattern.
__device__ __forceinline__ uint32_t sm_pair_lo(uint32_t w) {
  const uint32_t s = w >> 8;
  return (w & 0x007F007Fu) | (s & ~0x007F007Fu);  // one bit-select
}

// Exclusive warp prefix of per-lane counts `c` (0..8) and the warp total.
// Most rows hold at most one escape per lane: then two ballots suffice.
__device__ __forceinline__ uint32_t warp_prefix(uint32_t c, uint32_t lane, uint32_t* total) {
  const uint32_t lane_lt = (1u << lane) - 1u;
  const uint32_t b1 = __ballot_sync(FULL, c >= 1);
  const uint32_t b2 = __ballot_sync(FULL, c >= 2);
  if (b2 == 0) {
    *total = __popc(b1);
    return __popc(b1 & lane_lt);
  }
  uint32_t incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL, incl, d);
    if (lane >= uint32_t(d)) incl += o;
  }
  *total = __shfl_sync(FULL, incl, 31);
  return incl - c;
}

// Full tile, 8 elements per lane per row of 256 (4 rows per chunk).
// Same output as encode_chunk<true>: pk/sm of the chunk, its escapes in
// element order in (lslot, eslot); returns the escape count.
__device__ __forceinline__ uint32_t encode_chunk8(const EncStage& st, uint32_t warp, uint32_t lane, uint16_t* lslot,
                                                  uint8_t* eslot) {
  const uint8_t* lut = st.enc_lut;
  const uint64_t g = uint64_t(st.lt) * kTile;
  const uint32_t e0 = warp * kChunk + lane * 8u;
  const uint16_t* xw = st.x + e0;
  uint8_t* pkw = st.payload + (g >> 1) + (e0 >> 1);
  uint8_t* smw = st.payload + st.off_sm + g + e0;
  const bool sm8 = ((st.off_sm & 7u) == 0);
  uint32_t lane_esc = 0;  // bit 8*row + k: element k of this lane's 8 in `row` escapes
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
    uint32_t clo = lo & 0x0F0F0F0Fu, chi = hi & 0x0F0F0F0Fu;
    if ((lo | hi) & 0xF0F0F0F0u) {  // an enc_lut value >= 16: escape, stored as code 0
      const uint32_t mlo = (((lo & 0xF0F0F0F0u) >> 4) + 0x7F7F7F7Fu) & 0x80808080u;
      const uint32_t mhi = (((hi & 0xF0F0F0F0u) >> 4) + 0x7F7F7F7Fu) & 0x80808080u;
      clo &= ~((mlo >> 7) * 0xFFu);
      chi &= ~((mhi >> 7) * 0xFFu);
      // gather bit 7 of each byte (element k of the 8) into bit k of this row's byte
      const uint32_t g = ((((mlo >> 7) * 0x00204081u) >> 21) & 0xFu) | (((((mhi >> 7) * 0x00204081u) >> 21) & 0xFu) << 4);
      lane_esc |= g << (8 * row);
    }
    const uint32_t tlo = clo | (clo >> 4), thi = chi | (chi >> 4);
    *reinterpret_cast<uint32_t*>(pkw + row * 128) = __byte_perm(tlo, thi, 0x6420);
    const uint32_t s01 = __byte_perm(sm_pair_lo(v.x), sm_pair_lo(v.y), 0x6420);
    const uint32_t s23 = __byte_perm(sm_pair_lo(v.z), sm_pair_lo(v.w), 0x6420);
    if (sm8) {
      *reinterpret_cast<uint2*>(smw + row * 256) = make_uint2(s01, s23);
    } else {
      *reinterpret_cast<uint32_t*>(smw + row * 256) = s01;
      *reinterpret_cast<uint32_t*>(smw + row * 256 + 4) = s23;
    }
  }
  // Escapes of the chunk, in element order (row, lane, k): one pass per chunk.
  if (__ballot_sync(FULL, lane_esc != 0) == 0) return 0;
  const uint32_t lane_lt = (1u << lane) - 1u;
  uint32_t c[4], before[4];
  bool simple = true;  // at most one escape per lane and row: ballots give the prefixes
#pragma unroll
  for (int row = 0; row < 4; ++row) {
    c[row] = __popc((lane_esc >> (8 * row)) & 0xFFu);
    simple &= (c[row] <= 1);
  }
  uint32_t run = 0;
  if (__all_sync(FULL, simple)) {
#pragma unroll
    for (int row = 0; row < 4; ++row) {
      const uint32_t b = __ballot_sync(FULL, c[row] != 0);
      before[row] = run + __popc(b & lane_lt);
      run += __popc(b);
    }
  } else {
#pragma unroll
    for (int row = 0; row < 4; ++row) {
      uint32_t total;
      before[row] = run + warp_prefix(c[row], lane, &total);
      run += total;
    }
  }
  const uint16_t* xc = st.x + warp * kChunk;
#pragma unroll
  for (int row = 0; row < 4; ++row) {
    uint32_t pos = before[row];
    for (uint32_t m = (lane_esc >> (8 * row)) & 0xFFu; m; m &= m - 1) {
      const uint32_t elem = uint32_t(row) * 256u + lane * 8u + uint32_t(__ffs(m) - 1);  // chunk-local
      lslot[pos] = uint16_t(elem);
      eslot[pos] = uint8_t((xc[elem] >> 7) & 0xFFu);
      ++pos;
    }
  }
  return run;
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

  const uint64_t T = items.total_tiles;

  if (tid == 0) {
    for (int s = 0; s < kEncStages; ++s) {
      mbar_init(&sh.full[s], 1 + 32);
      mbar_init(&sh.empty[s], kEncChunkWarps);
    }
    fence_mbar_init();
  }
  if (items.count <= kCachedItems)
    for (uint32_t i = tid; i < items.count; i += kEncThreads) sh.item[i] = item_lite(items, ws, i);
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    // Tiles are handed out in runs of kRun from a device-wide ticket, so CTAs
    // that run faster (SM placement, neighbours) take more of them.
    unsigned long long run_base = 0;
    uint32_t run_pos = kRun;
    uint32_t cur = 0xFFFFFFFFu;
    ItemLite itm{};
    for (uint32_t it = 0;; ++it) {
      const int s = int(it % kEncStages);
      if (it >= uint32_t(kEncStages) && !warp_wait(&sh.empty[s], ((it / kEncStages) - 1) & 1)) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return;
      }
      if (run_pos == kRun) {
        if (lane == 0) run_base = atomicAdd(&ws.hdr->ticket, 1ull * kRun);
        run_base = __shfl_sync(FULL, run_base, 0);
        run_pos = 0;
      }
      const uint64_t t = run_base + run_pos++;
      EncStage& st = sh.st[s];
      if (t >= T) {
        if (lane == 0) {
          st.flags = kStageEnd;
          mbar_arrive(&sh.full[s]);
        }
        cp_async_mbar_arrive_noinc(&sh.full[s]);
        return;
      }
      if (cur == 0xFFFFFFFFu || t < itm.tile_begin || t >= itm.tile_begin + tiles_of(itm.n)) {
        if (items.count <= kCachedItems) {
          // last cached item with tile_begin <= t (empty items own no tile)
          uint32_t lo = 0, hi = items.count;
          while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (sh.item[mid].tile_begin <= t) lo = mid; else hi = mid;
          }
          cur = lo;
          itm = sh.item[cur];
        } else {
          cur = find_item(items, t);
          itm = item_lite(items, ws, cur);
        }
      }
      const uint64_t cur_begin = itm.tile_begin;
      const uint32_t lt = uint32_t(t - cur_begin);
      const uint64_t g = uint64_t(lt) * kTile;
      const bool invalid = itm.flags != 0 || g >= itm.n;
      const uint32_t nt = invalid ? 0u : ((itm.n - g < kTile) ? uint32_t(itm.n - g) : kTile);
      const uint32_t bulk = (nt * 2u) & ~15u;
      const uint32_t tail = nt * 2u - bulk;
      if (lane == 0) {
        st.tile = t;
        st.item = cur;
        st.lt = lt;
        st.n_tile = nt;
        st.flags = invalid ? kStageInvalid : 0u;
        if (!invalid) {
          st.payload = itm.payload;
          st.off_sm = layout_of(itm.n, 0).off_sm;
          mbar_arrive_expect_tx(&sh.full[s], bulk + 256u);
          if (bulk) bulk_g2s(st.x, itm.x + g, bulk, &sh.full[s]);
          bulk_g2s(st.enc_lut, itm.enc_lut, 256u, &sh.full[s]);
        } else {
          mbar_arrive(&sh.full[s]);
        }
      } else if (lane == 1 && tail) {
        cp_async16_zfill(reinterpret_cast<uint8_t*>(st.x) + bulk,
                         reinterpret_cast<const uint8_t*>(itm.x + g) + bulk, tail);
      }
      cp_async_mbar_arrive_noinc(&sh.full[s]);
    }
  }

  // ------------------------------------------------------------------ chunk warps
  // Escape totals per tensor are accumulated per warp and added to the global
  // total only when the tensor changes: one global atomic per chunk would pile
  // hundreds of thousands of updates onto a few words (one L2 slice).
  uint32_t acc_item = 0xFFFFFFFFu, acc = 0;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    if (!warp_wait(&sh.full[s], (it / kEncStages) & 1)) {
      if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      break;
    }
    const EncStage& st = sh.st[s];
    const uint32_t flags = st.flags;
    if (flags & kStageEnd) break;
    if (!(flags & kStageInvalid)) {
      const uint64_t chunk = st.tile * kChunksPerTile + uint32_t(warp);  // global chunk index
      uint16_t* lslot = ws.lpos + chunk * kChunk;
      uint8_t* eslot = ws.ev + chunk * kChunk;
      const uint32_t run = (st.n_tile == kTile)
                               ? encode_chunk8(st, uint32_t(warp), uint32_t(lane), lslot, eslot)
                               : encode_chunk<false>(st, uint32_t(warp), uint32_t(lane), lslot, eslot);
      if (st.item != acc_item) {
        if (lane == 0 && acc) atomicAdd(ws.item_esc + acc_item, acc);
        acc_item = st.item;
        acc = 0;
      }
      acc += run;
      if (lane == 0) ws.chunk_cnt[chunk] = uint16_t(run);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
  }
  if (lane == 0 && acc) atomicAdd(ws.item_esc + acc_item, acc);
}

// Decoupled lookback over the placement segments of one tensor: lane l reads
// the status of segment j - l (status word at the segment's first tile,
// tile_begin + seg * kSegTiles).  Segment 0 always publishes an inclusive
// prefix.  Returns the exclusive prefix of segment j + 1.  Bounded.
__device__ uint32_t segment_lookback(const unsigned long long* status, uint64_t tile_begin, int64_t j,
                                     bool* timed_out) {
  const uint32_t lane = threadIdx.x & 31u;
  uint32_t excl = 0;
  uint64_t t0 = 0;
  uint32_t spins = 0;
  for (;;) {
    if (j < 0) return excl;  // cannot happen: segment 0 is inclusive
    const int64_t seg = j - int64_t(lane);
    const unsigned long long v = seg >= 0 ? ld_relaxed_u64(status + tile_begin + uint64_t(seg) * kSegTiles) : kIncl;
    const unsigned long long flag = v & ~0xFFFFFFFFull;
    const uint32_t incl = __ballot_sync(FULL, flag == kIncl);
    const uint32_t zero = __ballot_sync(FULL, flag == 0);
    const uint32_t stop = incl ? uint32_t(__ffs(incl) - 1) : 31u;
    const uint32_t upto = (stop == 31u) ? FULL : ((2u << stop) - 1u);
    if (zero & upto) {
      __nanosleep(32);
      if ((++spins & 15) == 0) {
        const uint64_t now = global_timer_ns();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > kWaitTimeoutNs) {
          *timed_out = true;
          return excl;
        }
      }
      continue;
    }
    excl += __reduce_add_sync(FULL, lane <= stop ? uint32_t(v) : 0u);
    if (incl) return excl;
    j -= 32;
  }
}

constexpr int kPlaceThreads = kSegChunks;  // one thread per chunk of the segment

__global__ void __launch_bounds__(kPlaceThreads) enc_place(const __grid_constant__ Items items, EncWs ws) {
  __shared__ uint32_t off[kSegChunks + 1];  // exclusive offsets of the segment's chunks, then the total
  __shared__ uint32_t wsum[kPlaceThreads / 32];
  __shared__ uint32_t s_seg, s_base;
  const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
  if (ws.hdr->flags & SZ_FLAG_ITEMS) return;
  for (uint32_t i = blockIdx.y; i < items.count; i += gridDim.y) {
    const sz_item& it = item_at(items, i);
    uint32_t flags = ws.item_flags[i];
    const uint64_t n = (flags & SZ_FLAG_SIZE) ? 0 : it.n;
    const uint32_t e = ws.item_esc[i];
    const Layout l = layout_of(n, e);
    if (!flags && l.comp_bytes > it.capacity) flags |= SZ_FLAG_CAPACITY;
    if (blockIdx.x == 0) {
      if (!flags && tid < 12) {
        // pad bytes: pk -> sm, sm -> chunk_id, local_pos -> esc_val (each < 4 bytes)
        uint8_t* p = it.payload;
        if (tid < 4 && l.n_pairs + tid < l.off_sm) p[l.n_pairs + tid] = 0;
        if (tid >= 4 && tid < 8 && l.off_sm + n + (tid - 4) < l.off_cid) p[l.off_sm + n + (tid - 4)] = 0;
        if (tid >= 8 && l.off_lpos + 2ull * e + (tid - 8) < l.off_ev) p[l.off_lpos + 2ull * e + (tid - 8)] = 0;
      }
      if (tid == 0) {
        if (flags) set_flag(ws.hdr, flags);
        if (it.meta != nullptr && (reinterpret_cast<uintptr_t>(it.meta) & 15) == 0) {
          sz_meta m;
          m.n = n;
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
    if (flags) continue;
    const uint64_t chunks = (n + kChunk - 1) / kChunk;
    const uint64_t segs = (chunks + kSegChunks - 1) / kSegChunks;
    const uint64_t chunk_base = it.tile_begin * kChunksPerTile;
    uint8_t* const cid_p = it.payload + l.off_cid;
    uint8_t* const lpos_p = it.payload + l.off_lpos;
    uint8_t* const ev_p = it.payload + l.off_ev;
    for (;;) {
      __syncthreads();  // the previous segment's s_seg / off are no longer read
      if (tid == 0) s_seg = atomicAdd(ws.seg_ticket + i, 1u);
      __syncthreads();
      const uint64_t seg = s_seg;
      if (seg >= segs) break;
      // block exclusive scan of the segment's chunk counts
      const uint64_t c = seg * kSegChunks + tid;
      const uint32_t cnt = (c < chunks) ? ws.chunk_cnt[chunk_base + c] : 0u;
      uint32_t incl = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, incl, d);
        if (lane >= uint32_t(d)) incl += o;
      }
      if (lane == 31) wsum[warp] = incl;
      __syncthreads();
      uint32_t wbase = 0;
      for (uint32_t w = 0; w < warp; ++w) wbase += wsum[w];
      off[tid] = wbase + incl - cnt;
      if (tid == kPlaceThreads - 1) off[kSegChunks] = wbase + incl;
      __syncthreads();
      const uint32_t agg = off[kSegChunks];
      if (warp == 0) {
        unsigned long long* st = ws.status + it.tile_begin + seg * kSegTiles;
        uint32_t base = 0;
        if (seg == 0) {
          if (lane == 0) st_relaxed_u64(st, kIncl | agg);
        } else {
          if (lane == 0) st_relaxed_u64(st, kAgg | agg);
          bool timed_out = false;
          base = segment_lookback(ws.status, it.tile_begin, int64_t(seg) - 1, &timed_out);
          if (lane == 0) {
            if (timed_out) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
            st_relaxed_u64(st, kIncl | (base + agg));
          }
        }
        if (lane == 0) s_base = base;
      }
      __syncthreads();
      const uint32_t base = s_base;
      // scatter: escape j of the segment -> global index base + j
      for (uint32_t j = tid; j < agg; j += kPlaceThreads) {
        uint32_t lo = 0, hi = kSegChunks;  // last chunk q with off[q] <= j
        while (hi - lo > 1) {
          const uint32_t mid = (lo + hi) >> 1;
          if (off[mid] <= j) lo = mid; else hi = mid;
        }
        const uint32_t k = j - off[lo];
        const uint64_t slot = (chunk_base + seg * kSegChunks + lo) * kChunk + k;
        const uint64_t gidx = uint64_t(base) + j;
        if (gidx < e) {
          *reinterpret_cast<uint32_t*>(cid_p + 4 * gidx) = uint32_t(seg * kSegChunks + lo);
          *reinterpret_cast<uint16_t*>(lpos_p + 2 * gidx) = ws.lpos[slot] & uint16_t(kChunk - 1);
          ev_p[gidx] = ws.ev[slot];
        }
      }
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
    // blockIdx.y = tensor; x covers the average tensor's segments
    const uint64_t per_item = items.count ? (items.total_tiles + items.count - 1) / items.count : 0;
    uint64_t gx = (per_item + kSegTiles - 1) / kSegTiles;
    if (gx < 1) gx = 1;
    if (gx > 1024) gx = 1024;
    const unsigned gy = items.count < 65535u ? items.count : 65535u;
    enc_place<<<dim3(unsigned(gx), gy), kPlaceThreads, 0, stream>>>(items, ws);
    err = cudaGetLastError();
  }
  return err;
}

}  // namespace sz
