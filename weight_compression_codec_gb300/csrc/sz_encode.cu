// Encode ("splitzip_codec.py" encode_torch + assemble_payload): one streaming
// pass over the input, then the in-order placement of the escape stream.
//
// Launches per call (after a 256-byte header memset):
//   enc_prepare  validates the item table, zeroes per-tensor escape totals,
//                segment tickets and segment status words, and (tables of
//                more than 256 tensors) writes the tile -> tensor map;
//   enc_main     persistent CTAs take runs of 4 tiles (8192 elements each)
//                from a device-wide ticket.  A producer warp streams each
//                tile (and the tensor's enc_lut) into a 4-stage shared-memory
//                ring with TMA bulk copies; 8 chunk warps -- warp w owns chunk
//                w (1024 elements) -- split and pack with coalesced pk/sm
//                stores, and compact the chunk's escapes with ballot/popc in
//                element order into the chunk's staging slot.  The chunk
//                counts and each tensor's escape total are recorded.  No warp
//                ever waits on another CTA.
//   enc_place    writes each tensor's pads and meta and gives every escape its
//                global index: tensors of at most 256 chunks by one warp (a
//                warp scan of the chunk counts), larger ones by segments of
//                256 chunks claimed by ticket (so segments start in order), a
//                block scan of the chunk counts and a decoupled lookback
//                across the tensor's segments.  chunk_id, local_pos and
//                esc_val are then written once, in order, at their final
//                offsets (the tensor's total is already known, so every
//                offset is).
// Every wait is bounded (kWaitTimeoutNs); on timeout SZ_FLAG_TIMEOUT is raised.
#include "sz_chunk.cuh"
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

// What the producer needs of an item.  When a ticket's run of tiles leaves
// the current item, the producer's lanes resolve the run's tiles in parallel
// (tile -> item map or table search, then the item) into shared memory.
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
  EncStage st[kEncStages];
  ItemLite run_item[kRun];
  uint32_t run_idx[kRun];
  uint64_t full[kEncStages];
  uint64_t empty[kEncStages];
};

__global__ void enc_prepare(const __grid_constant__ Items items, EncWs ws) {
  pdl_trigger();
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
    if (ws.small && it.n > kSmallMax) atomicOr(&ws.hdr->large, 1u);
    if (bad) set_flag(ws.hdr, bad);
    // the coverage gate: a tensor below it is left uncompressed (not an error)
    else if (ws.gate >= 0.0 && it.codebook->coverage < ws.gate) bad = SZ_META_GATED;
    ws.item_flags[i] = bad;
    ws.item_esc[i] = 0;
    ws.seg_ticket[i] = 0;
  }
  if (ws.report != nullptr && gtid == 0) *ws.report = sz_gate_report{};
  if (ws.tile_item != nullptr) {
    // one warp per item writes the item's tile -> item map entries (clipped to the table's tiles)
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t nwarps = nthreads / 32;
    for (uint64_t i = gtid / 32; i < items.count; i += nwarps) {
      const sz_item& it = item_at(items, uint32_t(i));
      const uint64_t tb = it.tile_begin;
      const uint64_t te = (it.n > SZ_MAX_ELEMS) ? tb : tb + tiles_of(it.n);
      for (uint64_t t = tb + lane; t < te && t < items.total_tiles; t += 32) ws.tile_item[t] = uint32_t(i);
    }
  }
}

__global__ void __launch_bounds__(kEncThreads, kEncCtasPerSm)
    enc_main(const __grid_constant__ Items items, EncWs ws) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  EncShared& sh = *reinterpret_cast<EncShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  pdl_trigger();
  pdl_wait();  // enc_prepare's writes
  // an inconsistent item table (flagged by enc_prepare) is never walked; a
  // table of small tensors is encoded by small_main
  if ((ws.hdr->flags & SZ_FLAG_ITEMS) || (ws.small && !ws.hdr->large)) return;

  const uint64_t T = items.total_tiles;

  if (tid == 0) {
    for (int s = 0; s < kEncStages; ++s) {
      mbar_init(&sh.full[s], 1 + 32);
      mbar_init(&sh.empty[s], kEncChunkWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    // Tiles are handed out in runs of kRun from a device-wide ticket, so CTAs
    // that run faster (SM placement, neighbours) take more of them.
    unsigned long long run_base = 0;
    uint32_t run_pos = kRun;
    uint32_t cur = 0xFFFFFFFFu;
    ItemLite itm{};
    bool run_in_cur = false;
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
        // a run inside the current item needs no lookup
        run_in_cur = cur != 0xFFFFFFFFu && run_base >= itm.tile_begin &&
                     run_base + kRun <= itm.tile_begin + tiles_of(itm.n);
        if (!run_in_cur) {
          if (lane < kRun && run_base + lane < T) {
            const uint64_t tt = run_base + lane;
            uint32_t idx = ws.tile_item ? ws.tile_item[tt] : find_item(items, tt);
            if (idx >= items.count) idx = 0;  // never for a validated table; the range check below rejects it
            sh.run_idx[lane] = idx;
            sh.run_item[lane] = item_lite(items, ws, idx);
          }
          __syncwarp();
        }
      }
      const uint64_t t = run_base + run_pos;
      EncStage& st = sh.st[s];
      if (t >= T) {
        if (lane == 0) {
          st.flags = kStageEnd;
          mbar_arrive(&sh.full[s]);
        }
        cp_async_mbar_arrive_noinc(&sh.full[s]);
        return;
      }
      if (!run_in_cur) {
        cur = sh.run_idx[run_pos];
        itm = sh.run_item[run_pos];
      }
      ++run_pos;
      const bool in_item = t >= itm.tile_begin && t - itm.tile_begin < tiles_of(itm.n);
      const uint32_t lt = in_item ? uint32_t(t - itm.tile_begin) : 0u;
      const uint64_t g = uint64_t(lt) * kTile;
      const bool invalid = itm.flags != 0 || !in_item;
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
  bool dense = false;  // this warp staged no escapes of some chunk (enc_regen will write them)
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
      uint32_t* slot = ws.stage + chunk * kChunk;
      const uint32_t run = (st.n_tile == kTile)
                               ? encode_chunk8(st, uint32_t(warp), uint32_t(lane), slot)
                               : encode_chunk<false>(st, uint32_t(warp), uint32_t(lane), slot);
      if (st.item != acc_item) {
        if (lane == 0 && acc) atomicAdd(ws.item_esc + acc_item, acc);
        acc_item = st.item;
        acc = 0;
      }
      acc += run;
      dense |= run > kStageMax;
      if (lane == 0) ws.chunk_cnt[chunk] = uint16_t(run);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
  }
  if (lane == 0 && acc) atomicAdd(ws.item_esc + acc_item, acc);
  if (lane == 0 && dense) atomicOr(&ws.hdr->dense, 1u);
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
constexpr uint32_t kPlaceWarps = kPlaceThreads / 32;
constexpr uint64_t kSmallElems = uint64_t(kSegChunks) * kChunk;  // one segment: placed by one warp
constexpr uint32_t kScatterUnroll = 8;  // escapes per thread per scatter round
constexpr int kPlaceBlocksPerSm = 4;

// Writes the escapes of chunk `c` (cnt of them, the first at global index
// o) from its staging slot.  Threads r = 0..stride-1 of the caller.
__device__ __forceinline__ void scatter_chunk(const EncWs& ws, uint8_t* cid_p, uint8_t* lpos_p, uint8_t* ev_p,
                                              uint64_t slot0, uint32_t c, uint32_t o, uint32_t cnt, uint32_t e,
                                              uint32_t r, uint32_t stride) {
  for (uint32_t k = r; k < cnt; k += stride) {
    const uint64_t gidx = uint64_t(o) + k;
    if (gidx >= e) break;
    *reinterpret_cast<uint32_t*>(cid_p + 4 * gidx) = c;
    const uint32_t v = ws.stage[slot0 + k];
    *reinterpret_cast<uint16_t*>(lpos_p + 2 * gidx) = uint16_t(v & (kChunk - 1));
    ev_p[gidx] = uint8_t(v >> 16);
  }
}

// Whole placement of an item of at most one segment by one warp: warp scan
// of its chunk counts (lane l owns chunks 8l .. 8l+7), then the chunks'
// escapes in order, each chunk's written by the 32 lanes together.
__device__ void place_small(const Items& items, const EncWs& ws, uint32_t i, uint32_t lane, uint32_t* off) {
  const sz_item& it = item_at(items, i);
  uint32_t flags = ws.item_flags[i];
  const uint64_t n = (flags & SZ_FLAG_SIZE) ? 0 : it.n;
  const uint32_t e = ws.item_esc[i];
  const Layout l = layout_of(n, e);
  if (!flags && l.comp_bytes > it.capacity) flags |= SZ_FLAG_CAPACITY;
  finish_item(ws, it, l, n, e, flags, lane);
  if (flags) return;
  const uint32_t chunks = uint32_t((n + kChunk - 1) / kChunk);
  const uint64_t chunk_base = it.tile_begin * kChunksPerTile;
  uint32_t c8[8], sum = 0;
#pragma unroll
  for (uint32_t j = 0; j < 8; ++j) {
    const uint32_t c = lane * 8 + j;
    c8[j] = c < chunks ? ws.chunk_cnt[chunk_base + c] : 0u;
    sum += c8[j];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t v = __shfl_up_sync(FULL, incl, d);
    if (lane >= uint32_t(d)) incl += v;
  }
  uint32_t run = incl - sum;
#pragma unroll
  for (uint32_t j = 0; j < 8; ++j) {
    off[lane * 8 + j] = run;
    run += c8[j];
  }
  if (lane == 31) off[kSegChunks] = run;
  __syncwarp();
  uint8_t* const cid_p = it.payload + l.off_cid;
  uint8_t* const lpos_p = it.payload + l.off_lpos;
  uint8_t* const ev_p = it.payload + l.off_ev;
  for (uint32_t c = 0; c < chunks; ++c) {
    const uint32_t o = off[c], cnt = off[c + 1] - o;
    if (cnt > kStageMax) {
      if (lane == 0) ws.stage[(chunk_base + c) * kChunk] = o;  // for enc_regen
    } else if (cnt) {
      scatter_chunk(ws, cid_p, lpos_p, ev_p, (chunk_base + c) * kChunk, c, o, cnt, e, lane, 32);
    }
  }
  __syncwarp();  // off is reused by this warp's next item
}

// Rows of the grid (blockIdx.y) take groups of kPlaceWarps consecutive items.
// Items of at most one segment are placed by one warp of the row's first
// block; larger ones by the row's blocks dealt round-robin over them: segments
// of 256 chunks claimed by ticket (so they start in order), a block scan of
// the chunk counts and a decoupled lookback across the item's segments.
__global__ void __launch_bounds__(kPlaceThreads, kPlaceBlocksPerSm) enc_place(const __grid_constant__ Items items, EncWs ws) {
  __shared__ uint32_t off[kSegChunks + 1];   // exclusive offsets of the segment's chunks, then the total
  __shared__ uint32_t offs[kSegChunks + 1];  // the same over the staged chunks (count <= kStageMax)
  __shared__ uint32_t woff[kPlaceWarps][kSegChunks + 1];
  __shared__ uint64_t wsum[kPlaceThreads / 32];
  __shared__ uint32_t s_seg, s_base;
  const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();  // the encode pass's counts and staging
  if ((ws.hdr->flags & SZ_FLAG_ITEMS) || (ws.small && !ws.hdr->large)) return;
  const uint32_t groups = (items.count + kPlaceWarps - 1) / kPlaceWarps;
  for (uint32_t grp = blockIdx.y; grp < groups; grp += gridDim.y) {
    {
      const uint32_t i = grp * kPlaceWarps + warp;
      if (blockIdx.x == 0 && i < items.count) {
        const uint64_t n = item_at(items, i).n;
        if (n <= kSmallElems || (ws.item_flags[i] & SZ_FLAG_SIZE)) place_small(items, ws, i, lane, woff[warp]);
      }
    }
    // larger items: the row's blocks are dealt round-robin over its items
    const uint32_t in_row = min(kPlaceWarps, items.count - grp * kPlaceWarps);
    const uint32_t R = min(in_row, gridDim.x);
    const uint32_t rank = blockIdx.x / R;
    for (uint32_t q = blockIdx.x % R; q < in_row; q += R) {
      const uint32_t i = grp * kPlaceWarps + q;
      const sz_item& it = item_at(items, i);
      uint32_t flags = ws.item_flags[i];
      if (it.n <= kSmallElems || (flags & SZ_FLAG_SIZE)) continue;
      const uint64_t n = it.n;
      const uint32_t e = ws.item_esc[i];
      const Layout l = layout_of(n, e);
      if (!flags && l.comp_bytes > it.capacity) flags |= SZ_FLAG_CAPACITY;
      if (rank == 0) finish_item(ws, it, l, n, e, flags, tid);
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
        // block exclusive scan of the segment's chunk counts, and of those
        // of its staged chunks (both in one 64-bit word: staged << 32 | all)
        const uint64_t c = seg * kSegChunks + tid;
        const uint32_t cnt = (c < chunks) ? ws.chunk_cnt[chunk_base + c] : 0u;
        const uint64_t pair = (uint64_t(cnt <= kStageMax ? cnt : 0u) << 32) | cnt;
        uint64_t incl = pair;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint64_t o = __shfl_up_sync(FULL, incl, d);
          if (lane >= uint32_t(d)) incl += o;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        uint64_t wbase = 0;
        for (uint32_t w = 0; w < warp; ++w) wbase += wsum[w];
        off[tid] = uint32_t(wbase + incl - pair);
        offs[tid] = uint32_t((wbase + incl - pair) >> 32);
        if (tid == kPlaceThreads - 1) {
          off[kSegChunks] = uint32_t(wbase + incl);
          offs[kSegChunks] = uint32_t((wbase + incl) >> 32);
        }
        __syncthreads();
        const uint32_t agg = off[kSegChunks];
        const uint32_t agg_staged = offs[kSegChunks];
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
        // scatter of the staged chunks: staged escape j of the segment (in
        // chunk lo) -> global index base + off[lo] + (j - offs[lo]).  Each
        // thread takes kScatterUnroll escapes per round and issues all their
        // staging loads before any store, so a round costs one memory latency.
        for (uint32_t j0 = 0; j0 < agg_staged; j0 += kScatterUnroll * kPlaceThreads) {
          uint32_t q[kScatterUnroll], jj[kScatterUnroll], sv[kScatterUnroll];
#pragma unroll
          for (uint32_t u = 0; u < kScatterUnroll; ++u) {
            const uint32_t j = j0 + u * kPlaceThreads + tid;
            uint32_t lo = 0;  // last chunk lo with offs[lo] <= j (offs[kSegChunks] = agg_staged > j)
#pragma unroll
            for (uint32_t b = kSegChunks / 2; b >= 1; b >>= 1)
              if (offs[lo + b] <= j) lo += b;
            q[u] = lo;
            jj[u] = off[lo] + (j - offs[lo]);  // the escape's index in the segment
            if (j < agg_staged) {
              const uint64_t slot = (chunk_base + seg * kSegChunks + lo) * kChunk + (j - offs[lo]);
              sv[u] = ws.stage[slot];
            } else {
              jj[u] = agg;
            }
          }
#pragma unroll
          for (uint32_t u = 0; u < kScatterUnroll; ++u) {
            const uint64_t gidx = uint64_t(base) + jj[u];
            if (jj[u] < agg && gidx < e) {
              *reinterpret_cast<uint32_t*>(cid_p + 4 * gidx) = uint32_t(seg * kSegChunks + q[u]);
              *reinterpret_cast<uint16_t*>(lpos_p + 2 * gidx) = uint16_t(sv[u] & (kChunk - 1));
              ev_p[gidx] = uint8_t(sv[u] >> 16);
            }
          }
        }
        // chunks too dense to stage: their escapes' first global index, in
        // their (unused) staging slot, for enc_regen
        if (c < chunks && cnt > kStageMax) ws.stage[(chunk_base + c) * kChunk] = base + off[tid];
      }
    }
  }
}

constexpr int kRegenWarps = 8;

// The chunk a regeneration warp works on: where its escapes go.
struct RegenChunk {
  const uint8_t* lut;                 // the tensor's enc_lut
  uint8_t *cid_p, *lpos_p, *ev_p;     // the tensor's escape streams
  const uint16_t* xc;                 // the chunk's input
  uint32_t c, nvalid, e, bulk, first; // tensor-local chunk, elements, escapes of the tensor,
                                      // bytes copied to shared memory, its first escape's index
  uint32_t cnt;                       // the chunk's escapes
};

// The escapes of every chunk too dense to stage (count > kStageMax),
// regenerated from the input after enc_place has given each such chunk the
// global index of its first escape (in the first word of its staging slot).
// Warps take the chunks of the whole table grid-stride, so the work spreads
// over every SM however few segments hold it.  Each warp double-buffers its
// chunks in shared memory: one lane issues the TMA bulk copy of the next
// chunk's 2 KiB before the warp processes the current one.  Per chunk: rows
// of 32 elements (lane l holds element 32 r + l), an escape being an element
// whose enc_lut code has bit 4 set (as in the chunk encoder), compacted in
// element order by one ballot per row, so a row's escapes are written next to
// each other.  Items with a flag (failed, gated, over capacity) are skipped,
// as enc_place skips them.  Returns at once when enc_main found no dense
// chunk.
__global__ void __launch_bounds__(kRegenWarps * 32) enc_regen(const __grid_constant__ Items items, EncWs ws) {
  __shared__ __align__(128) uint16_t buf[kRegenWarps][2][kChunk];
  __shared__ __align__(16) uint8_t lut_sh[kRegenWarps][256];  // the current chunk's enc_lut
  __shared__ __align__(16) uint16_t lp_sh[kRegenWarps][kChunk + 8];  // a whole chunk's local_pos ...
  __shared__ __align__(16) uint8_t ev_sh[kRegenWarps][kChunk + 16];  // ... and esc_val, then copied out
  __shared__ uint64_t bar[kRegenWarps][2];
  pdl_wait();  // enc_place's offsets
  if (ws.hdr->dense == 0 || (ws.hdr->flags & SZ_FLAG_ITEMS) || (ws.small && !ws.hdr->large)) return;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t lane_lt = (1u << lane) - 1u;
  const uint64_t total = items.total_tiles * kChunksPerTile;
  const uint64_t stride = uint64_t(gridDim.x) * kRegenWarps;
  if (lane == 0) {
    mbar_init(&bar[warp][0], 1);
    mbar_init(&bar[warp][1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  // the item of the last chunk looked up: global chunks [cb0, cb1)
  uint64_t cb0 = 1, cb1 = 0, item_n = 0;
  RegenChunk item{};
  bool item_ok = false;
  // next dense chunk of this warp at or after g, with its item; total if none
  auto next = [&](uint64_t g, RegenChunk& rc) -> uint64_t {
    for (; g < total; g += stride) {
      if (ws.chunk_cnt[g] <= kStageMax) continue;
      if (g < cb0 || g >= cb1) {
        const uint64_t tile = g / kChunksPerTile;
        uint32_t idx = ws.tile_item ? ws.tile_item[tile] : find_item(items, tile);
        if (idx >= items.count) idx = 0;
        const sz_item& it = item_at(items, idx);
        const uint32_t flags = ws.item_flags[idx];
        const uint64_t n = (flags & SZ_FLAG_SIZE) ? 0 : it.n;
        const uint32_t e = ws.item_esc[idx];
        const Layout l = layout_of(n, e);
        cb0 = it.tile_begin * kChunksPerTile;
        cb1 = cb0 + (n + kChunk - 1) / kChunk;
        item_ok = flags == 0 && l.comp_bytes <= it.capacity;
        item.lut = item_ok ? it.codebook->enc_lut : nullptr;
        item.cid_p = it.payload + l.off_cid;
        item.lpos_p = it.payload + l.off_lpos;
        item.ev_p = it.payload + l.off_ev;
        item.xc = it.x;
        item.e = e;
        item_n = n;
      }
      if (!item_ok || g < cb0 || g >= cb1) {
        cb0 = 1;
        cb1 = 0;
        continue;
      }
      rc = item;
      rc.c = uint32_t(g - cb0);
      const uint64_t first = uint64_t(rc.c) * kChunk;
      rc.nvalid = (item_n - first < kChunk) ? uint32_t(item_n - first) : kChunk;
      rc.xc = item.xc + first;
      rc.bulk = (2u * rc.nvalid) & ~15u;
      rc.first = ws.stage[g * kChunk];
      rc.cnt = ws.chunk_cnt[g];
      return g;
    }
    return total;
  };
  RegenChunk cur{}, nxt{};
  const uint8_t* lut_src = nullptr;  // the enc_lut now in lut_sh[warp]
  uint64_t g = next(uint64_t(blockIdx.x) * kRegenWarps + warp, cur);
  auto issue = [&](const RegenChunk& rc, int b) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[warp][b], rc.bulk);
      if (rc.bulk) bulk_g2s(buf[warp][b], rc.xc, rc.bulk, &bar[warp][b]);
    }
  };
  if (g < total) issue(cur, 0);
  uint32_t phases = 0;  // bit b: parity of buffer b's next phase
  for (int b = 0; g < total; b ^= 1) {
    const uint64_t gn = next(g + stride, nxt);
    if (gn < total) issue(nxt, b ^ 1);
    if (!__all_sync(FULL, mbar_wait(&bar[warp][b], (phases >> b) & 1u))) {
      if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      if (gn < total) (void)__all_sync(FULL, mbar_wait(&bar[warp][b ^ 1], (phases >> (b ^ 1)) & 1u));  // in flight
      return;
    }
    phases ^= 1u << b;
    if (cur.lut != lut_src) {  // the tensor changed: its enc_lut into shared memory
      __syncwarp();
      reinterpret_cast<uint2*>(lut_sh[warp])[lane] = __ldg(reinterpret_cast<const uint2*>(cur.lut) + lane);
      lut_src = cur.lut;
      __syncwarp();
    }
    const uint8_t* lut = lut_sh[warp];
    const uint16_t* xs = buf[warp][b];
    // the chunk's escape streams from its first escape; `room`: escapes before the tensor's end
    uint32_t* const cid_c = reinterpret_cast<uint32_t*>(cur.cid_p) + cur.first;
    uint16_t* const lp_c = reinterpret_cast<uint16_t*>(cur.lpos_p) + cur.first;
    uint8_t* const ev_c = cur.ev_p + cur.first;
    const uint32_t room = cur.e > cur.first ? cur.e - cur.first : 0u;
    uint32_t run = 0;
    if (cur.bulk == 2u * kChunk) {
      // A whole chunk in shared memory.  Its escapes' chunk_id entries are
      // all c: written as a run (16-byte stores for its aligned body).
      const uint32_t m = cur.cnt < room ? cur.cnt : room;
      const uint32_t head = uint32_t((16u - (reinterpret_cast<uintptr_t>(cid_c) & 15u)) & 15u) / 4u;
      const uint32_t h = head < m ? head : m;
      if (lane < h) cid_c[lane] = cur.c;
      const uint32_t body4 = (m - h) / 4u;
      uint4* const cid4 = reinterpret_cast<uint4*>(cid_c + h);
      for (uint32_t k = lane; k < body4; k += 32) cid4[k] = make_uint4(cur.c, cur.c, cur.c, cur.c);
      for (uint32_t k = h + 4u * body4 + lane; k < m; k += 32) cid_c[k] = cur.c;
      // local_pos and esc_val: lane l takes elements 4 l .. 4 l + 3 of each
      // row of 128; four ballots give every lane the escapes before its
      // own.  They are collected in shared memory, at the same offset mod 16
      // as their destination, then copied out with 16-byte stores.
      const uint32_t lp_sh0 = uint32_t(reinterpret_cast<uintptr_t>(lp_c) & 15u) / 2u;  // elements
      const uint32_t ev_sh0 = uint32_t(reinterpret_cast<uintptr_t>(ev_c) & 15u);
      uint16_t* const lps = lp_sh[warp] + lp_sh0;
      uint8_t* const evs = ev_sh[warp] + ev_sh0;
      const uint2* const xs2 = reinterpret_cast<const uint2*>(xs);
#pragma unroll 2
      for (uint32_t r = 0; r < kChunk / 128; ++r) {
        const uint2 w = xs2[r * 32u + lane];
        const uint32_t e0 = (w.x >> 7) & 0xFFu, e1 = (w.x >> 23) & 0xFFu;
        const uint32_t e2 = (w.y >> 7) & 0xFFu, e3 = (w.y >> 23) & 0xFFu;
        const uint32_t f = ((lut[e0] >> 4) & 1u) | ((lut[e1] >> 3) & 2u) | ((lut[e2] >> 2) & 4u) | ((lut[e3] >> 1) & 8u);
        const uint32_t c4 = __popc(f);
        const uint32_t b1 = __ballot_sync(FULL, c4 >= 1u), b2 = __ballot_sync(FULL, c4 >= 2u);
        const uint32_t b3 = __ballot_sync(FULL, c4 >= 3u), b4 = __ballot_sync(FULL, c4 == 4u);
        uint32_t q = run + __popc(b1 & lane_lt) + __popc(b2 & lane_lt) + __popc(b3 & lane_lt) + __popc(b4 & lane_lt);
        const uint32_t p0 = r * 128u + 4u * lane;
        const uint32_t ex4 = e0 | (e1 << 8) | (e2 << 16) | (e3 << 24);
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k) {
          if ((f >> k) & 1u) {
            lps[q] = uint16_t(p0 + k);
            evs[q] = uint8_t(ex4 >> (8 * k));
            ++q;
          }
        }
        run += __popc(b1) + __popc(b2) + __popc(b3) + __popc(b4);
      }
      __syncwarp();
      // copy out: [0, m) at lp_c / ev_c, whole 16-byte words where both sides allow
      {
        const uint32_t lh = (lp_sh0 ? 8u - lp_sh0 : 0u) < m ? (lp_sh0 ? 8u - lp_sh0 : 0u) : m;
        if (lane < lh) lp_c[lane] = lps[lane];
        const uint32_t lb = (m - lh) / 8u;
        const uint4* const ls4 = reinterpret_cast<const uint4*>(lps + lh);
        uint4* const ld4 = reinterpret_cast<uint4*>(lp_c + lh);
        for (uint32_t k = lane; k < lb; k += 32) ld4[k] = ls4[k];
        for (uint32_t k = lh + 8u * lb + lane; k < m; k += 32) lp_c[k] = lps[k];
        const uint32_t eh = (ev_sh0 ? 16u - ev_sh0 : 0u) < m ? (ev_sh0 ? 16u - ev_sh0 : 0u) : m;
        if (lane < eh) ev_c[lane] = evs[lane];
        const uint32_t eb = (m - eh) / 16u;
        const uint4* const es4 = reinterpret_cast<const uint4*>(evs + eh);
        uint4* const ed4 = reinterpret_cast<uint4*>(ev_c + eh);
        for (uint32_t k = lane; k < eb; k += 32) ed4[k] = es4[k];
        for (uint32_t k = eh + 16u * eb + lane; k < m; k += 32) ev_c[k] = evs[k];
      }
    } else {
      // a tensor's last chunk: elements past the copied body (under 8) are read directly
      for (uint32_t r = 0; r < kChunk / 32; ++r) {
        const uint32_t p = r * 32u + lane;
        const uint32_t v = 2u * p + 2u <= cur.bulk ? uint32_t(xs[p])
                                                   : (p < cur.nvalid ? uint32_t(__ldg(cur.xc + p)) : 0u);
        const uint32_t ex = (v >> 7) & 0xFFu;
        const bool esc = p < cur.nvalid && ((lut[ex] >> 4) & 1u);
        const uint32_t bal = __ballot_sync(FULL, esc);
        const uint32_t q = run + __popc(bal & lane_lt);
        if (esc && q < room) {
          cid_c[q] = cur.c;
          lp_c[q] = uint16_t(p);
          ev_c[q] = uint8_t(ex);
        }
        run += __popc(bal);
      }
    }
    __syncwarp();  // buf[b] is read before it is refilled
    g = gn;
    cur = nxt;
  }
}

}  // namespace

cudaError_t launch_encode(const Items& items, void* ws_base, cudaStream_t stream, const DeviceInfo& dev, double gate,
                          sz_gate_report* report) {
  EncWs ws = enc_ws(ws_base, items.count, items.total_tiles);
  ws.gate = gate;
  ws.report = report;
  ws.small = small_route(items);
  cudaError_t err = cudaMemsetAsync(ws_base, 0, sizeof(WsHeader), stream);
  if (err != cudaSuccess) return err;
  {
    // threads for the tiles, or a warp per item when the tile map is written per item
    uint64_t work = items.total_tiles > items.count ? items.total_tiles : items.count;
    if (enc_uses_tile_map(items.count) && uint64_t(items.count) * 32 > work)
      work = uint64_t(items.count) * 32;
    const uint64_t blocks = (work + 255) / 256;
    const unsigned grid = unsigned(blocks < 2048 ? (blocks ? blocks : 1) : 2048);
    enc_prepare<<<grid, 256, 0, stream>>>(items, ws);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  // tables of small tensors: whole tensors in shared memory, one CTA per SM
  // (the general kernels below then return at once, unless a tensor is too large)
  TimingHook hook = g_timing;
  if (ws.small) {
    if ((err = launch_small(items, ws, nullptr, stream, dev)) != cudaSuccess) return err;
    g_timing = TimingHook{nullptr, nullptr};
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
    err = launch_pdl(enc_main, dim3(grid), dim3(kEncThreads), smem, stream, items, ws);
    if (g_timing.after) cudaEventRecord(g_timing.after, stream);
    if (err != cudaSuccess) {
      g_timing = hook;
      return err;
    }
  }
  err = launch_place(items, ws, stream, dev);
  g_timing = hook;
  return err;
}

cudaError_t launch_place(const Items& items, const EncWs& ws, cudaStream_t stream, const DeviceInfo& dev) {
  cudaError_t err;
  {
    // blockIdx.y = group of kPlaceWarps tensors; x covers the average tensor's
    // segments times the tensors a row takes in turn (1 when tensors are of
    // one segment or less: their warps need no other block)
    const uint64_t per_item = items.count ? (items.total_tiles + items.count - 1) / items.count : 0;
    const uint64_t seg_per_item = (per_item + kSegTiles - 1) / kSegTiles;
    const uint64_t per_row = items.count < kPlaceWarps ? items.count : kPlaceWarps;
    uint64_t gx = seg_per_item <= 1 ? 1 : seg_per_item * per_row;
    if (gx > 1024) gx = 1024;
    const uint64_t groups = (uint64_t(items.count) + kPlaceWarps - 1) / kPlaceWarps;
    const unsigned gy = unsigned(groups < 65535u ? (groups ? groups : 1) : 65535u);
    // blocks take segments by ticket: about two waves of resident blocks suffice
    const uint64_t cap = 2ull * kPlaceBlocksPerSm * uint64_t(dev.num_sms) / gy;
    if (gx > cap) gx = cap > 0 ? cap : 1;
    err = launch_pdl(enc_place, dim3(unsigned(gx), gy), dim3(kPlaceThreads), 0, stream, items, ws);
    if (err != cudaSuccess) return err;
  }
  if (items.total_tiles > 0) {
    // chunks too dense to stage (returns at once when there are none)
    const uint64_t chunks = items.total_tiles * kChunksPerTile;
    const uint64_t blocks = (chunks + kRegenWarps - 1) / kRegenWarps;
    const uint64_t cap = uint64_t(dev.num_sms) * 8;
    err = launch_pdl(enc_regen, dim3(unsigned(blocks < cap ? blocks : cap)), dim3(kRegenWarps * 32), 0, stream,
                     items, ws);
  }
  return err;
}

}  // namespace sz
