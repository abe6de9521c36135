// Calibration and encode in one call ("splitzip_codec.py"
// calibrate_codebook followed by encode_torch + assemble_payload, for many
// tensors).  The results are those of sz_calibrate_many followed by
// sz_encode_many, byte for byte; only the order of the work differs.
//
// The separate calls read every input twice from HBM: once to count its
// exponents, once to split and pack it with the codebook the counts give.
// Here the tensors are taken in groups of about kGroupTiles tiles (32 MiB of
// BF16) and one persistent kernel works through
//     count(g0), count(g1), count(g2), encode(g0), count(g3), encode(g1), ...
// every CTA counting its own slice of each group and then taking runs of the
// group's tiles to encode from a ticket, so a group's input is read again
// soon after it was counted (two other groups' count passes lie in between).
// On a GB300 the traffic in between is larger than L2 and the second read
// comes from HBM; the gain over the separate calls is the launches saved.
//
// Launches per call (after a 256-byte header memset):
//   ce_prepare  validates the table for both passes, zeroes histograms,
//               completion counters, ready flags, escape totals, tickets and
//               segment words, writes the codebook of empty tensors, the first
//               tile of every group and the tile -> tensor map;
//   ce_main     cooperative (all CTAs resident: an encode tile waits for its
//               tensor's codebook, which other CTAs' count passes produce).
//               Per CTA: a producer warp streams the tiles of each job through
//               a 4-stage TMA ring, resolving 32 tiles at a time (one per
//               lane) through the map; 8 consumer warps either count a tile
//               (the calibration counters) or split and pack it (a chunk per
//               warp, escapes to the staging slots); a select warp ranks each
//               tensor whose counts are complete and publishes its codebook.
//               A count job's counts are flushed when it ends, before any
//               wait, and a tensor lies in one group only, so every wait ends.
//   enc_place   as for sz_encode_many.
// Every wait is bounded (kWaitTimeoutNs); on timeout SZ_FLAG_TIMEOUT is raised.
#include "sz_chunk.cuh"
#include "sz_count.cuh"
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kCeConsumerWarps = 8;
constexpr int kCeConsumers = kCeConsumerWarps * 32;  // 256: one thread per exponent bin
constexpr int kCeProducerWarp = kCeConsumerWarps;
constexpr int kCeSelectWarp = kCeConsumerWarps + 1;
constexpr int kCeThreads = kCeConsumers + 64;
constexpr int kCeStages = 4;
constexpr int kCeCtasPerSm = 2;
constexpr uint32_t kCeRun = 8;      // encode tiles per ticket
constexpr uint64_t kLookahead = 2;  // groups counted ahead of the group being encoded
// stage flags: kStageCount = a tile to count (else to encode); kStageJobEnd = the
// last stage of a count job (its counts are flushed after it)
constexpr uint32_t kStageEnd = 1u, kStageInvalid = 2u, kStageCount = 4u, kStageJobEnd = 8u;
constexpr uint32_t kSelectEnd = 0xFFFFFFFFu;
constexpr uint32_t kNoItem = 0xFFFFFFFFu;
constexpr unsigned FULL = 0xFFFFFFFFu;
static_assert(kCeConsumers == 256, "one consumer thread per exponent bin");

struct __align__(128) CeStage {
  uint16_t x[kTile];     // the tile's BF16 patterns
  uint8_t enc_lut[256];  // encode stages: the tensor's codebook enc_lut
  unsigned long long tile;
  uint8_t* payload;
  uint64_t off_sm;
  uint32_t lt, n_tile, flags, item;
};

struct CeShared {
  uint32_t cnt[256 * 32];  // [bin][lane] exponent counters
  CeStage st[kCeStages];
  uint64_t full[kCeStages];
  uint64_t empty[kCeStages];
  alignas(16) uint32_t h[2][256];  // histograms handed to the select warp
  uint32_t sel_item[2];
  uint64_t sel_full[2];
  uint64_t sel_empty[2];
  SelectScratch sel;
  uint64_t fbar;  // the consumer warps' own barrier (bounded waits) for flushes
  int s_last;
};

// First tile of group g: the start of the first tensor whose first tile is at
// or after g * kGroupTiles (total_tiles if none).
__device__ uint64_t group_first_tile(const Items& items, uint64_t g) {
  const uint64_t t = g * kGroupTiles;
  if (t >= items.total_tiles) return items.total_tiles;
  const sz_item& it = item_at(items, find_item(items, t));
  if (it.tile_begin >= t) return it.tile_begin;
  const uint64_t end = it.tile_begin + tiles_of(it.n);
  return end < items.total_tiles ? end : items.total_tiles;
}

__global__ void ce_prepare(const __grid_constant__ Items items, CeWs ws) {
  pdl_trigger();
  const uint64_t nthreads = uint64_t(gridDim.x) * blockDim.x;
  const uint64_t gtid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (uint64_t w = gtid; w < uint64_t(items.count) * 256; w += nthreads) ws.cal.hist[w] = 0;
  for (uint64_t t = gtid; t < items.total_tiles; t += nthreads) ws.enc.status[t] = 0ull;
  for (uint64_t i = gtid; i < items.count; i += nthreads) {
    const sz_item& it = item_at(items, uint32_t(i));
    uint32_t table = 0;
    if (items.table) {
      const uint64_t expect = (i == 0) ? 0 : items.table[i - 1].tile_begin + tiles_of(items.table[i - 1].n);
      if (it.tile_begin != expect) table |= SZ_FLAG_ITEMS;
      if (i + 1 == items.count && it.tile_begin + tiles_of(it.n) != items.total_tiles) table |= SZ_FLAG_ITEMS;
    }
    // what the count pass needs
    uint32_t cal_bad = table;
    if (it.n > SZ_MAX_ELEMS) cal_bad |= SZ_FLAG_SIZE;
    if (it.codebook == nullptr || (reinterpret_cast<uintptr_t>(it.codebook) & 15)) cal_bad |= SZ_FLAG_ALIGN;
    if (it.n > 0 && (it.x == nullptr || (reinterpret_cast<uintptr_t>(it.x) & 15))) cal_bad |= SZ_FLAG_ALIGN;
    // what the encode pass needs besides
    uint32_t enc_bad = cal_bad;
    if (it.meta == nullptr || (reinterpret_cast<uintptr_t>(it.meta) & 15)) enc_bad |= SZ_FLAG_ALIGN;
    if (it.n > 0 && (it.payload == nullptr || (reinterpret_cast<uintptr_t>(it.payload) & 15)))
      enc_bad |= SZ_FLAG_ALIGN;
    if (!(enc_bad & SZ_FLAG_SIZE) && layout_of(it.n, 0).off_cid > it.capacity) enc_bad |= SZ_FLAG_CAPACITY;
    ws.cal.done[i] = cal_bad ? kItemInvalid : 0u;
    ws.enc.item_flags[i] = enc_bad;
    if (ws.enc.small && it.n > kSmallMax) atomicOr(&ws.enc.hdr->large, 1u);
    ws.enc.item_esc[i] = 0;
    ws.enc.seg_ticket[i] = 0;
    ws.ready[i] = 0;
    if (enc_bad) set_flag(ws.cal.hdr, enc_bad);
    if (!cal_bad && it.n == 0) {
      write_empty_codebook(it.codebook);
      ws.ready[i] = 1;
    }
  }
  // first tile of every group (the table is searched only if consecutive; an
  // inconsistent one stops ce_main before it reads these)
  const uint64_t groups = ce_groups(items.total_tiles);
  for (uint64_t g = gtid; g <= groups; g += nthreads) {
    ws.group_first[g] = group_first_tile(items, g);
    ws.group_ticket[g] = 0;
  }
  // tile -> item map, one warp per item (clipped to the table's tiles)
  const uint32_t lane = threadIdx.x & 31u;
  for (uint64_t i = gtid / 32; i < items.count; i += nthreads / 32) {
    const sz_item& it = item_at(items, uint32_t(i));
    const uint64_t tb = it.tile_begin;
    const uint64_t te = (it.n > SZ_MAX_ELEMS) ? tb : tb + tiles_of(it.n);
    for (uint64_t t = tb + lane; t < te && t < items.total_tiles; t += 32) ws.enc.tile_item[t] = uint32_t(i);
  }
}


__global__ void __launch_bounds__(kCeThreads, kCeCtasPerSm) ce_main(const __grid_constant__ Items items, CeWs ws) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  CeShared& sh = *reinterpret_cast<CeShared*>(smem_raw);
  const uint32_t tid = threadIdx.x;
  const uint32_t warp = tid >> 5, lane = tid & 31u;
  // an inconsistent item table (flagged by ce_prepare) is never walked; a
  // table of small tensors is done by small_main
  if ((ws.cal.hdr->flags & SZ_FLAG_ITEMS) || (ws.enc.small && !ws.enc.hdr->large)) return;

  for (uint32_t w = tid; w < 256 * 32; w += kCeThreads) sh.cnt[w] = 0;
  if (tid == 0) {
    for (int s = 0; s < kCeStages; ++s) {
      mbar_init(&sh.full[s], 1 + 32);
      mbar_init(&sh.empty[s], kCeConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.sel_full[b], 1);
      mbar_init(&sh.sel_empty[b], 1);
    }
    mbar_init(&sh.fbar, kCeConsumerWarps);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCeProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    const uint64_t T = items.total_tiles;
    const uint64_t groups = ce_groups(T);
    uint32_t it = 0;  // stages handed out
    auto acquire = [&](int& s) -> bool {
      s = int(it % kCeStages);
      if (it >= uint32_t(kCeStages) && !__all_sync(FULL, mbar_wait(&sh.empty[s], ((it / kCeStages) - 1) & 1))) {
        if (lane == 0) set_flag(ws.cal.hdr, SZ_FLAG_TIMEOUT);
        return false;
      }
      return true;
    };
    auto shfl64 = [&](uint64_t v, uint32_t src) {
      return (uint64_t(__shfl_sync(FULL, uint32_t(v >> 32), src)) << 32) | __shfl_sync(FULL, uint32_t(v), src);
    };
    uint32_t ready_item = kNoItem;  // the last item whose codebook was seen published
    // Streams tiles [s0, s1) as a count job or an encode job.
    auto job = [&](uint64_t s0, uint64_t s1, bool count) -> bool {
      for (uint64_t w0 = s0; w0 < s1; w0 += 32) {
        // lane l resolves tile w0 + l
        const uint64_t mine = w0 + lane;
        bool ok = false;
        uint32_t idx = 0, nt = 0, lt = 0;
        const uint16_t* x = nullptr;
        uint8_t* payload = nullptr;
        const uint8_t* lut = nullptr;
        uint64_t off_sm = 0;
        if (mine < s1) {
          idx = ws.enc.tile_item[mine];
          if (idx < items.count) {
            const sz_item& itm = item_at(items, idx);
            const bool valid = count ? !(ws.cal.done[idx] & kItemInvalid) : ws.enc.item_flags[idx] == 0;
            const uint64_t tb = itm.tile_begin;
            if (valid && mine >= tb && mine - tb < tiles_of(itm.n)) {
              lt = uint32_t(mine - tb);
              const uint64_t g = uint64_t(lt) * kTile;
              nt = (itm.n - g < kTile) ? uint32_t(itm.n - g) : kTile;
              x = itm.x + g;
              payload = itm.payload;
              lut = itm.codebook->enc_lut;
              off_sm = layout_of(itm.n, 0).off_sm;
              ok = true;
            }
          }
        }
        const uint32_t nw = (s1 - w0 < 32) ? uint32_t(s1 - w0) : 32u;
        for (uint32_t k = 0; k < nw; ++k) {
          int s;
          if (!acquire(s)) return false;
          CeStage& st = sh.st[s];
          const bool last = count && (w0 + k + 1 == s1);
          const uint32_t jflags = (count ? kStageCount : 0u) | (last ? kStageJobEnd : 0u);
          const bool tok = __shfl_sync(FULL, ok, k);
          const uint32_t titem = __shfl_sync(FULL, idx, k);
          bool go = tok;
          if (go && !count && titem != ready_item) {
            // the tensor's codebook must be published before its tiles are encoded
            bool seen = false;
            if (lane == 0) {
              const uint64_t t0 = global_timer_ns();
              for (uint32_t spin = 0;; ++spin) {
                if (ld_acquire_u32(ws.ready + titem) != 0) {
                  seen = true;
                  break;
                }
                __nanosleep(256);
                if ((spin & 15) == 15 && global_timer_ns() - t0 > kWaitTimeoutNs) break;
              }
              if (!seen) set_flag(ws.cal.hdr, SZ_FLAG_TIMEOUT);
            }
            seen = __shfl_sync(FULL, seen, 0);
            if (seen) ready_item = titem;
            go = seen;
          }
          if (!go) {
            if (lane == 0) {
              st.flags = jflags | kStageInvalid;
              mbar_arrive(&sh.full[s]);
            }
            cp_async_mbar_arrive_noinc(&sh.full[s]);
            ++it;
            continue;
          }
          const uint32_t tnt = __shfl_sync(FULL, nt, k);
          const uint16_t* tx = reinterpret_cast<const uint16_t*>(shfl64(reinterpret_cast<uint64_t>(x), k));
          const uint32_t bulk = (tnt * 2u) & ~15u;
          const uint32_t tail = tnt * 2u - bulk;
          if (lane == 0) {
            st.item = titem;
            st.n_tile = tnt;
            st.flags = jflags;
            if (count) {
              mbar_arrive_expect_tx(&sh.full[s], bulk);
            } else {
              st.tile = w0 + k;
              mbar_arrive_expect_tx(&sh.full[s], bulk + 256u);
            }
          }
          if (!count) {
            const uint32_t tlt = __shfl_sync(FULL, lt, k);
            uint8_t* tpay = reinterpret_cast<uint8_t*>(shfl64(reinterpret_cast<uint64_t>(payload), k));
            const uint8_t* tlut = reinterpret_cast<const uint8_t*>(shfl64(reinterpret_cast<uint64_t>(lut), k));
            const uint64_t toff = shfl64(off_sm, k);
            if (lane == 0) {
              st.lt = tlt;
              st.payload = tpay;
              st.off_sm = toff;
              bulk_g2s(st.enc_lut, tlut, 256u, &sh.full[s]);
            }
          }
          if (lane == 0) {
            if (bulk) bulk_g2s(st.x, tx, bulk, &sh.full[s]);
          } else if (lane == 1 && tail) {
            cp_async16_zfill(reinterpret_cast<uint8_t*>(st.x) + bulk, reinterpret_cast<const uint8_t*>(tx) + bulk,
                             tail);
          }
          cp_async_mbar_arrive_noinc(&sh.full[s]);
          ++it;
        }
      }
      return true;
    };
    // The first non-empty group at or after g (groups if none): a tensor
    // larger than a group leaves the groups whose start it covers empty.
    auto next_group = [&](uint64_t g) -> uint64_t {
      while (g < groups && ws.group_first[g] == ws.group_first[g + 1]) ++g;
      return g;
    };
    // count(g0), count(g1), count(g2), encode(g0), count(g3), encode(g1), ...
    // over the non-empty groups: every CTA counts the same share of each
    // group, kLookahead groups ahead of the group it encodes, so codebooks
    // are ready when encoding starts
    uint64_t gc = next_group(0), ge = gc;
    for (uint64_t k = 0; gc < groups || ge < groups; ++k) {
      if (gc < groups) {
        const uint64_t a = ws.group_first[gc], z = ws.group_first[gc + 1];
        const uint64_t per = (z - a + gridDim.x - 1) / gridDim.x;
        const uint64_t s0 = min(z, a + uint64_t(blockIdx.x) * per), s1 = min(z, s0 + per);
        if (!job(s0, s1, true)) return;
        gc = next_group(gc + 1);
      }
      if (k >= kLookahead || gc >= groups) {
        // encode(ge): runs of kCeRun tiles from the group's ticket, so CTAs
        // that count faster encode more
        const uint64_t e = ge;
        ge = next_group(ge + 1);
        const uint64_t a = ws.group_first[e], z = ws.group_first[e + 1];
        for (;;) {
          uint32_t rb = 0;
          if (lane == 0) rb = atomicAdd(ws.group_ticket + e, kCeRun);
          rb = __shfl_sync(FULL, rb, 0);
          if (a + rb >= z) break;
          if (!job(a + rb, min(z, a + rb + kCeRun), false)) return;
        }
      }
    }
    int s;
    if (!acquire(s)) return;
    if (lane == 0) {
      sh.st[s].flags = kStageEnd;
      mbar_arrive(&sh.full[s]);
    }
    cp_async_mbar_arrive_noinc(&sh.full[s]);
    return;
  }

  if (warp == kCeSelectWarp) {
    // ---------------------------------------------------------------- select warp
    for (uint32_t k = 0;; ++k) {
      const uint32_t b = k & 1u;
      if (!__all_sync(FULL, mbar_wait(&sh.sel_full[b], (k >> 1) & 1u))) {
        if (lane == 0) set_flag(ws.cal.hdr, SZ_FLAG_TIMEOUT);
        return;
      }
      const uint32_t item = sh.sel_item[b];
      if (item == kSelectEnd) return;
      select_top16(item_at(items, item), sh.h[b], sh.sel, lane);
      if (lane == 0) {
        __threadfence();
        st_release_u32(ws.ready + item, 1u);  // the codebook is written
        mbar_arrive(&sh.sel_empty[b]);
      }
    }
  }

  // ------------------------------------------------------------------ consumer warps
  // Each warp waits for its stages on its own (no lock-step between warps);
  // the consumer warps meet only when counts are flushed, on an mbarrier with
  // bounded waits, so a timed-out warp unwinds instead of leaving the others
  // waiting.
  char* const col = reinterpret_cast<char*>(sh.cnt + lane);  // this lane's counter column
  uint32_t cur = kNoItem;
  uint32_t run = 0;    // tiles of `cur` counted since the last flush
  uint32_t posts = 0;  // histograms handed to the select warp
  uint32_t meets = 0;  // completed phases of sh.fbar
  auto meet = [&]() -> bool {  // all consumer warps here; writes before it visible after it
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.fbar);
    const bool ok = warp_wait(&sh.fbar, meets & 1u);
    ++meets;
    if (!ok && lane == 0) set_flag(ws.cal.hdr, SZ_FLAG_TIMEOUT);
    return ok;
  };
  auto wait_buffer = [&]() -> bool {
    if (posts < 2) return true;
    const bool ok = warp_wait(&sh.sel_empty[posts & 1u], ((posts >> 1) - 1) & 1u);
    if (!ok && lane == 0) set_flag(ws.cal.hdr, SZ_FLAG_TIMEOUT);
    return ok;
  };
  auto post = [&](uint32_t item) {  // after a meet
    if (tid == 0) {
      sh.sel_item[posts & 1u] = item;
      mbar_arrive(&sh.sel_full[posts & 1u]);
    }
    ++posts;
  };
  auto flush = [&]() -> bool {
    if (!meet()) return false;  // every count of the tensor's tiles is in
    const uint32_t sum = take_bin(sh.cnt, tid);
    const uint64_t tiles = tiles_of(item_at(items, cur).n);
    if (uint64_t(run) == tiles) {
      if (!wait_buffer()) return false;
      sh.h[posts & 1u][tid] = sum;
      if (!meet()) return false;  // sums written, counters clear
      post(cur);
    } else {
      uint32_t* gh = ws.cal.hist + uint64_t(cur) * 256;
      if (sum) atomicAdd(gh + tid, sum);
      __threadfence();
      if (!meet()) return false;
      if (tid == 0) {
        const uint32_t old = atomicAdd(ws.cal.done + cur, run);
        sh.s_last = ((old & kItemInvalid) == 0) && (uint64_t(old) + run == tiles);
      }
      if (!meet()) return false;
      if (sh.s_last) {
        __threadfence();
        if (!wait_buffer()) return false;
        sh.h[posts & 1u][tid] = __ldcg(gh + tid);
        if (!meet()) return false;
        post(cur);
      }
    }
    run = 0;
    return true;
  };
  // escape totals per tensor, per warp, added when the tensor changes
  uint32_t acc_item = kNoItem, acc = 0;
  bool dense = false;  // this warp staged no escapes of some chunk (enc_regen will write them)
  bool failed = false;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kCeStages);
    if (!warp_wait(&sh.full[s], (it / kCeStages) & 1)) {
      if (lane == 0) set_flag(ws.cal.hdr, SZ_FLAG_TIMEOUT);
      failed = true;
      break;
    }
    const CeStage& st = sh.st[s];
    const uint32_t flags = st.flags, item = st.item, n_tile = st.n_tile;
    if (flags & kStageEnd) break;
    if (flags & kStageCount) {
      if (!(flags & kStageInvalid)) {
        if (item != cur) {
          if (run && !flush()) {
            failed = true;
            break;
          }
          cur = item;
        }
        count_tile(st.x, n_tile, col, tid);
        ++run;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[s]);
      if (flags & kStageJobEnd) {
        // the job's counts go out now: this CTA may wait for those codebooks next
        if (run && !flush()) {
          failed = true;
          break;
        }
        cur = kNoItem;
      }
      continue;
    }
    if (!(flags & kStageInvalid)) {
      const uint64_t chunk = st.tile * kChunksPerTile + warp;  // global chunk index
      uint32_t* slot = ws.enc.stage + chunk * kChunk;
      const uint32_t run_e = (n_tile == kTile) ? encode_chunk8(st, warp, lane, slot)
                                               : encode_chunk<false>(st, warp, lane, slot);
      if (item != acc_item) {
        if (lane == 0 && acc) atomicAdd(ws.enc.item_esc + acc_item, acc);
        acc_item = item;
        acc = 0;
      }
      acc += run_e;
      dense |= run_e > kStageMax;
      if (lane == 0) ws.enc.chunk_cnt[chunk] = uint16_t(run_e);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
  }
  if (lane == 0 && acc) atomicAdd(ws.enc.item_esc + acc_item, acc);
  if (lane == 0 && dense) atomicOr(&ws.enc.hdr->dense, 1u);
  if (failed) return;  // the select warp stops on its own timeout
  if (run && !flush()) return;
  // tell the select warp to stop once it has ranked everything posted
  if (!wait_buffer() || !meet()) return;
  post(kSelectEnd);
}

}  // namespace

cudaError_t launch_calibrate_encode(const Items& items, void* ws_base, cudaStream_t stream, const DeviceInfo& dev) {
  CeWs ws = ce_ws(ws_base, items.count, items.total_tiles);
  ws.enc.small = small_route(items);
  cudaError_t err = cudaMemsetAsync(ws_base, 0, sizeof(WsHeader), stream);
  if (err != cudaSuccess) return err;
  {
    uint64_t work = items.total_tiles > items.count ? items.total_tiles : items.count;
    if (uint64_t(items.count) * 32 > work) work = uint64_t(items.count) * 32;
    if (uint64_t(items.count) * 256 > work) work = uint64_t(items.count) * 256;
    const uint64_t blocks = (work + 255) / 256;
    const unsigned grid = unsigned(blocks < 2048 ? (blocks ? blocks : 1) : 2048);
    ce_prepare<<<grid, 256, 0, stream>>>(items, ws);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  // tables of small tensors: whole tensors in shared memory, each read once,
  // one CTA per SM (the general kernels below then return at once, unless a
  // tensor is too large)
  TimingHook hook = g_timing;
  if (ws.enc.small) {
    if ((err = launch_small(items, ws.enc, ws.cal.done, stream, dev)) != cudaSuccess) return err;
    g_timing = TimingHook{nullptr, nullptr};
  }
  if (items.total_tiles > 0) {
    static thread_local int configured_device = -1;
    static thread_local int resident = 0;
    const size_t smem = sizeof(CeShared);
    if (configured_device != dev.device) {
      err = cudaFuncSetAttribute(ce_main, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (err != cudaSuccess) return err;
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, ce_main, kCeThreads, smem);
      if (err != cudaSuccess) return err;
      if (resident <= 0) return cudaErrorLaunchOutOfResources;
      configured_device = dev.device;
    }
    // every CTA resident at once (cooperative launch): encode tiles wait for
    // codebooks that other CTAs' count passes produce
    const int per_sm = resident < kCeCtasPerSm ? resident : kCeCtasPerSm;
    const unsigned grid = unsigned(per_sm * dev.num_sms);
    Items items_arg = items;
    void* args[] = {&items_arg, &ws};
    if (g_timing.before) cudaEventRecord(g_timing.before, stream);
    err = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(ce_main), dim3(grid), dim3(kCeThreads), args,
                                      smem, stream);
    if (g_timing.after) cudaEventRecord(g_timing.after, stream);
    if (err != cudaSuccess) {
      g_timing = hook;
      return err;
    }
  }
  err = launch_place(items, ws.enc, stream, dev);
  g_timing = hook;
  return err;
}

}  // namespace sz
