// Calibration: per-tensor exponent histogram and Top-16 codebook selection
// ("splitzip_codec.py" calibrate_codebook: unique exponent counts, order by
// count, keep min(16, distinct) values, coverage = kept / all).
//
// Two launches per call (after a 256-byte header memset):
//   cal_prepare  zeroes the per-item histograms and completion counters,
//                validates the item table, writes the codebook of n == 0 items;
//   cal_hist     persistent CTAs own contiguous runs of tiles.  A producer
//                warp streams them (16 KiB tiles) through a 4-stage
//                shared-memory ring with TMA bulk copies, so the counting
//                warps never wait on global loads; it steps through the item
//                table instead of searching it.  The 8 counting warps share
//                one 32-bit counter per (bin, lane), cnt[bin][lane]: the byte
//                offset of an element's counter is its exponent byte times
//                128 -- a shift and a mask of the BF16 pattern -- and the 32
//                lanes of a warp always hit 32 different banks whatever their
//                bins.  The adds are shared-memory atomics without a return
//                value; keying the columns by lane rather than by thread keeps
//                the counters at 32 KiB, so 16 counting warps fit on an SM.
//                When the tensor changes, thread b sums and clears bin b.  A
//                tensor counted whole by one CTA goes straight to the CTA's
//                select warp (two histogram buffers), which ranks it while the
//                counting warps go on; otherwise the sums go to a global
//                histogram (one atomic per non-zero bin) and the CTA that adds
//                a tensor's last tiles hands it over.  The ranking (ties by
//                ascending exponent value) compares only the non-zero bins.
#include "sz_count.cuh"
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kCountWarps = 8;
constexpr int kCountThreads = kCountWarps * 32;
constexpr int kProducerWarp = kCountWarps;
constexpr int kSelectWarp = kCountWarps + 1;
constexpr int kCalThreads = kCountThreads + 64;  // + producer warp + select warp
constexpr int kCalStages = 4;
constexpr int kCalCtasPerSm = 2;
constexpr uint32_t kStageEnd = 1u, kStageInvalid = 2u;
constexpr uint32_t kSelectEnd = 0xFFFFFFFFu;  // posted to the select warp when the CTA is done
constexpr unsigned FULL = 0xFFFFFFFFu;

struct __align__(128) CalStageBuf {
  uint16_t x[kTile];
};
struct CalHdr {
  uint32_t item, n, flags, pad;
};
static_assert(kCountThreads == 256, "one counting thread per exponent bin");

struct CalShared {
  uint32_t cnt[256 * 32];  // [bin][lane]
  CalStageBuf st[kCalStages];
  CalHdr hdr[kCalStages];
  uint64_t full[kCalStages];
  uint64_t empty[kCalStages];
  // histograms handed from the counting warps to the select warp (double buffered)
  alignas(16) uint32_t h[2][256];
  uint32_t sel_item[2];
  uint64_t sel_full[2];
  uint64_t sel_empty[2];
  SelectScratch sel;  // select warp scratch
  uint64_t fbar;      // the counting warps meet here when counts are flushed
  int s_last;
};

__global__ void cal_prepare(const __grid_constant__ Items items, CalWs ws) {
  pdl_trigger();
  const uint64_t nthreads = uint64_t(gridDim.x) * blockDim.x;
  const uint64_t gtid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (uint64_t w = gtid; w < uint64_t(items.count) * 256; w += nthreads) ws.hist[w] = 0;
  for (uint64_t i = gtid; i < items.count; i += nthreads) {
    const sz_item& it = item_at(items, uint32_t(i));
    uint32_t bad = 0;
    if (it.n > SZ_MAX_ELEMS) bad |= SZ_FLAG_SIZE;
    if (it.codebook == nullptr || (reinterpret_cast<uintptr_t>(it.codebook) & 15)) bad |= SZ_FLAG_ALIGN;
    if (it.n > 0 && (it.x == nullptr || (reinterpret_cast<uintptr_t>(it.x) & 15))) bad |= SZ_FLAG_ALIGN;
    if (items.table) {
      const uint64_t expect = (i == 0) ? 0 : items.table[i - 1].tile_begin + tiles_of(items.table[i - 1].n);
      if (it.tile_begin != expect) bad |= SZ_FLAG_ITEMS;
      if (i + 1 == items.count && it.tile_begin + tiles_of(it.n) != items.total_tiles) bad |= SZ_FLAG_ITEMS;
    }
    ws.done[i] = bad ? kItemInvalid : 0u;
    if (bad) {
      set_flag(ws.hdr, bad);
    } else if (it.n == 0) {
      write_empty_codebook(it.codebook);
    }
  }
}

__global__ void __launch_bounds__(kCalThreads, kCalCtasPerSm) cal_hist(const __grid_constant__ Items items, CalWs ws) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  CalShared& sh = *reinterpret_cast<CalShared*>(smem_raw);
  const uint32_t tid = threadIdx.x;
  const uint32_t warp = tid >> 5, lane = tid & 31u;
  const uint64_t T = items.total_tiles;
  const uint64_t per = (T + gridDim.x - 1) / gridDim.x;
  const uint64_t t0 = uint64_t(blockIdx.x) * per;
  const uint64_t t1 = (t0 + per < T) ? t0 + per : T;
  if (t0 >= t1) return;
  // An inconsistent item table (flagged by cal_prepare) is never walked: every
  // warp reads the flags, the producer after its first (bounds-safe) search.
  pdl_wait();  // cal_prepare's writes
  const uint32_t hdr_flags = ws.hdr->flags;

  for (uint32_t w = tid; w < 256 * 32; w += kCalThreads) sh.cnt[w] = 0;
  if (tid == 0) {
    for (int s = 0; s < kCalStages; ++s) {
      mbar_init(&sh.full[s], 1 + 32);
      mbar_init(&sh.empty[s], kCountWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.sel_full[b], 1);
      mbar_init(&sh.sel_empty[b], 1);
    }
    mbar_init(&sh.fbar, kCountWarps);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    // Lane l holds table entry wb + l (tile range, data pointer, invalid
    // mark), loaded 32 at a time, so crossing into the next tensor costs
    // shuffles rather than dependent global loads.
    uint32_t cur = find_item_warp(items, t0, lane);
    if (hdr_flags & SZ_FLAG_ITEMS) return;
    uint32_t wb = 0;
    uint64_t w_tb = 0, w_n = 0;
    const uint16_t* w_x = nullptr;
    uint32_t w_inv = 0;
    auto load_window = [&](uint32_t base) {
      wb = base;
      const uint32_t i = base + lane;
      if (i < items.count) {
        const sz_item& e = item_at(items, i);
        w_tb = e.tile_begin;
        w_n = e.n;
        w_x = e.x;
        w_inv = ws.done[i] & kItemInvalid;
      }
    };
    auto shfl64 = [&](uint64_t v, uint32_t src) {
      return (uint64_t(__shfl_sync(FULL, uint32_t(v >> 32), src)) << 32) | __shfl_sync(FULL, uint32_t(v), src);
    };
    load_window(cur);
    uint64_t cur_begin = 0, cur_end = 0, cur_n = 0;
    const uint16_t* cur_x = nullptr;
    bool cur_inv = false;
    uint32_t it = 0;
    for (uint64_t t = t0;; ++t, ++it) {
      const int s = int(it % kCalStages);
      if (it >= uint32_t(kCalStages) && !__all_sync(FULL, mbar_wait(&sh.empty[s], ((it / kCalStages) - 1) & 1))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return;
      }
      CalHdr& hd = sh.hdr[s];
      if (t >= t1) {
        if (lane == 0) {
          hd.flags = kStageEnd;
          mbar_arrive(&sh.full[s]);
        }
        cp_async_mbar_arrive_noinc(&sh.full[s]);
        return;
      }
      if (t >= cur_end) {
        // the next tensor with a tile at t (the table is validated as consecutive)
        if (t != t0) ++cur;
        for (;;) {
          if (cur >= items.count) {  // cannot happen for a consecutive table; ends the walk
            cur_inv = true;
            cur_end = t1;
            break;
          }
          if (cur - wb >= 32) load_window(cur);
          const uint32_t l = cur - wb;
          cur_begin = shfl64(w_tb, l);
          cur_n = shfl64(w_n, l);
          cur_x = reinterpret_cast<const uint16_t*>(shfl64(reinterpret_cast<uint64_t>(w_x), l));
          cur_inv = __shfl_sync(FULL, w_inv, l) != 0;
          cur_end = cur_begin + tiles_of(cur_n);
          if (t < cur_end) break;
          ++cur;  // an empty tensor owns no tile
        }
      }
      const uint64_t g = (t - cur_begin) * kTile;
      const bool invalid = cur_inv || t < cur_begin || g >= cur_n;
      const uint32_t nh = invalid ? 0u : ((cur_n - g < kTile) ? uint32_t(cur_n - g) : kTile);
      const uint32_t bulk = (nh * 2u) & ~15u;
      const uint32_t tail = nh * 2u - bulk;
      if (lane == 0) {
        hd.item = cur;
        hd.n = nh;
        hd.flags = invalid ? kStageInvalid : 0u;
        mbar_arrive_expect_tx(&sh.full[s], bulk);
        // evict-first: the step's previous decode may have left ~100 MB of
        // dirty output in L2; counting x (read once) should not evict those
        // lines, which costs their write-back inside this kernel (KV cache
        // 64 x 4 Mi: 102.7 -> 94.5 us, the step 5 us shorter)
        if (bulk) bulk_g2s_evict_first(sh.st[s].x, cur_x + g, bulk, &sh.full[s]);
      } else if (lane == 1 && tail) {
        cp_async16_zfill(reinterpret_cast<uint8_t*>(sh.st[s].x) + bulk,
                         reinterpret_cast<const uint8_t*>(cur_x + g) + bulk, tail);
      }
      cp_async_mbar_arrive_noinc(&sh.full[s]);
    }
  }

  if (hdr_flags & SZ_FLAG_ITEMS) return;

  if (warp == kSelectWarp) {
    // ---------------------------------------------------------------- select warp
    // Ranks each histogram the counting warps hand over, while they count on.
    for (uint32_t k = 0;; ++k) {
      const uint32_t b = k & 1u;
      if (!__all_sync(FULL, mbar_wait(&sh.sel_full[b], (k >> 1) & 1u))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return;
      }
      const uint32_t item = sh.sel_item[b];
      if (item == kSelectEnd) return;
      select_top16(item_at(items, item), sh.h[b], sh.sel, lane);
      if (lane == 0) mbar_arrive(&sh.sel_empty[b]);
    }
  }

  // ------------------------------------------------------------------ counting warps
  // Each warp waits for its stages on its own (no lock-step between warps:
  // a warp may run up to the ring's depth ahead of another); the warps meet
  // only when counts are flushed, on an mbarrier with bounded waits, so a
  // timed-out warp unwinds instead of leaving the others waiting.
  // this lane's counter column, as a byte address: bin b at col + 128 * b
  char* const col = reinterpret_cast<char*>(sh.cnt + lane);
  uint32_t cur = 0xFFFFFFFFu;
  uint32_t run = 0;    // tiles of `cur` counted since the last flush
  uint32_t posts = 0;  // histograms handed to the select warp
  uint32_t meets = 0;  // completed phases of sh.fbar
  auto meet = [&]() -> bool {  // all counting warps here; writes before it visible after it
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.fbar);
    const bool ok = __all_sync(FULL, mbar_wait(&sh.fbar, meets & 1u));
    ++meets;
    if (!ok && lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
    return ok;
  };
  // Waits until buffer posts & 1 is free again (its previous histogram ranked).
  auto wait_buffer = [&]() -> bool {
    if (posts < 2) return true;
    const bool ok = __all_sync(FULL, mbar_wait(&sh.sel_empty[posts & 1u], ((posts >> 1) - 1) & 1u));
    if (!ok && lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
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
    const uint32_t sum = take_bin(sh.cnt, tid);  // thread b sums and clears bin b
    const uint64_t tiles = tiles_of(item_at(items, cur).n);
    if (uint64_t(run) == tiles) {
      // this CTA counted every tile of the tensor: hand the sums over directly
      if (!wait_buffer()) return false;
      sh.h[posts & 1u][tid] = sum;
      if (!meet()) return false;  // sums written; counters clear for the next tensor
      post(cur);
    } else {
      uint32_t* gh = ws.hist + uint64_t(cur) * 256;
      if (sum) atomicAdd(gh + tid, sum);
      __threadfence();
      if (!meet()) return false;
      if (tid == 0) {
        const uint32_t old = atomicAdd(ws.done + cur, run);
        sh.s_last = ((old & kItemInvalid) == 0) && (uint64_t(old) + run == tiles);
      }
      if (!meet()) return false;
      if (sh.s_last) {
        // the last CTA to add its counts ranks the tensor
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
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kCalStages);
    if (!__all_sync(FULL, mbar_wait(&sh.full[s], (it / kCalStages) & 1))) {
      if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      return;  // the select warp stops on its own timeout
    }
    const CalHdr hd = sh.hdr[s];
    if (hd.flags & kStageEnd) break;
    if (hd.item != cur) {
      if (run && !flush()) return;
      cur = hd.item;
    }
    if (!(hd.flags & kStageInvalid)) {
      count_tile(sh.st[s].x, hd.n, col, tid);
      ++run;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
  }
  if (run && !flush()) return;
  // tell the select warp to stop once it has ranked everything posted
  if (!wait_buffer() || !meet()) return;
  post(kSelectEnd);
}

}  // namespace

cudaError_t launch_calibrate(const Items& items, void* ws_base, cudaStream_t stream, const DeviceInfo& dev) {
  CalWs ws = cal_ws(ws_base, items.count);
  cudaError_t err = cudaMemsetAsync(ws_base, 0, sizeof(WsHeader), stream);
  if (err != cudaSuccess) return err;
  {
    const uint64_t work = uint64_t(items.count) * 256;
    const uint64_t blocks = (work + 255) / 256;
    const unsigned grid = unsigned(blocks < 1024 ? (blocks ? blocks : 1) : 1024);
    cal_prepare<<<grid, 256, 0, stream>>>(items, ws);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (items.total_tiles == 0) return cudaSuccess;
  static thread_local int configured_device = -1;
  const size_t smem = sizeof(CalShared);
  if (configured_device != dev.device) {
    err = cudaFuncSetAttribute(cal_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (err != cudaSuccess) return err;
    configured_device = dev.device;
  }
  const uint64_t cap = uint64_t(dev.num_sms) * kCalCtasPerSm;
  const unsigned grid = unsigned(items.total_tiles < cap ? items.total_tiles : cap);
  if (g_timing.before) cudaEventRecord(g_timing.before, stream);
  err = launch_pdl(cal_hist, dim3(grid), dim3(kCalThreads), smem, stream, items, ws);
  if (g_timing.after) cudaEventRecord(g_timing.after, stream);
  return err;
}

}  // namespace sz
