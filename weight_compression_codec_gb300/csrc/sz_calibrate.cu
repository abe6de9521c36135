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
//                warps never wait on global loads.  The 8 counting warps share
//                one 32-bit counter per (bin, lane), cnt[bin][lane]: the byte
//                offset of an element's counter is its exponent byte times
//                128 -- a shift and a mask of the BF16 pattern -- and the 32
//                lanes of a warp always hit 32 different banks whatever their
//                bins.  The adds are shared-memory atomics without a return
//                value; keying the columns by lane rather than by thread keeps
//                the counters at 32 KiB, so 16 counting warps fit on an SM.  Counters are flushed with one global atomic
//                per non-zero bin when the tensor changes; the CTA that
//                flushes a tensor's last tiles ranks its 256 bins and writes
//                the codebook (ties by ascending exponent value).
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kCountWarps = 8;
constexpr int kCountThreads = kCountWarps * 32;
constexpr int kCalThreads = kCountThreads + 32;  // + producer warp
constexpr int kCalStages = 4;
constexpr int kCalCtasPerSm = 2;
constexpr uint32_t kItemInvalid = 0x80000000u;
constexpr uint32_t kStageEnd = 1u, kStageInvalid = 2u;
constexpr unsigned FULL = 0xFFFFFFFFu;

struct __align__(128) CalStageBuf {
  uint16_t x[kTile];
};
struct CalHdr {
  uint32_t item, n, flags, pad;
};
struct CalShared {
  uint32_t cnt[256 * 32];  // [bin][lane]
  CalStageBuf st[kCalStages];
  CalHdr hdr[kCalStages];
  uint64_t full[kCalStages];
  uint64_t empty[kCalStages];
  uint32_t h[256];
  unsigned long long s_top;
  uint32_t s_nz;
  int s_last;
  uint8_t dl[16];
};



__device__ void write_empty_codebook(sz_codebook* cb) {
  for (int v = 0; v < 256; ++v) cb->enc_lut[v] = kEscape;
  for (int c = 0; c < 16; ++c) cb->dec_lut[c] = 0;
  cb->n_top = 0;
  cb->reserved0 = 0;
  cb->top_count = 0;
  cb->n = 0;
  cb->coverage = 1.0;
}

__global__ void cal_prepare(const __grid_constant__ Items items, CalWs ws) {
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

// Ranks the 256 bins of `it` (count desc, value asc) and writes its codebook.
// Run by the kCountThreads counting threads (named barrier 1).
__device__ void select_top16(const sz_item& it, const uint32_t* __restrict__ ghist, CalShared& sh) {
  const uint32_t tid = threadIdx.x;
  __threadfence();
  for (uint32_t b = tid; b < 256; b += kCountThreads) sh.h[b] = __ldcg(ghist + b);
  if (tid < 16) sh.dl[tid] = 0;
  if (tid == 0) {
    sh.s_top = 0;
    sh.s_nz = 0;
  }
  named_bar_sync(1, kCountThreads);
  sz_codebook* cb = it.codebook;
  unsigned long long top = 0;
  uint32_t nz = 0;
  for (uint32_t b = tid; b < 256; b += kCountThreads) {
    const uint32_t c = sh.h[b];
    uint32_t rank = 0;
#pragma unroll 8
    for (uint32_t j = 0; j < 256; ++j) {
      const uint32_t cj = sh.h[j];
      rank += (cj > c) | ((cj == c) & (j < b));
    }
    uint32_t code = kEscape;
    if (c > 0 && rank < 16) {
      code = rank;
      sh.dl[rank] = uint8_t(b);
      top += c;
    }
    nz += (c > 0);
    cb->enc_lut[b] = uint8_t(code);
  }
  atomicAdd(&sh.s_top, top);
  atomicAdd(&sh.s_nz, nz);
  named_bar_sync(1, kCountThreads);
  if (tid < 16) cb->dec_lut[tid] = sh.dl[tid];
  if (tid == 0) {
    const uint64_t n = it.n;
    cb->n_top = sh.s_nz < 16 ? sh.s_nz : 16;
    cb->reserved0 = 0;
    cb->top_count = sh.s_top;
    cb->n = n;
    cb->coverage = n ? double(sh.s_top) / double(n) : 1.0;
  }
  named_bar_sync(1, kCountThreads);  // h, dl and the sums are reused by the next select
}

__global__ void __launch_bounds__(kCalThreads, kCalCtasPerSm) cal_hist(const __grid_constant__ Items items, CalWs ws) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  CalShared& sh = *reinterpret_cast<CalShared*>(smem_raw);
  const uint32_t tid = threadIdx.x;
  const uint32_t warp = tid >> 5, lane = tid & 31u;
  // an inconsistent item table (flagged by cal_prepare) is never walked
  if (ws.hdr->flags & SZ_FLAG_ITEMS) return;

  const uint64_t T = items.total_tiles;
  const uint64_t per = (T + gridDim.x - 1) / gridDim.x;
  const uint64_t t0 = uint64_t(blockIdx.x) * per;
  const uint64_t t1 = (t0 + per < T) ? t0 + per : T;
  if (t0 >= t1) return;

  for (uint32_t w = tid; w < 256 * 32; w += kCalThreads) sh.cnt[w] = 0;
  if (tid == 0) {
    for (int s = 0; s < kCalStages; ++s) {
      mbar_init(&sh.full[s], 1 + 32);
      mbar_init(&sh.empty[s], kCountWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCountWarps) {
    // ---------------------------------------------------------------- producer warp
    uint32_t cur = 0;
    uint64_t cur_begin = 0, cur_end = 0;
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
        cur = find_item(items, t);
        cur_begin = item_at(items, cur).tile_begin;
        cur_end = cur_begin + tiles_of(item_at(items, cur).n);
      }
      const sz_item& itm = item_at(items, cur);
      const uint64_t g = (t - cur_begin) * kTile;
      const bool invalid = (ws.done[cur] & kItemInvalid) != 0 || t - cur_begin >= tiles_of(itm.n);
      const uint32_t nh = (invalid || g >= itm.n) ? 0u : ((itm.n - g < kTile) ? uint32_t(itm.n - g) : kTile);
      const uint32_t bulk = (nh * 2u) & ~15u;
      const uint32_t tail = nh * 2u - bulk;
      if (lane == 0) {
        hd.item = cur;
        hd.n = nh;
        hd.flags = invalid ? kStageInvalid : 0u;
        mbar_arrive_expect_tx(&sh.full[s], bulk);
        if (bulk) bulk_g2s(sh.st[s].x, itm.x + g, bulk, &sh.full[s]);
      } else if (lane == 1 && tail) {
        cp_async16_zfill(reinterpret_cast<uint8_t*>(sh.st[s].x) + bulk,
                         reinterpret_cast<const uint8_t*>(itm.x + g) + bulk, tail);
      }
      cp_async_mbar_arrive_noinc(&sh.full[s]);
    }
  }

  // ------------------------------------------------------------------ counting warps
  // this lane's counter column, as a byte address: bin b at col + 128 * b
  char* const col = reinterpret_cast<char*>(sh.cnt + lane);
  uint32_t cur = 0xFFFFFFFFu;
  uint32_t run = 0;  // tiles of `cur` counted since the last flush
  auto flush = [&]() {
    named_bar_sync(1, kCountThreads);
    uint32_t* gh = ws.hist + uint64_t(cur) * 256;
    for (uint32_t b = tid; b < 256; b += kCountThreads) {
      uint32_t* row = sh.cnt + b * 32;
      uint32_t sum = 0;
#pragma unroll 8
      for (uint32_t j = 0; j < 32; ++j) {
        const uint32_t c = (j + lane) & 31u;  // lanes read 32 different banks
        sum += row[c];
        row[c] = 0;
      }
      if (sum) atomicAdd(gh + b, sum);
    }
    __threadfence();
    named_bar_sync(1, kCountThreads);
    if (tid == 0) {
      const uint32_t old = atomicAdd(ws.done + cur, run);
      sh.s_last = ((old & kItemInvalid) == 0) && (uint64_t(old) + run == tiles_of(item_at(items, cur).n));
    }
    named_bar_sync(1, kCountThreads);
    if (sh.s_last) select_top16(item_at(items, cur), ws.hist + uint64_t(cur) * 256, sh);
    run = 0;
  };
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kCalStages);
    const bool ok = mbar_wait(&sh.full[s], (it / kCalStages) & 1);
    const CalHdr hd = sh.hdr[s];  // read before the vote: the stage may be released right after
    if (named_bar_red_or(1, kCountThreads, !ok)) {
      if (tid == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      return;
    }
    if (hd.flags & kStageEnd) break;
    if (hd.item != cur) {
      if (run) flush();
      cur = hd.item;
    }
    if (!(hd.flags & kStageInvalid)) {
      const uint4* xs = reinterpret_cast<const uint4*>(sh.st[s].x);
      if (hd.n == kTile) {
        uint4 v[kTile / 8 / kCountThreads];
#pragma unroll
        for (int k = 0; k < kTile / 8 / kCountThreads; ++k) v[k] = xs[tid + k * kCountThreads];
#pragma unroll
        for (int k = 0; k < kTile / 8 / kCountThreads; ++k) {
          const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            atomicAdd(reinterpret_cast<uint32_t*>(col + (w[q] & 0x7F80u)), 1u);
            atomicAdd(reinterpret_cast<uint32_t*>(col + ((w[q] >> 16) & 0x7F80u)), 1u);
          }
        }
      } else {
        const uint16_t* xe = sh.st[s].x;
        for (uint32_t e = tid; e < hd.n; e += kCountThreads)
          atomicAdd(reinterpret_cast<uint32_t*>(col + (uint32_t(xe[e]) & 0x7F80u)), 1u);
      }
      ++run;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
  }
  if (run) flush();
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
  cal_hist<<<grid, kCalThreads, smem, stream>>>(items, ws);
  err = cudaGetLastError();
  if (g_timing.after) cudaEventRecord(g_timing.after, stream);
  return err;
}

}  // namespace sz
