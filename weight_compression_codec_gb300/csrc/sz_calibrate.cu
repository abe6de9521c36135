// Calibration: per-tensor exponent histogram and Top-16 codebook selection
// ("splitzip_codec.py" calibrate_codebook: unique exponent counts, order by
// count, keep min(16, distinct) values, coverage = kept / all).
//
// Two launches per call (after a 256-byte header memset):
//   cal_prepare  zeroes the per-item histograms and completion counters,
//                validates the item table, writes the codebook of n == 0 items;
//   cal_hist     streams every tile once (16-byte loads, ~48 KiB in flight per
//                SM) into privatised shared-memory counters, flushes them with
//                one global atomic per non-zero bin, and the CTA that flushes
//                an item's last tiles ranks the 256 bins and writes the
//                codebook (ties by ascending exponent value).
//
// Counters: 16-bit halves of a 32-bit word, word (bin >> 1) of the thread's
// own column -- cnt[(bin >> 1) * kHistThreads + tid] -- so the 32 lanes of a
// warp always hit 32 different banks whatever their bins are, and the adds
// are shared-memory reductions with no return value (no read-modify-write
// dependency chain).  A thread adds at most 64 per tile, so a flush every
// kFlushTiles tiles keeps every half below 65536.
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kHistThreads = 128;
constexpr int kHistCtasPerSm = 3;
constexpr int kPairs = 128;                       // 256 bins / 2 per word
constexpr uint32_t kFlushTiles = 1000;            // 1000 * 64 < 65536
constexpr size_t kHistSmem = size_t(kPairs) * kHistThreads * 4;  // 64 KiB
constexpr uint32_t kItemInvalid = 0x80000000u;

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

// Ranks the 256 bins of item `ii` (count desc, value asc) and writes its
// codebook.  Called by all kHistThreads threads of the CTA.
__device__ void select_top16(const sz_item& it, const uint32_t* __restrict__ ghist, uint32_t* h,
                             uint8_t* dl, unsigned long long* s_top, uint32_t* s_nz) {
  const int tid = threadIdx.x;
  __threadfence();
  for (int b = tid; b < 256; b += kHistThreads) h[b] = __ldcg(ghist + b);
  if (tid < 16) dl[tid] = 0;
  if (tid == 0) {
    *s_top = 0;
    *s_nz = 0;
  }
  __syncthreads();
  sz_codebook* cb = it.codebook;
  unsigned long long top = 0;
  uint32_t nz = 0;
  for (int b = tid; b < 256; b += kHistThreads) {
    const uint32_t c = h[b];
    uint32_t rank = 0;
#pragma unroll 8
    for (int j = 0; j < 256; ++j) {
      const uint32_t cj = h[j];
      rank += (cj > c) | ((cj == c) & (j < b));
    }
    uint32_t code = kEscape;
    if (c > 0 && rank < 16) {
      code = rank;
      dl[rank] = uint8_t(b);
      top += c;
    }
    nz += (c > 0);
    cb->enc_lut[b] = uint8_t(code);
  }
  atomicAdd(s_top, top);
  atomicAdd(s_nz, nz);
  __syncthreads();
  if (tid < 16) cb->dec_lut[tid] = dl[tid];
  if (tid == 0) {
    const uint64_t n = it.n;
    cb->n_top = *s_nz < 16 ? *s_nz : 16;
    cb->reserved0 = 0;
    cb->top_count = *s_top;
    cb->n = n;
    cb->coverage = n ? double(*s_top) / double(n) : 1.0;
  }
}

__global__ void __launch_bounds__(kHistThreads, kHistCtasPerSm)
    cal_hist(const __grid_constant__ Items items, CalWs ws) {
  extern __shared__ __align__(16) uint32_t cnt[];  // [kPairs][kHistThreads]
  __shared__ uint32_t h[256];
  __shared__ uint8_t dl[16];
  __shared__ unsigned long long s_top;
  __shared__ uint32_t s_nz;
  __shared__ int s_last;

  const int tid = threadIdx.x;
  // an inconsistent item table (flagged by cal_prepare) is never walked
  if (ws.hdr->flags & SZ_FLAG_ITEMS) return;
  for (int q = 0; q < kPairs; ++q) cnt[q * kHistThreads + tid] = 0;

  const uint64_t T = items.total_tiles;
  const uint64_t per = (T + gridDim.x - 1) / gridDim.x;
  const uint64_t t0 = uint64_t(blockIdx.x) * per;
  const uint64_t t1 = (t0 + per < T) ? t0 + per : T;
  __syncthreads();
  if (t0 >= t1) return;

  uint32_t cur = find_item(items, t0);
  uint64_t cur_begin = item_at(items, cur).tile_begin;
  uint64_t cur_tiles = tiles_of(item_at(items, cur).n);
  uint32_t run = 0;  // tiles counted since the last flush

  uint32_t* mycol = cnt + tid;
  auto count = [&](uint32_t x) {
    const uint32_t b = (x >> 7) & 0xFFu;
    atomicAdd(mycol + (b >> 1) * kHistThreads, 1u << ((b & 1u) << 4));
  };
  auto count_word = [&](uint32_t w) {
    count(w & 0xFFFFu);
    count(w >> 16);
  };

  auto flush = [&]() {
    __syncthreads();
    {
      const int q = tid;  // bins 2q, 2q+1
      uint32_t lo = 0, hi = 0;
      uint32_t* row = cnt + q * kHistThreads;
#pragma unroll 8
      for (int j = 0; j < kHistThreads; ++j) {
        const int c = (j + tid) & (kHistThreads - 1);
        const uint32_t w = row[c];
        row[c] = 0;
        lo += w & 0xFFFFu;
        hi += w >> 16;
      }
      uint32_t* gh = ws.hist + uint64_t(cur) * 256;
      if (lo) atomicAdd(gh + 2 * q, lo);
      if (hi) atomicAdd(gh + 2 * q + 1, hi);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const uint32_t old = atomicAdd(ws.done + cur, run);
      s_last = ((old & kItemInvalid) == 0) && (uint64_t(old) + run == cur_tiles);
    }
    __syncthreads();
    if (s_last) select_top16(item_at(items, cur), ws.hist + uint64_t(cur) * 256, h, dl, &s_top, &s_nz);
    run = 0;
  };

  for (uint64_t t = t0; t < t1; ++t) {
    if (t >= cur_begin + cur_tiles) {
      if (run) flush();
      cur = find_item(items, t);
      cur_begin = item_at(items, cur).tile_begin;
      cur_tiles = tiles_of(item_at(items, cur).n);
    }
    const sz_item& it = item_at(items, cur);
    if ((ws.done[cur] & kItemInvalid) || t - cur_begin >= cur_tiles) {  // invalid item: nothing is read
      continue;
    }
    const uint64_t base = (t - cur_begin) * kTile;
    const uint64_t left = it.n - base;
    const uint32_t nt = left < kTile ? uint32_t(left) : kTile;
    const uint4* src = reinterpret_cast<const uint4*>(it.x + base);
    if (nt == kTile) {
      uint4 r[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) r[k] = __ldg(src + tid + k * kHistThreads);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        count_word(r[k].x);
        count_word(r[k].y);
        count_word(r[k].z);
        count_word(r[k].w);
      }
    } else {
      const uint32_t nvec = nt >> 3;
      for (uint32_t v = tid; v < nvec; v += kHistThreads) {
        const uint4 r = __ldg(src + v);
        count_word(r.x);
        count_word(r.y);
        count_word(r.z);
        count_word(r.w);
      }
      const uint32_t rem = nt & 7u;
      if (uint32_t(tid) < rem) count(it.x[base + (nvec << 3) + tid]);
    }
    if (++run == kFlushTiles) flush();
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
  if (configured_device != dev.device) {
    err = cudaFuncSetAttribute(cal_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kHistSmem));
    if (err != cudaSuccess) return err;
    configured_device = dev.device;
  }
  const uint64_t cap = uint64_t(dev.num_sms) * kHistCtasPerSm;
  const unsigned grid = unsigned(items.total_tiles < cap ? items.total_tiles : cap);
  if (g_timing.before) cudaEventRecord(g_timing.before, stream);
  cal_hist<<<grid, kHistThreads, kHistSmem, stream>>>(items, ws);
  err = cudaGetLastError();
  if (g_timing.after) cudaEventRecord(g_timing.after, stream);
  return err;
}

}  // namespace sz
