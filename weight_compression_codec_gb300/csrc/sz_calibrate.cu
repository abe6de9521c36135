// Calibration: per-tensor exponent histogram and Top-16 codebook selection
// ("splitzip_codec.py" calibrate_codebook: unique exponent counts, order by
// count, keep min(16, distinct) values, coverage = kept / all).
//
// Two launches per call (after a 256-byte header memset):
//   cal_prepare  zeroes the per-item histograms and completion counters,
//                validates the item table, writes the codebook of n == 0 items;
//   cal_hist     streams every tile once into privatised shared-memory
//                counters, flushes them with one global atomic per non-zero
//                bin, and the CTA that flushes an item's last tiles ranks the
//                256 bins and writes the codebook (ties by ascending exponent
//                value).
//
// The histogram is bound by instruction issue, not by the atomics' conflicts,
// so the counters are laid out to make an element as cheap as possible: one
// 32-bit counter per (bin, thread), cnt[bin][tid] with 64 threads, so the
// byte offset of an element's counter is its exponent byte times 256 -- a
// shift and a mask of the BF16 pattern -- and the 32 lanes of a warp always
// hit 32 different banks whatever their bins.  The adds are shared-memory
// reductions without a return value.  Each thread keeps the next tile's
// 16 x 16 bytes in flight (register double buffer) while it counts the
// current one.
#include "sz_internal.h"

namespace sz {
namespace {

constexpr int kHistThreads = 64;
constexpr int kHistCtasPerSm = 3;
constexpr int kVecPerThread = kTile / 8 / kHistThreads;  // 16 x 16-byte vectors per tile
constexpr size_t kHistSmem = size_t(256) * kHistThreads * 4;  // 64 KiB
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
  extern __shared__ __align__(16) uint32_t cnt[];  // [256 bins][kHistThreads]
  __shared__ uint32_t h[256];
  __shared__ uint8_t dl[16];
  __shared__ unsigned long long s_top;
  __shared__ uint32_t s_nz;
  __shared__ int s_last;

  const int tid = threadIdx.x;
  // an inconsistent item table (flagged by cal_prepare) is never walked
  if (ws.hdr->flags & SZ_FLAG_ITEMS) return;
  for (int b = 0; b < 256; ++b) cnt[b * kHistThreads + tid] = 0;

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

  // this thread's counter column, as a byte address: counter of bin b is at
  // col + 256 * b
  char* const col = reinterpret_cast<char*>(cnt + tid);
  auto count_lo = [&](uint32_t w) {  // element in bits 0..15
    atomicAdd(reinterpret_cast<uint32_t*>(col + ((w << 1) & 0xFF00u)), 1u);
  };
  auto count_hi = [&](uint32_t w) {  // element in bits 16..31
    atomicAdd(reinterpret_cast<uint32_t*>(col + ((w >> 15) & 0xFF00u)), 1u);
  };
  auto count_vec = [&](const uint4& v) {
    count_lo(v.x);
    count_hi(v.x);
    count_lo(v.y);
    count_hi(v.y);
    count_lo(v.z);
    count_hi(v.z);
    count_lo(v.w);
    count_hi(v.w);
  };

  auto flush = [&]() {
    __syncthreads();
    {
      uint32_t* gh = ws.hist + uint64_t(cur) * 256;
#pragma unroll
      for (int q = 0; q < 256 / kHistThreads; ++q) {
        const int b = tid * (256 / kHistThreads) + q;
        uint32_t* row = cnt + b * kHistThreads;
        uint32_t sum = 0;
#pragma unroll 8
        for (int j = 0; j < kHistThreads; ++j) {
          const int c = (j + tid) & (kHistThreads - 1);  // lanes read 32 different banks
          sum += row[c];
          row[c] = 0;
        }
        if (sum) atomicAdd(gh + b, sum);
      }
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

  // r holds the current full tile once `have` is set: the next full tile of
  // the same item is loaded before the current one is counted.
  uint4 r[kVecPerThread];
  bool have = false;
  for (uint64_t t = t0; t < t1; ++t) {
    if (t >= cur_begin + cur_tiles) {
      if (run) flush();
      cur = find_item(items, t);
      cur_begin = item_at(items, cur).tile_begin;
      cur_tiles = tiles_of(item_at(items, cur).n);
      have = false;
    }
    const sz_item& it = item_at(items, cur);
    if ((ws.done[cur] & kItemInvalid) || t - cur_begin >= cur_tiles) {  // invalid item: nothing is read
      have = false;
      continue;
    }
    const uint64_t base = (t - cur_begin) * kTile;
    const uint64_t left = it.n - base;
    const uint32_t nt = left < kTile ? uint32_t(left) : kTile;
    const uint4* src = reinterpret_cast<const uint4*>(it.x + base);
    if (nt == kTile) {
      if (!have) {
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) r[k] = __ldg(src + tid + k * kHistThreads);
      }
      const bool next_full = (t + 1 < t1) && (t + 1 < cur_begin + cur_tiles) && (left >= 2 * uint64_t(kTile));
      uint4 q[kVecPerThread];
      if (next_full) {
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) q[k] = __ldg(src + kTile / 8 + tid + k * kHistThreads);
      }
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) count_vec(r[k]);
      if (next_full) {
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) r[k] = q[k];
      }
      have = next_full;
    } else {
      have = false;
      const uint32_t nvec = nt >> 3;
      for (uint32_t v = tid; v < nvec; v += kHistThreads) count_vec(__ldg(src + v));
      const uint32_t rem = nt & 7u;
      if (uint32_t(tid) < rem) count_lo(it.x[base + (nvec << 3) + tid]);
    }
    ++run;
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
