// Exponent histograms and the Top-16 select, shared by the calibration kernel
// and the fused calibrate + encode kernel.
#pragma once

#include "sz_device.cuh"

namespace sz {

constexpr uint32_t kItemInvalid = 0x80000000u;  // completion counter mark of an item not to be counted

// Scratch of one select warp.
struct SelectScratch {
  unsigned long long key[256];  // non-zero bins in bin order: count << 8 | (255 - bin)
  alignas(16) uint8_t lut[256];
  uint8_t dl[16];
};

__device__ inline void write_empty_codebook(sz_codebook* cb) {
  for (int v = 0; v < 256; ++v) cb->enc_lut[v] = kEscape;
  for (int c = 0; c < 16; ++c) cb->dec_lut[c] = 0;
  cb->n_top = 0;
  cb->reserved0 = 0;
  cb->top_count = 0;
  cb->n = 0;
  cb->coverage = 1.0;
}

// t / n correctly rounded (to nearest, ties to even) to an IEEE double, for
// integers 0 <= t <= n < 2^31, in integer arithmetic -- the value a double
// division t / n gives, at a fraction of the cost of FP64 work on this part.
// Schoolbook long division: t is scaled by 2^s so that n <= T < 2n; the
// quotient floor(T 2^53 / n) (54 bits: 53 for the significand, one to round
// on) comes from two steps of 22 and 31 bits, and the last remainder tells
// whether anything lies below the rounding bit.
__device__ __forceinline__ double ratio_rn(uint32_t t, uint32_t n) {
  if (t == 0) return 0.0;
  if (t >= n) return 1.0;
  int s = __clz(t) - __clz(n);  // t 2^s has the bit length of n
  uint64_t T = uint64_t(t) << s;
  if (T < n) {
    T <<= 1;
    ++s;
  }
  const uint64_t A = T << 22;                // < 2^54
  const uint64_t q1 = A / n, r1 = A % n;     // q1 < 2^23
  const uint64_t B = r1 << 31;               // < 2^62
  const uint64_t q2 = B / n, r2 = B % n;     // q2 < 2^31
  const uint64_t Q = (q1 << 31) | q2;        // floor(T 2^53 / n), in [2^53, 2^54)
  uint64_t mant = Q >> 1;                    // in [2^52, 2^53)
  if ((Q & 1u) && (r2 != 0 || (mant & 1u))) ++mant;
  int e = -s;                                // t / n = mant 2^-52 2^e
  if (mant == (1ull << 53)) {
    mant >>= 1;
    ++e;
  }
  return __longlong_as_double(static_cast<long long>((uint64_t(1023 + e) << 52) | (mant & ((1ull << 52) - 1u))));
}

// Ranks the 256 bins of histogram h (count desc, value asc) and writes the
// codebook of `it`; run by one warp, lane l loading bins 8l .. 8l+7.  Only
// non-zero bins take part: they are compacted in bin order as keys
// count << 8 | (255 - bin) -- a larger key ranks first, which puts the
// smaller bin first among equal counts -- and each counts the keys above its
// own.
__device__ inline void select_top16(const sz_item& it, const uint32_t* h, SelectScratch& sh, uint32_t lane) {
  const uint4 lo = reinterpret_cast<const uint4*>(h)[2 * lane];
  const uint4 hi = reinterpret_cast<const uint4*>(h)[2 * lane + 1];
  const uint32_t c[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t nz = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) nz += c[j] > 0;
  uint32_t incl = nz;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= uint32_t(d)) incl += v;
  }
  const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  uint32_t pos = incl - nz;
#pragma unroll
  for (uint32_t j = 0; j < 8; ++j)
    if (c[j]) sh.key[pos++] = (static_cast<unsigned long long>(c[j]) << 8) | (255u - (8u * lane + j));
  reinterpret_cast<uint2*>(sh.lut)[lane] = make_uint2(0x10101010u, 0x10101010u);  // kEscape
  if (lane < 16) sh.dl[lane] = 0;
  __syncwarp();
  for (uint32_t p = lane; p < total; p += 32) {
    const unsigned long long key = sh.key[p];
    uint32_t rank = 0;
    for (uint32_t j = 0; j < total; ++j) rank += sh.key[j] > key;
    if (rank < 16) {
      const uint32_t bin = 255u - uint32_t(key & 0xFFu);
      sh.lut[bin] = uint8_t(rank);
      sh.dl[rank] = uint8_t(bin);
    }
  }
  __syncwarp();
  sz_codebook* cb = it.codebook;
  reinterpret_cast<uint2*>(cb->enc_lut)[lane] = reinterpret_cast<const uint2*>(sh.lut)[lane];
  const uint32_t n_top = total < 16 ? total : 16u;
  unsigned long long top = lane < n_top ? h[sh.dl[lane]] : 0ull;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) top += __shfl_xor_sync(0xFFFFFFFFu, top, d);
  if (lane < 16) cb->dec_lut[lane] = sh.dl[lane];
  if (lane == 0) {
    const uint64_t n = it.n;
    cb->n_top = n_top;
    cb->reserved0 = 0;
    cb->top_count = top;
    cb->n = n;
    // the division in integer arithmetic where it fits (FP64 is slow on this part)
    cb->coverage = n == 0 ? 1.0 : (n < (1ull << 31) ? ratio_rn(uint32_t(top), uint32_t(n)) : double(top) / double(n));
  }
  __syncwarp();  // key, lut and dl are reused by the next select
}

// Index of the item holding global tile `tile` (the last item with
// tile_begin <= tile; empty items share the next one's tile_begin), found by
// the 32 lanes of a warp probing 32 entries per round: ceil(log32(count)) + 1
// dependent loads.  Needs a table validated as consecutive.
__device__ inline uint32_t find_item_warp(const Items& items, uint64_t tile, uint32_t lane) {
  if (items.table == nullptr) return 0;
  uint32_t lo = 0, hi = items.count;  // table[lo].tile_begin <= tile; the answer is in [lo, hi)
  while (hi - lo > 32) {
    const uint32_t step = (hi - lo + 31) / 32;
    const uint32_t p = lo + lane * step;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, p < hi && items.table[p].tile_begin <= tile);
    if (m) lo += (31u - __clz(m)) * step;  // m has lane 0 unless the table is not consecutive
    if (lo + step < hi) hi = lo + step;
  }
  const uint32_t p = lo + lane;
  const uint32_t m = __ballot_sync(0xFFFFFFFFu, p < hi && items.table[p].tile_begin <= tile);
  return m ? lo + (31u - __clz(m)) : lo;
}

// Counts the exponents of n_el BF16 patterns x (a staged tile, 16-byte
// aligned) into the (bin, lane) counters whose column for this lane starts at
// col: the counter of exponent v is at col + 128 * v.  Run by 256 threads.
__device__ __forceinline__ void count_tile(const uint16_t* x, uint32_t n_el, char* col, uint32_t tid) {
  if (n_el == kTile) {
    const uint4* xs = reinterpret_cast<const uint4*>(x);
    uint4 v[kTile / 8 / 256];
#pragma unroll
    for (int k = 0; k < kTile / 8 / 256; ++k) v[k] = xs[tid + k * 256];
#pragma unroll
    for (int k = 0; k < kTile / 8 / 256; ++k) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        atomicAdd(reinterpret_cast<uint32_t*>(col + (w[q] & 0x7F80u)), 1u);
        atomicAdd(reinterpret_cast<uint32_t*>(col + ((w[q] >> 16) & 0x7F80u)), 1u);
      }
    }
  } else {
    for (uint32_t e = tid; e < n_el; e += 256)
      atomicAdd(reinterpret_cast<uint32_t*>(col + (uint32_t(x[e]) & 0x7F80u)), 1u);
  }
}

// Sum of the 32 lane counters of bin `bin` in cnt[bin][lane], which it
// clears: 16-byte accesses, rotated so that the 8 threads of a quarter warp
// touch 8 different bank groups.
__device__ __forceinline__ uint32_t take_bin(uint32_t* cnt, uint32_t bin) {
  uint4* const row = reinterpret_cast<uint4*>(cnt + bin * 32);
  uint32_t sum = 0;
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    const uint32_t q = (k + bin) & 7u;
    const uint4 v = row[q];
    sum += v.x + v.y + v.z + v.w;
    row[q] = make_uint4(0u, 0u, 0u, 0u);
  }
  return sum;
}

}  // namespace sz
