// Calibrate + encode, and encode alone, of tables of small tensors
// ("splitzip_codec.py" calibrate_codebook followed by encode_torch +
// assemble_payload, per tensor, for many tensors such as the blocks of a
// paged KV cache): a whole tensor of at most kSmallMax elements (two tiles,
// 32 KiB of BF16) is held in shared memory, so each input is read from HBM
// once and nothing is staged.
//
// One CTA per SM: a producer warp copies the CTA's tensors (tensors b,
// b + G, b + 2G, ... of the G CTAs) with their table entries (fetched four
// tensors ahead, one load per lane) -- and, encoding alone, their codebooks
// -- into a ring of whole-tensor buffers by TMA;
// groups of 8 warps (two calibrating, three encoding alone) take the tensors
// in turn (group g of G' the tensors k = g, g + G', ... of the CTA), each
// with its own counters and barrier, so one group's barriers and serial
// steps overlap the others' work.  Per tensor, in a group:
//   1. calibrate only: the 256 threads count the exponents into counters
//      keyed by (bin, lane) (count_tile); thread b sums bin b, and ranks it
//      among the non-zero bins (count desc, value asc, as select_top16 does)
//      against their keys compacted per warp; the ranks below 16 are the
//      codes, and enc_lut / dec_lut go to the codebook;
//   2. warp w splits and packs chunks w and w + 8 (pk and sm straight to the
//      payload) and keeps, per lane, which of its elements are escapes;
//   3. after one group barrier every chunk's escape count is known, so each
//      warp writes its chunks' chunk_id / local_pos / esc_val at their final
//      offsets -- in element order, as the pages' encode_torch lists them;
//   4. the pads; the buffer goes back to the producer, which writes the
//      metas (and, calibrating, the codebooks' headers) 32 tensors at a
//      time, one lane each, so that their scalar work runs side by side.
// The output is byte for byte that of the general kernels (enc_main,
// enc_place, enc_regen; cal_hist; ce_main).
//
// Routing: the host takes this path for a table whose tensors average at
// most two tiles; the prepare kernel then sets WsHeader::large if some tensor
// has more than kSmallMax elements, in which case these kernels return at
// once and the general kernels, launched after them, do the work (they
// return at once otherwise).
#include <cstddef>

#include "sz_chunk.cuh"
#include "sz_count.cuh"
#include "sz_internal.h"

namespace sz {
namespace {

constexpr uint32_t kSmallChunks = kSmallMax / kChunk;  // 16
constexpr int kGroupWarps = 8;
constexpr int kGroupThreads = kGroupWarps * 32;  // 256: one thread per exponent bin
// Groups of 8 warps: 2 beside the counters when calibrating, 3 otherwise
// (with the producer, 25 warps at 80 registers a thread).
template <bool CALIBRATE>
__host__ __device__ constexpr uint32_t groups_of() { return CALIBRATE ? 2u : 3u; }
template <bool CALIBRATE>
__host__ __device__ constexpr uint32_t threads_of() { return (groups_of<CALIBRATE>() * kGroupWarps + 1u) * 32u; }
constexpr uint32_t kRecs = 64;  // finished tensors awaiting their meta
constexpr unsigned FULL = 0xFFFFFFFFu;
constexpr uint32_t kNoItem = 0xFFFFFFFFu;
static_assert(kGroupThreads == 256, "one thread per exponent bin");
// Whole-tensor buffers in the ring: 4 beside the two groups' 32 KiB of
// counters when calibrating, 6 otherwise.
template <bool CALIBRATE>
__host__ __device__ constexpr uint32_t small_bufs() { return CALIBRATE ? 4u : 6u; }

// A tensor of the ring: what a group needs of it (filled by the producer with
// the tensor's data, so that no global round trip lies on the group's path)
// and what the producer needs afterwards to write its meta.
struct SmallSlot {
  sz_item it;             // the table entry
  uint32_t i;             // its index (kNoItem: the CTA has no more tensors)
  uint32_t flags;         // the prepare pass's flags for it
  uint32_t cal_ok;        // calibrate: the count pass may run on it
  uint32_t load;          // its data (and, encoding alone, its codebook) were copied
};

// What the producer needs of a finished tensor to write its meta (and,
// calibrating, its codebook's header), written by its group.
struct SmallRec {
  uint32_t e;       // escapes
  uint32_t status;  // the prepare pass's flags | what encoding found (capacity)
  uint32_t top;     // calibrated here: elements whose exponent got a code
  uint32_t n_top;   // calibrated here: codes in use; 0xFFFFFFFF otherwise
};

// A group's own scratch.
template <bool CALIBRATE>
struct SmallGroup {
  uint32_t cnt[CALIBRATE ? 256 * 32 : 1];      // calibrate: [bin][lane] exponent counters
  alignas(16) uint32_t key[CALIBRATE ? 8 : 1][32];  // calibrate: warp w's non-zero bins, compacted
  alignas(16) uint32_t wcnt[8];                // calibrate: how many
  alignas(16) uint8_t lut[CALIBRATE ? 256 : 1];     // calibrate: the enc_lut
  uint8_t dl[16];                              // calibrate: the dec_lut
  uint32_t ccnt[2][kSmallChunks];              // escapes per chunk, by the parity of the group's tensor
};

template <bool CALIBRATE>
struct SmallShared {
  static constexpr uint32_t kBufs = small_bufs<CALIBRATE>();
  alignas(128) uint16_t x[kBufs][kSmallMax];            // the ring of tensors
  alignas(16) sz_codebook cb[CALIBRATE ? 1 : kBufs];    // encoding alone: each tensor's codebook
  SmallSlot slot[kBufs];                                // the tensor of x[b]
  SmallGroup<CALIBRATE> grp[groups_of<CALIBRATE>()];
  SmallRec rec[kRecs];    // tensor k of the CTA at k % kRecs
  uint64_t full[kBufs];   // x[b], cb[b] and slot[b] are filled
  uint64_t empty[kBufs];  // the 8 warps of the group done with x[b] have released it
};
static_assert(sizeof(sz_codebook) % 16 == 0, "copied by TMA");

// Which elements of the lane's 8 per row (4 rows of 256) of a chunk are
// escapes: element 8 lane + k of row r at bit 8 (k & 3) + 2 r + (k >> 2), as
// encode_chunk8 keeps them.
struct ChunkFlags {
  uint32_t lane_esc;
  uint32_t total;  // the chunk's escapes (warp-uniform)
};

// Split + pack of chunk c (elements [1024 c, 1024 c + nvalid)) of the tensor
// in xs: pk and sm written to the payload, escapes flagged.  Lane l takes
// elements 256 r + 8 l .. 256 r + 8 l + 7 of rows r = 0..3; an element past
// nvalid has code 0 (the odd-n pad nibble) and no sm byte.
__device__ ChunkFlags small_pack(const uint16_t* xs, const uint8_t* lut, uint32_t c, uint32_t nvalid, uint8_t* payload,
                                 uint64_t off_sm, uint32_t lane) {
  const uint32_t e0 = c * kChunk + lane * 8u;  // element of this lane in row 0
  const uint16_t* xw = xs + e0;
  uint8_t* pkw = payload + (e0 >> 1);
  uint8_t* smw = payload + off_sm + e0;
  const bool full = nvalid == kChunk;
  const bool sm8 = (off_sm & 7u) == 0;
  uint32_t lane_esc = 0;
#pragma unroll
  for (uint32_t row = 0; row < 4; ++row) {
    const uint32_t first = row * 256u + lane * 8u;  // chunk-local element
    const uint32_t nv = full ? 8u : (first >= nvalid ? 0u : (nvalid - first < 8u ? nvalid - first : 8u));
    const uint4 v = *reinterpret_cast<const uint4*>(xw + row * 256);
    const uint32_t a0 = v.x << 1, a1 = v.y << 1, a2 = v.z << 1, a3 = v.w << 1;
    uint32_t lo = uint32_t(lut[__byte_perm(a0, 0, 0x4441)]) | (uint32_t(lut[__byte_perm(a0, 0, 0x4443)]) << 8) |
                  (uint32_t(lut[__byte_perm(a1, 0, 0x4441)]) << 16) | (uint32_t(lut[__byte_perm(a1, 0, 0x4443)]) << 24);
    uint32_t hi = uint32_t(lut[__byte_perm(a2, 0, 0x4441)]) | (uint32_t(lut[__byte_perm(a2, 0, 0x4443)]) << 8) |
                  (uint32_t(lut[__byte_perm(a3, 0, 0x4441)]) << 16) | (uint32_t(lut[__byte_perm(a3, 0, 0x4443)]) << 24);
    if (nv < 8u) {  // elements past the tensor: code 0, no escape
      lo &= nv >= 4u ? 0xFFFFFFFFu : ((1u << (8u * nv)) - 1u);
      hi &= nv >= 8u ? 0xFFFFFFFFu : (nv <= 4u ? 0u : ((1u << (8u * (nv - 4u))) - 1u));
    }
    lane_esc |= (((lo >> 4) & 0x01010101u) | ((hi >> 3) & 0x02020202u)) << (2 * row);
    const uint32_t clo = lo & 0x0F0F0F0Fu, chi = hi & 0x0F0F0F0Fu;
    const uint32_t tlo = clo | (clo >> 4), thi = chi | (chi >> 4);
    const uint32_t pk4 = __byte_perm(tlo, thi, 0x6420);
    const uint32_t s01 = sm_quad(v.x, v.y);
    const uint32_t s23 = sm_quad(v.z, v.w);
    if (nv == 8u) {
      *reinterpret_cast<uint32_t*>(pkw + row * 128) = pk4;
      if (sm8) {
        *reinterpret_cast<uint2*>(smw + row * 256) = make_uint2(s01, s23);
      } else {
        *reinterpret_cast<uint32_t*>(smw + row * 256) = s01;
        *reinterpret_cast<uint32_t*>(smw + row * 256 + 4) = s23;
      }
    } else if (nv > 0u) {
      for (uint32_t q = 0; 2u * q < nv; ++q) pkw[row * 128 + q] = uint8_t(pk4 >> (8u * q));
      for (uint32_t k = 0; k < nv; ++k) smw[row * 256 + k] = uint8_t((k < 4u ? s01 : s23) >> (8u * (k & 3u)));
    }
  }
  ChunkFlags f;
  f.lane_esc = lane_esc;
  f.total = __reduce_add_sync(FULL, uint32_t(__popc(lane_esc)));
  return f;
}

// The escapes of chunk c (flags as small_pack left them), at global indices
// o, o + 1, ... in element order (row, lane, k): chunk_id c, the chunk-local
// position, the exponent byte from xs.  Rows where no lane has two escapes
// take one ballot; others a warp prefix of the lanes' counts.
__device__ void small_emit(const uint16_t* xs, uint32_t c, const ChunkFlags& f, uint32_t o, uint32_t e, uint8_t* cid_p,
                           uint8_t* lpos_p, uint8_t* ev_p, uint32_t lane) {
  if (f.total == 0) return;
  const uint16_t* xc = xs + c * kChunk;
  uint32_t run = o;
#pragma unroll
  for (uint32_t row = 0; row < 4; ++row) {
    const uint32_t m = (f.lane_esc >> (2 * row)) & 0x03030303u;
    if (__ballot_sync(FULL, m != 0) == 0) continue;  // no escape in this row
    const uint32_t m0 = m & 0x01010101u, m1 = (m >> 1) & 0x01010101u;
    // bit k: element 8 lane + k of the row
    const uint32_t bits = (((m0 * 0x00204081u) >> 21) & 0xFu) | ((((m1 * 0x00204081u) >> 21) & 0xFu) << 4);
    uint32_t total;
    uint32_t pos = run + warp_prefix(uint32_t(__popc(bits)), lane, &total);
    for (uint32_t b = bits; b; b &= b - 1) {
      const uint32_t elem = row * 256u + lane * 8u + uint32_t(__ffs(b) - 1);  // chunk-local
      if (pos < e) {
        *reinterpret_cast<uint32_t*>(cid_p + 4ull * pos) = c;
        *reinterpret_cast<uint16_t*>(lpos_p + 2ull * pos) = uint16_t(elem);
        ev_p[pos] = uint8_t(xc[elem] >> 7);
      }
      ++pos;
    }
    run += total;
  }
}

static_assert(sizeof(SmallShared<true>) <= 227u * 1024u && sizeof(SmallShared<false>) <= 227u * 1024u,
              "one CTA's shared memory");

// The producer's part of the CTA's tensors [j0, j1) (at most 32, released by
// their groups): lane l writes the meta -- and, calibrated here, the
// codebook's header -- of tensor j0 + l, so that the scalar work of 32
// tensors runs side by side.
template <bool CALIBRATE>
__device__ void small_finalize(const Items& items, const EncWs& ws, const SmallRec* rec, uint32_t j0, uint32_t j1,
                               uint32_t lane) {
  const uint32_t j = j0 + lane;
  if (j >= j1) return;
  const sz_item it = items.table[blockIdx.x + uint64_t(j) * gridDim.x];
  const SmallRec r = rec[j % kRecs];
  const uint64_t n = (r.status & SZ_FLAG_SIZE) ? 0 : it.n;
  double coverage;
  if (CALIBRATE && r.n_top != 0xFFFFFFFFu) {
    coverage = ratio_rn(r.top, uint32_t(it.n));  // n <= kSmallMax
    sz_codebook* cb = it.codebook;
    cb->n_top = r.n_top;
    cb->reserved0 = 0;
    cb->top_count = r.top;
    cb->n = it.n;
    cb->coverage = coverage;
  } else {
    coverage = codebook_coverage(it);
  }
  finish_meta(ws, it, layout_of(n, r.e), n, r.e, r.status, coverage);
}

// CALIBRATE: sz_calibrate_encode_many (cal_done: the count pass's validity
// marks of ce_prepare); else sz_encode_many (the codebooks are given).
template <bool CALIBRATE>
__global__ void __launch_bounds__(threads_of<CALIBRATE>(), 1)
    small_main(const __grid_constant__ Items items, EncWs ws, const uint32_t* cal_done) {
  using Shared = SmallShared<CALIBRATE>;
  constexpr uint32_t kBufs = Shared::kBufs;
  constexpr uint32_t kGroups = groups_of<CALIBRATE>();
  constexpr uint32_t kThreads = threads_of<CALIBRATE>();
  constexpr uint32_t kProducer = kGroups * kGroupWarps;  // the producer warp
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
  pdl_wait();  // the prepare kernel's checks and marks
  if (ws.hdr->large || (ws.hdr->flags & SZ_FLAG_ITEMS)) return;

  if (CALIBRATE)
    for (uint32_t w = tid; w < kGroups * 256 * 32; w += kThreads) sh.grp[w / (256 * 32)].cnt[w % (256 * 32)] = 0;
  if (tid == 0) {
    for (uint32_t b = 0; b < kBufs; ++b) {
      mbar_init(&sh.full[b], 1 + 32);
      mbar_init(&sh.empty[b], kGroupWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t G = gridDim.x;

  if (warp == kProducer) {
    // ---------------------------------------------------------------- producer warp
    // Tensor k into buffer k % kBufs once the group done with tensor
    // j = k - kBufs has released it (and j's meta is written); a flagged or
    // empty tensor lands as no bytes; after the CTA's K tensors, one kNoItem
    // slot per group; then the metas of the tensors still in the ring.
    const uint32_t K = blockIdx.x < items.count ? (items.count - 1u - blockIdx.x) / G + 1u : 0u;
    auto release = [&](uint32_t j) -> bool {  // waits until tensor j's group is done with it
      const uint32_t b = j % kBufs;
      if (!__all_sync(FULL, mbar_wait(&sh.empty[b], (j / kBufs) & 1u))) {
        if (lane == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
        return false;
      }
      if (j + 1 == K || (j + 1) % 32u == 0) small_finalize<CALIBRATE>(items, ws, sh.rec, j & ~31u, j + 1, lane);
      return true;
    };
    // What tensor k needs from global memory, fetched kAhead tensors early by
    // one load per lane: lanes 0..15 the words of its table entry, lane 16
    // its flags, lane 17 its count-pass mark.
    constexpr uint32_t kAhead = 4;
    static_assert(sizeof(sz_item) == 64, "16 words");
    auto fetch = [&](uint32_t k) -> uint32_t {
      if (k >= K) return 0u;
      const uint32_t i = blockIdx.x + k * G;
      if (lane < 16) return reinterpret_cast<const uint32_t*>(items.table + i)[lane];
      if (lane == 16) return ws.item_flags[i];
      if (CALIBRATE && lane == 17) return cal_done[i];
      return 0u;
    };
    auto word64 = [&](uint32_t v, size_t offset) -> uint64_t {
      const uint32_t lo = __shfl_sync(FULL, v, uint32_t(offset / 4)), hi = __shfl_sync(FULL, v, uint32_t(offset / 4 + 1));
      return (uint64_t(hi) << 32) | lo;
    };
    auto fill = [&](uint32_t k, uint32_t v) {
      const uint32_t b = k % kBufs;
      const uint32_t i = k < K ? blockIdx.x + k * G : kNoItem;
      SmallSlot& sl = sh.slot[b];
      uint32_t bytes = 0, cb_bytes = 0;
      const uint16_t* src = nullptr;
      const sz_codebook* cb_src = nullptr;
      if (i != kNoItem) {  // warp-uniform
        if (lane < 16) reinterpret_cast<uint32_t*>(&sl.it)[lane] = v;
        const uint32_t flags = __shfl_sync(FULL, v, 16);
        // calibrating, a tensor whose only faults are on the encode side
        // still gets its codebook, as in the general kernels
        const bool cal_ok = CALIBRATE && __shfl_sync(FULL, v, 17) == 0u;
        const uint64_t n = word64(v, offsetof(sz_item, n));
        const bool load = (CALIBRATE ? cal_ok : flags == 0) && n > 0 && n <= kSmallMax;
        if (load) {
          bytes = uint32_t(n) * 2u;
          src = reinterpret_cast<const uint16_t*>(word64(v, offsetof(sz_item, x)));
          if (!CALIBRATE) {
            cb_bytes = sizeof(sz_codebook);
            cb_src = reinterpret_cast<const sz_codebook*>(word64(v, offsetof(sz_item, codebook)));
          }
        }
        if (lane == 0) {
          sl.flags = flags;
          sl.cal_ok = cal_ok;
          sl.load = load;
        }
      }
      if (lane == 0) sl.i = i;
      __syncwarp();  // the slot is written before the barrier's arrivals
      const uint32_t bulk = bytes & ~15u;
      if (lane == 0) {
        mbar_arrive_expect_tx(&sh.full[b], bulk + cb_bytes);
        if (bulk) bulk_g2s(sh.x[b], src, bulk, &sh.full[b]);
        if (cb_bytes) bulk_g2s(&sh.cb[CALIBRATE ? 0 : b], cb_src, cb_bytes, &sh.full[b]);
      } else if (lane == 1 && bytes > bulk) {
        cp_async16_zfill(reinterpret_cast<uint8_t*>(sh.x[b]) + bulk, reinterpret_cast<const uint8_t*>(src) + bulk,
                         bytes - bulk);
      }
      cp_async_mbar_arrive_noinc(&sh.full[b]);
    };
    uint32_t ahead[kAhead];
#pragma unroll
    for (uint32_t d = 0; d < kAhead; ++d) ahead[d] = fetch(d);
    for (uint32_t k0 = 0; k0 < K + kGroups; k0 += kAhead) {
#pragma unroll
      for (uint32_t d = 0; d < kAhead; ++d) {
        const uint32_t k = k0 + d;
        if (k < K + kGroups) {
          if (k >= kBufs && !release(k - kBufs)) return;
          fill(k, ahead[d]);
          ahead[d] = fetch(k + kAhead);
        }
      }
    }
    // the tensors whose buffers were not taken again
    for (uint32_t j = (K + kGroups > kBufs ? K + kGroups - kBufs : 0u); j < K; ++j)
      if (!release(j)) return;
    return;
  }

  // ------------------------------------------------------------------ consumer groups
  const uint32_t g = warp / kGroupWarps;
  const uint32_t gw = warp % kGroupWarps;   // warp within the group
  const uint32_t gt = tid % kGroupThreads;  // thread within the group
  const uint32_t bar_id = 1u + g;
  SmallGroup<CALIBRATE>& my = sh.grp[g];
  for (uint32_t k = g;; k += kGroups) {
    const uint32_t b = k % kBufs;
    const bool ok = mbar_wait(&sh.full[b], (k / kBufs) & 1u);
    if (named_bar_red_or(bar_id, kGroupThreads, !ok)) {
      if (gt == 0) set_flag(ws.hdr, SZ_FLAG_TIMEOUT);
      break;
    }
    SmallSlot& sl = sh.slot[b];
    if (sl.i == kNoItem) break;
    const sz_item& it = sl.it;
    const uint32_t flags = sl.flags;
    const uint64_t n = (flags & SZ_FLAG_SIZE) ? 0 : it.n;
    const uint16_t* xs = sh.x[b];
    SmallRec& rec = sh.rec[k % kRecs];
    if constexpr (CALIBRATE) {
      if (sl.cal_ok && sl.load) {
        if (gt == 0) rec.top = 0;
        // 1. histogram (thread gt keeps bin gt), then the rank of each
        // non-zero bin among all (count desc, value asc) as in select_top16:
        // keys count << 8 | (255 - bin), count <= 16384
        char* col = reinterpret_cast<char*>(my.cnt) + lane * 4;
        count_tile(xs, n < kTile ? uint32_t(n) : kTile, col, gt);
        if (n > kTile) count_tile(xs + kTile, uint32_t(n - kTile), col, gt);
        named_bar_sync(bar_id, kGroupThreads);
        const uint32_t hb = take_bin(my.cnt, gt);
        const uint32_t key = hb ? (hb << 8) | (255u - gt) : 0u;
        const uint32_t nzm = __ballot_sync(FULL, hb != 0);
        my.key[gw][lane] = 0u;
        __syncwarp();
        if (hb) my.key[gw][__popc(nzm & ((1u << lane) - 1u))] = key;
        if (lane == 0) my.wcnt[gw] = uint32_t(__popc(nzm));
        if (gt < 16) my.dl[gt] = 0;
        named_bar_sync(bar_id, kGroupThreads);
        uint32_t rank = 0, total = 0;
#pragma unroll
        for (uint32_t w = 0; w < kGroupWarps; ++w) {
          const uint32_t c = my.wcnt[w];
          total += c;
          if (hb) {
            const uint4* kw = reinterpret_cast<const uint4*>(my.key[w]);
            for (uint32_t q = 0; 4 * q < c; ++q) {
              const uint4 v = kw[q];  // entries past c are 0 and never rank above
              rank += uint32_t(v.x > key) + uint32_t(v.y > key) + uint32_t(v.z > key) + uint32_t(v.w > key);
            }
          }
        }
        const bool coded = hb && rank < 16;
        my.lut[gt] = coded ? uint8_t(rank) : uint8_t(kEscape);
        if (coded) my.dl[rank] = uint8_t(gt);
        uint32_t top = coded ? hb : 0u;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) top += __shfl_xor_sync(FULL, top, d);
        if (lane == 0 && top) atomicAdd(&rec.top, uint32_t(top));
        if (gt == 0) rec.n_top = total < 16 ? total : 16u;
        named_bar_sync(bar_id, kGroupThreads);
        it.codebook->enc_lut[gt] = my.lut[gt];
        if (gt < 16) it.codebook->dec_lut[gt] = my.dl[gt];
      }
    }
    const uint8_t* lut = CALIBRATE ? my.lut : sh.cb[CALIBRATE ? 0 : b].enc_lut;
    uint32_t* const ccnt = my.ccnt[(k / kGroups) & 1u];
    // 2. split + pack, escape flags
    const uint32_t chunks = uint32_t((n + kChunk - 1) / kChunk);
    const uint64_t off_sm = layout_of(n, 0).off_sm;
    ChunkFlags f0{0u, 0u}, f1{0u, 0u};
    if (!flags && n > 0) {
      if (gw < chunks) {
        const uint32_t nv = (n - uint64_t(gw) * kChunk < kChunk) ? uint32_t(n - uint64_t(gw) * kChunk) : kChunk;
        f0 = small_pack(xs, lut, gw, nv, it.payload, off_sm, lane);
      }
      if (gw + kGroupWarps < chunks) {
        const uint32_t c = gw + kGroupWarps;
        const uint32_t nv = (n - uint64_t(c) * kChunk < kChunk) ? uint32_t(n - uint64_t(c) * kChunk) : kChunk;
        f1 = small_pack(xs, lut, c, nv, it.payload, off_sm, lane);
      }
      if (lane == 0) {
        ccnt[gw] = f0.total;
        ccnt[gw + kGroupWarps] = f1.total;
      }
    }
    named_bar_sync(bar_id, kGroupThreads);
    // 3. escapes at their final offsets
    uint32_t e = 0, status = flags;
    const uint32_t cc = (!flags && n > 0 && lane < kSmallChunks) ? ccnt[lane] : 0u;
    e = __reduce_add_sync(FULL, cc);
    const Layout l = layout_of(n, e);
    if (!status && l.comp_bytes > it.capacity) status |= SZ_FLAG_CAPACITY;
    if (!status && e > 0) {
      const uint32_t o0 = __reduce_add_sync(FULL, lane < gw ? cc : 0u);
      const uint32_t o1 = __reduce_add_sync(FULL, lane < gw + kGroupWarps ? cc : 0u);
      uint8_t* const cid_p = it.payload + l.off_cid;
      uint8_t* const lpos_p = it.payload + l.off_lpos;
      uint8_t* const ev_p = it.payload + l.off_ev;
      small_emit(xs, gw, f0, o0, e, cid_p, lpos_p, ev_p, lane);
      small_emit(xs, gw + kGroupWarps, f1, o1, e, cid_p, lpos_p, ev_p, lane);
    }
    // 4. pads; the producer writes the meta once the 8 warps have released the buffer
    finish_pads(it, l, n, e, status, gt);
    if (gt == 0) {
      rec.e = e;
      rec.status = status;
      if (!(CALIBRATE && sl.cal_ok && sl.load)) rec.n_top = 0xFFFFFFFFu;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[b]);
  }
}

}  // namespace

bool small_route(const Items& items) {
  return items.table != nullptr && items.count > 0 && items.total_tiles <= 2ull * items.count;
}

cudaError_t launch_small(const Items& items, const EncWs& ws, const uint32_t* cal_done, cudaStream_t stream,
                         const DeviceInfo& dev) {
  static thread_local int configured_device = -1;
  const size_t smem_cal = sizeof(SmallShared<true>), smem_enc = sizeof(SmallShared<false>);
  if (configured_device != dev.device) {
    cudaError_t err = cudaFuncSetAttribute(small_main<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_cal));
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(small_main<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_enc));
    if (err != cudaSuccess) return err;
    configured_device = dev.device;
  }
  const uint64_t cap = uint64_t(dev.num_sms);  // one CTA per SM
  const unsigned grid = unsigned(items.count < cap ? items.count : cap);
  if (g_timing.before) cudaEventRecord(g_timing.before, stream);
  const cudaError_t err =
      cal_done ? launch_pdl(small_main<true>, dim3(grid), dim3(threads_of<true>()), smem_cal, stream, items, ws, cal_done)
               : launch_pdl(small_main<false>, dim3(grid), dim3(threads_of<false>()), smem_enc, stream, items, ws, cal_done);
  if (g_timing.after) cudaEventRecord(g_timing.after, stream);
  return err;
}

}  // namespace sz
