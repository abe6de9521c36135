// Device-side building blocks shared by the SplitZip kernels (sm_103a only).
//
// - wire-layout arithmetic of the GPU path (payload offsets, tiles);
// - inline-PTX wrappers for mbarriers, bulk (TMA) copies, cp.async with
//   zero-fill, proxy fences, acquire/release accesses and the global timer;
// - the item table view used by every multi-tensor kernel;
// - the workspace layouts.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "splitzip.h"

namespace sz {

constexpr uint32_t kChunk = SZ_CHUNK_SIZE;          // 1024
constexpr uint32_t kTile = SZ_TILE_ELEMS;           // 8192
constexpr uint32_t kChunksPerTile = kTile / kChunk; // 8
constexpr uint32_t kEscape = SZ_ESCAPE_CODE;        // 16
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // bounded waits give up after 2 s
constexpr uint32_t kSmallMax = 2 * kTile;           // elements of a tensor the small-tensor kernels hold whole

// ------------------------------------------------------------------ layout
// Wire layout of "splitzip_codec.py" assemble_payload: pk | sm | chunk_id |
// local_pos | esc_val, each section start rounded up to 4 bytes except
// local_pos, which follows chunk_id directly.
struct Layout {
  uint64_t n_pairs, off_sm, off_cid, off_lpos, off_ev, comp_bytes;
};

__host__ __device__ inline uint64_t round_up4(uint64_t v) { return (v + 3u) & ~uint64_t(3); }
__host__ __device__ inline uint64_t tiles_of(uint64_t n) { return (n + kTile - 1) / kTile; }

__host__ __device__ inline Layout layout_of(uint64_t n, uint64_t n_esc) {
  Layout l;
  l.n_pairs = (n + 1) >> 1;
  l.off_sm = round_up4(l.n_pairs);
  l.off_cid = round_up4(l.off_sm + n);
  l.off_lpos = l.off_cid + 4 * n_esc;
  l.off_ev = round_up4(l.off_lpos + 2 * n_esc);
  l.comp_bytes = l.off_ev + n_esc;
  return l;
}

// ------------------------------------------------------------------ items
// A kernel sees its tensors either through a device item table or, for the
// single-tensor entry points, through one item passed by value.
struct Items {
  const sz_item* table;  // nullptr: use `one`
  sz_item one;
  uint32_t count;
  uint64_t total_tiles;
};

__device__ __forceinline__ const sz_item& item_at(const Items& it, uint32_t i) {
  return it.table ? it.table[i] : it.one;
}

// Index of the item whose tile range holds global tile `tile` (items are in
// ascending tile_begin order; empty items own no tile).
__device__ inline uint32_t find_item(const Items& it, uint64_t tile) {
  if (it.table == nullptr) return 0;
  uint32_t lo = 0, hi = it.count;  // answer in [lo, hi)
  while (hi - lo > 1) {
    uint32_t mid = (lo + hi) >> 1;
    if (it.table[mid].tile_begin <= tile) lo = mid; else hi = mid;
  }
  // skip empty items that share the same tile_begin
  while (lo + 1 < it.count && it.table[lo + 1].tile_begin <= tile) ++lo;
  return lo;
}

// Tile -> item maps (filled by the prepare kernels) let a producer resolve any
// tile with one load: in the decode workspace of every table of more than one
// item, in the encode workspace of tables of more than kEncMapItems items
// (smaller ones are searched directly, and only when a run of tiles leaves
// the current item).
constexpr uint32_t kEncMapItems = 256;
__host__ __device__ inline bool dec_uses_tile_map(uint32_t count) { return count > 1; }
__host__ __device__ inline bool enc_uses_tile_map(uint32_t count) { return count > kEncMapItems; }
__host__ __device__ inline uint64_t tile_map_bytes(bool used, uint64_t tiles) {
  return used ? ((tiles * 4 + 255u) & ~uint64_t(255)) : 0;
}

// ------------------------------------------------------------------ workspace
// Every workspace starts with this header (256 bytes).
struct WsHeader {
  uint32_t flags;        // SZ_FLAG_* bits
  uint32_t pad0;
  unsigned long long ticket;  // dynamic tile counter (encode)
  uint32_t tiles_differ;      // in-place decode: set when the tensors' tile counts are not all equal
  uint32_t dense;             // encode: some chunk had too many escapes to stage (kStageMax)
  uint32_t large;             // small-tensor route: some tensor is larger than kSmallMax
  uint32_t reserved[57];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

__host__ __device__ inline uint64_t round_up256(uint64_t v) { return (v + 255u) & ~uint64_t(255); }

// calibrate: header | hist[count][256] u32 | done[count] u32
struct CalWs {
  WsHeader* hdr;
  uint32_t* hist;
  uint32_t* done;
};
__host__ __device__ inline uint64_t cal_ws_bytes(uint32_t count) {
  return 256 + round_up256(uint64_t(count) * 1024) + round_up256(uint64_t(count) * 4);
}
__host__ __device__ inline CalWs cal_ws(void* base, uint32_t count) {
  char* p = static_cast<char*>(base);
  CalWs w;
  w.hdr = reinterpret_cast<WsHeader*>(p);
  w.hist = reinterpret_cast<uint32_t*>(p + 256);
  w.done = reinterpret_cast<uint32_t*>(p + 256 + round_up256(uint64_t(count) * 1024));
  return w;
}

// encode: header | item_flags[count] u32 | item_esc[count] u32 (escape total) |
//         seg_ticket[count] u32 | status[total_tiles] u64 (segment lookback words,
//         at each segment's first tile) | chunk_cnt[total_tiles * 8] u16 |
//         escape staging[total_tiles * 8192] u32 (chunk-local position | esc_val << 16) |
//         tile_item[total_tiles] u32 (tables of more than kEncMapItems items)
// Staging slot of chunk c (global chunk index tile * 8 + chunk) starts at
// entry c * 1024 and holds the chunk's escapes in element order, one word each.
struct EncWs {
  WsHeader* hdr;
  uint32_t* item_flags;
  uint32_t* item_esc;
  uint32_t* seg_ticket;
  unsigned long long* status;
  uint16_t* chunk_cnt;
  uint32_t* stage;
  uint32_t* tile_item;
  double gate;              // coverage gate (< 0: none)
  sz_gate_report* report;   // build report of a gated call, or nullptr
  bool small;               // the small-tensor kernels were launched first: the general
                            // kernels work only if the prepare pass found a large tensor
};
// Bytes of the encode workspace after its header (map excluded).
__host__ __device__ inline uint64_t enc_body_bytes(uint32_t count, uint64_t tiles) {
  return 3 * round_up256(uint64_t(count) * 4) + round_up256(tiles * 8) + round_up256(tiles * 16) +
         round_up256(tiles * kTile * 4);
}
__host__ __device__ inline uint64_t enc_ws_bytes(uint32_t count, uint64_t tiles) {
  return 256 + enc_body_bytes(count, tiles) + tile_map_bytes(enc_uses_tile_map(count), tiles);
}
// The encode workspace with its header at hdr and its body at `body`.
__host__ __device__ inline EncWs enc_ws_at(WsHeader* hdr, void* body, uint32_t count, uint64_t tiles,
                                           uint32_t* tile_item) {
  char* p = static_cast<char*>(body);
  EncWs w;
  w.hdr = hdr;
  w.item_flags = reinterpret_cast<uint32_t*>(p);
  p += round_up256(uint64_t(count) * 4);
  w.item_esc = reinterpret_cast<uint32_t*>(p);
  p += round_up256(uint64_t(count) * 4);
  w.seg_ticket = reinterpret_cast<uint32_t*>(p);
  p += round_up256(uint64_t(count) * 4);
  w.status = reinterpret_cast<unsigned long long*>(p);
  p += round_up256(tiles * 8);
  w.chunk_cnt = reinterpret_cast<uint16_t*>(p);
  p += round_up256(tiles * 16);
  w.stage = reinterpret_cast<uint32_t*>(p);
  w.tile_item = tile_item;
  w.gate = -1.0;
  w.report = nullptr;
  w.small = false;
  return w;
}
__host__ __device__ inline EncWs enc_ws(void* base, uint32_t count, uint64_t tiles) {
  char* p = static_cast<char*>(base);
  uint32_t* map = enc_uses_tile_map(count)
                      ? reinterpret_cast<uint32_t*>(p + 256 + enc_body_bytes(count, tiles))
                      : nullptr;
  return enc_ws_at(reinterpret_cast<WsHeader*>(p), p + 256, count, tiles, map);
}

// fused calibrate + encode: header | hist[count][256] u32 | done[count] u32 |
//   ready[count] u32 (codebook written) | group_first[groups + 1] u64 |
//   group_ticket[groups + 1] u32 | tile_item[tiles] u32 | encode body.
//   Tensors are taken in groups by first tile, kGroupTiles tiles (32 MiB of
//   BF16) per group.
constexpr uint64_t kGroupTiles = 2048;
__host__ __device__ inline uint64_t ce_groups(uint64_t tiles) { return (tiles + kGroupTiles - 1) / kGroupTiles; }
struct CeWs {
  CalWs cal;
  EncWs enc;
  uint32_t* ready;
  uint64_t* group_first;
  uint32_t* group_ticket;
};
__host__ __device__ inline uint64_t ce_ws_bytes(uint32_t count, uint64_t tiles) {
  return 256 + round_up256(uint64_t(count) * 1024) + 2 * round_up256(uint64_t(count) * 4) +
         round_up256((ce_groups(tiles) + 1) * 8) + round_up256((ce_groups(tiles) + 1) * 4) + round_up256(tiles * 4) +
         enc_body_bytes(count, tiles);
}
__host__ __device__ inline CeWs ce_ws(void* base, uint32_t count, uint64_t tiles) {
  char* p = static_cast<char*>(base);
  CeWs w;
  w.cal = cal_ws(base, count);  // header, hist, done
  p += 256 + round_up256(uint64_t(count) * 1024) + round_up256(uint64_t(count) * 4);
  w.ready = reinterpret_cast<uint32_t*>(p);
  p += round_up256(uint64_t(count) * 4);
  w.group_first = reinterpret_cast<uint64_t*>(p);
  p += round_up256((ce_groups(tiles) + 1) * 8);
  w.group_ticket = reinterpret_cast<uint32_t*>(p);
  p += round_up256((ce_groups(tiles) + 1) * 4);
  uint32_t* map = reinterpret_cast<uint32_t*>(p);
  p += round_up256(tiles * 4);
  w.enc = enc_ws_at(w.cal.hdr, p, count, tiles, map);
  return w;
}

// out-of-place decode: the 256-byte header only.  Each CTA of the decode
// kernel validates the tensors of its tiles and finds its tiles' escape
// ranges itself, so there is nothing to prepare.
__host__ __device__ constexpr uint64_t dec_ws_bytes(uint32_t /*count*/, uint64_t /*tiles*/) { return 256; }

// in-place decode, prepared by dec_prepare: header | item_flags[count] u32 |
// ranges[total_tiles] (k0, k1) u32x2 | tile_item[total_tiles] u32 (tables of
// more than one item) | read_done | stash (see ip_ws)
struct DecWs {
  WsHeader* hdr;
  uint32_t* item_flags;
  uint2* ranges;
  uint32_t* tile_item;
  uint32_t* read_done;  // in-place decode: per tile, its in-place input has been read
  uint8_t* stash;       // in-place decode: the bytes copied aside
  bool small_done;      // out of place: dec_small ran first; dec_flat takes only what it left
};
__host__ __device__ inline uint64_t prep_ws_bytes(uint32_t count, uint64_t tiles) {
  return 256 + round_up256(uint64_t(count) * 4) + round_up256(tiles * 8) + tile_map_bytes(dec_uses_tile_map(count), tiles);
}
__host__ __device__ inline DecWs prep_ws(void* base, uint32_t count, uint64_t tiles) {
  char* p = static_cast<char*>(base);
  DecWs w;
  w.hdr = reinterpret_cast<WsHeader*>(p);
  p += 256;
  w.item_flags = reinterpret_cast<uint32_t*>(p);
  p += round_up256(uint64_t(count) * 4);
  w.ranges = reinterpret_cast<uint2*>(p);
  p += round_up256(tiles * 8);
  w.tile_item = dec_uses_tile_map(count) ? reinterpret_cast<uint32_t*>(p) : nullptr;
  w.read_done = nullptr;
  w.stash = nullptr;
  w.small_done = false;
  return w;
}
// the out-of-place decode's view of its workspace: the header alone
__host__ __device__ inline DecWs dec_ws(void* base) {
  DecWs w;
  w.hdr = static_cast<WsHeader*>(base);
  w.item_flags = nullptr;
  w.ranges = nullptr;
  w.tile_item = nullptr;
  w.read_done = nullptr;
  w.stash = nullptr;
  w.small_done = false;
  return w;
}

// ------------------------------------------------------------------ in-place slot decode
// The payload occupies the leading comp_bytes of the tensor's own 2n-byte
// output (its slot) and the weight is decoded over it.  Output tile u covers
// slot bytes [16384 u, 16384 u + 2 nt); a payload byte read by tile r and
// overwritten by tile w = byte / 16384 must be read before w stores, so the
// tiles of a tensor are decoded in an order that reads as much as possible in
// place, in three phases (tA = ceil(off_sm / 8192), tB = off_sm / 16384):
//   A  tiles [tA, T), from the top down.  pk bytes of tile t start at 4096 t,
//      under tile t / 4 <= t; sm bytes of tile t >= tA lie under tiles <= t.
//   B  tiles [0, tB), from the top down.  pk as in A; their sm bytes lie
//      under tiles of C, which come later.
//   C  tiles [tB, tA), from the bottom up.  Their sm bytes lie under tiles of
//      C at or above them (off_sm + i >= 2 i for i < off_sm); their pk bytes
//      lie under tile t / 4, of B (or of C below t when tB = 0), which comes
//      before, so they are copied to a stash before the decode, with the
//      escape streams (under tiles of A) -- but those of tile 0, which lie
//      under tile 0 itself.
// The stash is about n / 8 + 7 e bytes (the whole payload is 1.5 n + 7 e).
// A tile stores its output only after the tiles whose in-place bytes lie
// under it have read them (ip_deps); all of them come earlier in the order.
struct IpPhases {
  uint64_t T, tA, tB;
};
__host__ __device__ inline IpPhases ip_phases(uint64_t n, uint64_t off_sm) {
  IpPhases p;
  p.T = (n + kTile - 1) / kTile;
  p.tA = (off_sm + kTile - 1) / kTile;
  if (p.tA > p.T) p.tA = p.T;
  p.tB = off_sm / (2 * kTile);
  if (p.tB > p.tA) p.tB = p.tA;
  return p;
}
// position of tile t in the tensor's decode order, and its inverse
__host__ __device__ inline uint64_t ip_rank(const IpPhases& p, uint64_t t) {
  if (t >= p.tA) return p.T - 1 - t;
  if (t < p.tB) return (p.T - p.tA) + (p.tB - 1 - t);
  return (p.T - p.tA) + p.tB + (t - p.tB);
}
__host__ __device__ inline uint64_t ip_tile_at(const IpPhases& p, uint64_t r) {
  if (r < p.T - p.tA) return p.T - 1 - r;
  r -= p.T - p.tA;
  if (r < p.tB) return p.tB - 1 - r;
  return p.tB + (r - p.tB);
}

// Stash of one tensor: payload bytes [pk_from, pk_to) (the pk bytes of phase
// C, but those of tile 0, which lie under tile 0 itself) at offset 0 and
// [floor16(off_cid), comp_bytes) at esc_off; both keep their payload offsets
// mod 16 (pk_from is a multiple of 4096).
struct IpStash {
  uint64_t pk_from, pk_to;    // payload byte range of the pk part
  uint64_t esc_from, esc_to;  // payload byte range of the escape part (empty without escapes)
  uint64_t esc_off;           // stash offset of the escape part (16-byte multiple)
  uint64_t bytes;             // stash bytes used
};
__host__ __device__ inline IpStash ip_stash(uint64_t n, uint64_t n_esc, uint64_t off_sm, uint64_t off_cid,
                                            uint64_t comp_bytes) {
  const IpPhases p = ip_phases(n, off_sm);
  const uint64_t n_pairs = (n + 1) / 2;
  IpStash s;
  s.pk_from = (p.tB > 0 ? p.tB : 1) * (kTile / 2);
  s.pk_to = p.tA * (kTile / 2) < n_pairs ? p.tA * (kTile / 2) : n_pairs;
  if (s.pk_to < s.pk_from) s.pk_to = s.pk_from;
  s.esc_from = off_cid & ~uint64_t(15);
  s.esc_to = n_esc ? comp_bytes : s.esc_from;
  s.esc_off = (s.pk_to - s.pk_from + 15) & ~uint64_t(15);
  s.bytes = s.esc_off + (s.esc_to - s.esc_from);
  return s;
}

// Stash budget of a tensor of `tiles` tiles: enough for any payload of at
// most 2n bytes (pk part <= min(n_pairs, n / 8 + 8200), escape part
// <= n - off_sm + 15 with off_sm >= n / 2, n <= 8192 tiles).
constexpr uint64_t kIpStashPerTile = 8192;
constexpr uint64_t kIpStashPerItem = 4096 + 256;
__host__ __device__ inline uint64_t ip_stash_at(uint64_t tile_begin, uint32_t item) {
  return tile_begin * kIpStashPerTile + uint64_t(item) * kIpStashPerItem;
}

// Tiles (local indices, inclusive ranges, empty when lo > hi) whose in-place
// bytes lie under output tile u: pk of tiles 4u .. 4u + 3 outside phase C
// (two ranges, below tB and from tA up), and the tiles whose sm bytes meet
// [16384 u, 16384 u + 16384).  Every one of them other than u comes earlier
// in the decode order (ip_rank).
struct IpDeps {
  uint64_t pk_lo, pk_hi, pk2_lo, pk2_hi, sm_lo, sm_hi;
};
__host__ __device__ inline IpDeps ip_deps(uint64_t n, uint64_t off_sm, uint64_t u) {
  const IpPhases p = ip_phases(n, off_sm);
  IpDeps d;
  const uint64_t lo = 4 * u, hi = (4 * u + 3 < p.T) ? 4 * u + 3 : p.T - 1;
  d.pk_lo = lo;
  d.pk_hi = (hi < p.tB) ? hi : p.tB - 1;  // below tB (empty when tB == 0: hi wraps below lo)
  if (p.tB == 0) d.pk_lo = 1, d.pk_hi = 0;
  d.pk2_lo = (lo > p.tA) ? lo : p.tA;
  d.pk2_hi = hi;
  if (lo > hi) d.pk_lo = d.pk2_lo = 1, d.pk_hi = d.pk2_hi = 0;
  const uint64_t w0 = 2 * kTile * u, w1 = w0 + 2 * kTile;  // the output bytes of tile u (at most)
  // tile t's sm bytes [off_sm + 8192 t, off_sm + 8192 t + 8192) meet [w0, w1)
  d.sm_lo = (w0 >= off_sm + kTile) ? (w0 - off_sm - kTile) / kTile + 1 : 0;
  d.sm_hi = (w1 > off_sm) ? (w1 - off_sm - 1) / kTile : 0;
  if (w1 <= off_sm) d.sm_lo = 1, d.sm_hi = 0;
  if (d.sm_hi >= p.T) d.sm_hi = p.T - 1;
  return d;
}

// in-place decode workspace: the prepared layout | read_done[tiles] u32 | stash
__host__ __device__ inline uint64_t ip_ws_bytes(uint32_t count, uint64_t tiles) {
  return prep_ws_bytes(count, tiles) + round_up256(tiles * 4) + tiles * kIpStashPerTile +
         uint64_t(count) * kIpStashPerItem;
}
__host__ __device__ inline DecWs ip_ws(void* base, uint32_t count, uint64_t tiles) {
  DecWs w = prep_ws(base, count, tiles);
  char* p = static_cast<char*>(base) + prep_ws_bytes(count, tiles);
  w.read_done = reinterpret_cast<uint32_t*>(p);
  w.stash = reinterpret_cast<uint8_t*>(p + round_up256(tiles * 4));
  return w;
}

#ifdef __CUDACC__
// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// One bounded probe of the phase: the thread may be suspended in hardware
// (up to kSuspendHintNs) until the phase completes, instead of spinning.
constexpr uint32_t kSuspendHintNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete; gives up
// after kWaitTimeoutNs and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0 && global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// Bulk (TMA) copy global -> shared; completion is reported to `bar` as
// transaction bytes.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// The same with an L2 evict-first policy: lines read once should leave L2
// before lines that other work still has to write back or read again.
__device__ __forceinline__ void bulk_g2s_evict_first(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// Bulk (TMA) copy shared -> global, tracked by the issuing thread's bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Make this thread's generic-proxy writes to shared memory visible to the
// async proxy (before a bulk store reads them).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy global accesses (e.g. an
// acquire that saw another CTA's flag) before its later async-proxy global
// accesses (a bulk store).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// 16-byte cp.async that reads only `src_bytes` (0..16) bytes and zero-fills
// the rest of the destination; nothing beyond src + src_bytes is read.
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

// Arrive on `bar` once all cp.async issued so far by this thread completed
// (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Relaxed GPU-scope accesses: coherent single-copy-atomic 64-bit words with
// no ordering of other memory (enough for a word that carries its own data).
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier over `threads` threads that also returns the OR of `pred`
// across them.
__device__ __forceinline__ bool named_bar_red_or(uint32_t id, uint32_t threads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(uint32_t(pred)), "r"(id), "r"(threads)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void set_flag(WsHeader* h, uint32_t bits) { atomicOr(&h->flags, bits); }

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while the kernel before it in the stream is still running: pdl_wait blocks
// until that kernel has completed and its writes are visible (a no-op when
// the kernel was launched normally), so it comes before any read of what the
// earlier kernel wrote.  pdl_trigger lets the next kernel's CTAs be scheduled
// once every CTA of this one has issued it; it orders nothing, since the next
// kernel waits for this one's completion all the same.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

#endif  // __CUDACC__

}  // namespace sz
