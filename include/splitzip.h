/*
 * splitzip.h -- C ABI of the GB300 (sm_103a) SplitZip lossless BF16 codec.
 *
 * The method (from "splitzip_codec.py", module docstring, and
 * "docs/developer/splitzip.md", "What it does"): view each BF16 value as a
 * 16-bit pattern x; split it into the exponent byte exp = (x >> 7) & 0xFF and
 * the sign + low-7-mantissa byte sm = ((x >> 8) & 0x80) | (x & 0x7F).  A
 * per-tensor codebook maps the 16 most frequent exponents to 4-bit codes; sm is
 * stored verbatim; every element whose exponent is not in the codebook goes to
 * an ordered escape stream with chunk-local positions (chunk = 1024).  Decode
 * rebuilds x = ((sm & 0x80) << 8) | (exp << 7) | (sm & 0x7F) bit for bit.
 *
 * Payload (wire) layout, from "splitzip_codec.py" assemble_payload / PayloadMeta
 * and "docs/developer/splitzip.md" "Invariants common to both routes" item 1;
 * all integers little-endian, align4(v) = (v + 3) & ~3:
 *   off_pk   = 0                          uint8  pk[n_pairs], n_pairs = ceil(n/2)
 *   off_sm   = align4(n_pairs)            uint8  sm[n]
 *   off_cid  = align4(off_sm + n)         int32  chunk_id[n_esc]
 *   off_lpos = off_cid + 4 n_esc          uint16 local_pos[n_esc]
 *   off_ev   = align4(off_lpos + 2 n_esc) uint8  esc_val[n_esc]
 *   comp_bytes = off_ev + n_esc; every pad byte is 0.
 * Conventions this codec fixes (the pages leave them open or disagree):
 *   - element 2i is the LOW nibble of pk[i], element 2i+1 the high nibble
 *     (the pages' pure-PyTorch codec uses the opposite order; a per-byte nibble
 *     swap converts between the two);
 *   - an escaped element is stored in pk as code 0; escapes are listed in
 *     ascending element index (chunk_id non-decreasing);
 *   - Top-16 ties are broken by ascending exponent value;
 *   - n == 0 is valid: empty payload, codebook with no codes, coverage 1.0.
 *
 * Memory and streams.  Every pointer argument is named d_* (device memory) or
 * h_* (host memory).  The library allocates nothing: the caller owns every
 * buffer, including the workspace, whose size the *_workspace_bytes queries
 * give.  All compute calls are asynchronous on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and never synchronise.  A workspace may be
 * reused by calls ordered on one stream; calls that may overlap on the GPU
 * need separate workspaces.
 *
 * Alignment.  Every BF16 input/output and payload pointer must be 16-byte
 * aligned; codebook, meta and item-table pointers 16-byte aligned; workspaces
 * 256-byte aligned.  Violations are rejected with SZ_ERR_ALIGN (single-tensor
 * calls) or flagged on the device with SZ_FLAG_ALIGN (item tables).
 *
 * Errors.  Every call returns an sz_status.  Host-side checks (null pointers,
 * sizes, alignment, workspace size) happen before anything is launched and
 * leave all buffers untouched.  Conditions only the GPU can see (a capacity
 * overrun, a malformed payload, a wait that timed out) never fault the GPU:
 * the kernels skip the offending writes, record SZ_FLAG_* bits in the
 * workspace's status word (and in sz_meta.status for encode), and the caller
 * reads them with sz_workspace_flags after the work completes.
 */
#ifndef SPLITZIP_H
#define SPLITZIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SZ_API __attribute__((visibility("default")))
#else
#define SZ_API
#endif

struct CUstream_st;
typedef struct CUstream_st* sz_stream; /* the same type as cudaStream_t */

#define SZ_VERSION 1
#define SZ_CHUNK_SIZE 1024u     /* escape chunk ("splitzip_codec.py" encode_torch chunk_size) */
#define SZ_TILE_ELEMS 8192u     /* elements per work tile; items start on tile boundaries   */
#define SZ_ESCAPE_CODE 16u      /* enc_lut value of an exponent outside the codebook          */
#define SZ_MAX_ELEMS 4294967295ull       /* largest n per tensor (chunk_id fits int32)      */
#define SZ_MANY_MAX_ITEMS 65535u         /* largest item count of the *_many calls           */

/* Status codes returned by every call. */
typedef enum sz_status {
  SZ_OK = 0,
  SZ_ERR_ARG = 1,        /* null pointer, size out of range, count out of range   */
  SZ_ERR_ALIGN = 2,      /* a pointer breaks the alignment rules above             */
  SZ_ERR_CAPACITY = 3,   /* a host-known size does not fit its buffer             */
  SZ_ERR_META = 4,       /* a host meta disagrees with the wire layout for its n  */
  SZ_ERR_WORKSPACE = 5,  /* workspace null, misaligned or smaller than required   */
  SZ_ERR_CUDA = 6,       /* a CUDA runtime call failed (launch, copy, no device)  */
  SZ_ERR_DEVICE = 7      /* sz_workspace_flags found SZ_FLAG_* bits set           */
} sz_status;

/* Device-side status bits (sz_workspace_flags, sz_meta.status). */
#define SZ_FLAG_CAPACITY 0x01u    /* encode: payload larger than the item's capacity      */
#define SZ_FLAG_META 0x02u        /* decode: meta disagrees with the layout / capacity    */
#define SZ_FLAG_ESCAPE 0x04u      /* decode: an escape points outside its tile or tensor  */
#define SZ_FLAG_TIMEOUT 0x08u     /* a bounded wait gave up (results of the call invalid) */
#define SZ_FLAG_ALIGN 0x10u       /* an item-table pointer breaks the alignment rules     */
#define SZ_FLAG_ITEMS 0x20u       /* item table: tile_begin chain inconsistent            */
#define SZ_FLAG_SIZE 0x40u        /* an item's n is out of range for the call             */

/* sz_meta.status bit that is not an error: the tensor was left uncompressed
 * by the coverage gate of sz_encode_gated_many (its payload holds nothing). */
#define SZ_META_GATED 0x100u

/* Per-tensor codebook ("splitzip_codec.py" SplitZipCodebook and
 * calibrate_codebook).  304 bytes, 16-byte aligned in device memory. */
typedef struct sz_codebook {
  uint8_t enc_lut[256];  /* exponent byte -> code 0..15, or SZ_ESCAPE_CODE (the page's enc_lut_marked) */
  uint8_t dec_lut[16];   /* code -> exponent byte; codes >= n_top hold 0                              */
  uint32_t n_top;        /* min(16, number of distinct exponents)                                     */
  uint32_t reserved0;
  uint64_t top_count;    /* elements whose exponent has a code                                        */
  uint64_t n;            /* elements the codebook was calibrated on                                   */
  double coverage;       /* top_count / n as an IEEE double division; 1.0 when n == 0                 */
} sz_codebook;

/* Payload metadata ("splitzip_codec.py" PayloadMeta).  96 bytes. */
typedef struct sz_meta {
  uint64_t n, n_pairs, n_esc, comp_bytes;
  uint64_t off_pk, off_sm, off_cid, off_lpos, off_ev;
  uint32_t chunk_size;   /* always SZ_CHUNK_SIZE                            */
  uint32_t status;       /* encode: SZ_FLAG_* bits of this tensor (0 = ok)   */
  double coverage;       /* copied from the codebook used to encode          */
  uint64_t reserved1;
} sz_meta;

/* One tensor of a *_many call, in device memory.  64 bytes.
 * Fields a call does not use are ignored (see each call). */
typedef struct sz_item {
  const uint16_t* x;       /* calibrate/encode: n BF16 bit patterns                   */
  uint16_t* out;           /* decode: n BF16 bit patterns written                     */
  uint8_t* payload;        /* encode: written (capacity bytes); decode: read          */
  sz_codebook* codebook;   /* calibrate: written; encode/decode: read                 */
  sz_meta* meta;           /* encode: written; decode: read                           */
  uint64_t n;              /* elements                                                */
  uint64_t capacity;       /* bytes available at payload                              */
  uint64_t tile_begin;     /* *_many only: sum of sz_tiles(n) of the items before it  */
} sz_item;

/* Build report of sz_encode_gated_many (the shard-cache builder's report of
 * "docs/developer/splitzip.md": tensors encoded, tensors skipped for
 * coverage, payload ratio).  64 bytes, in device memory. */
typedef struct sz_gate_report {
  uint64_t tensors_encoded;    /* coverage >= the gate, encoded                        */
  uint64_t tensors_gated;      /* coverage below the gate, left uncompressed           */
  uint64_t raw_bytes_encoded;  /* 2 n summed over the encoded tensors                  */
  uint64_t payload_bytes;      /* comp_bytes summed over the encoded tensors           */
  uint64_t raw_bytes_gated;    /* 2 n summed over the gated tensors                    */
  uint64_t tensors_expanded;   /* encoded tensors whose payload exceeds 2 n            */
  uint64_t escapes;            /* n_esc summed over the encoded tensors                */
  uint64_t tensors_failed;     /* tensors with an error flag (neither encoded nor gated) */
} sz_gate_report;

/* ------------------------------------------------------------------ host-only queries */

SZ_API int sz_version(void);
SZ_API const char* sz_strerror(int status);

/* Tiles of SZ_TILE_ELEMS elements covering n elements: ceil(n / 8192). */
SZ_API uint64_t sz_tiles(uint64_t n);

/* Fills h_meta's sizes and offsets for n elements with n_esc escapes (the
 * wire layout above); status and coverage are set to 0.  SZ_ERR_ARG if
 * n > SZ_MAX_ELEMS or n_esc > n. */
SZ_API int sz_layout(uint64_t n, uint64_t n_esc, sz_meta* h_meta);

/* comp_bytes of a payload of n elements and n_esc escapes. */
SZ_API uint64_t sz_payload_bytes(uint64_t n, uint64_t n_esc);

/* Largest possible payload of n elements (every element escaped):
 * a payload buffer of this size never overflows. */
SZ_API uint64_t sz_max_payload_bytes(uint64_t n);

/* Fills tile_begin of h_items[0..count) (host copy of an item table) and
 * returns the total tile count in *h_total_tiles. */
SZ_API int sz_items_prepare(sz_item* h_items, uint32_t count, uint64_t* h_total_tiles);

/* Workspace sizes (bytes) of the compute calls.  The out-of-place decode
 * needs only its 256-byte status header, whatever the tensors: each CTA of its
 * single kernel checks the tensors of its tiles and finds their escape ranges
 * itself. */
SZ_API size_t sz_calibrate_workspace_bytes(uint32_t count);
SZ_API size_t sz_encode_workspace_bytes(uint32_t count, uint64_t total_tiles);
SZ_API size_t sz_decode_workspace_bytes(uint32_t count, uint64_t total_tiles);
SZ_API size_t sz_calibrate_encode_workspace_bytes(uint32_t count, uint64_t total_tiles);

/* Copies the workspace's SZ_FLAG_* word to *h_flags after synchronising
 * `stream`.  Returns SZ_OK when no bit is set, SZ_ERR_DEVICE otherwise. */
SZ_API int sz_workspace_flags(const void* d_workspace, uint32_t* h_flags, sz_stream stream);

/* ------------------------------------------------------------------ single tensor */

/* Calibration ("splitzip_codec.py" calibrate_codebook): histogram of the
 * exponent bytes of d_x[0..n), then the 16 most frequent values (ties by
 * ascending value) become codes 0..15; writes *d_codebook. */
SZ_API int sz_calibrate(const uint16_t* d_x, uint64_t n, sz_codebook* d_codebook,
                        void* d_workspace, size_t workspace_bytes, sz_stream stream);

/* Encode ("splitzip_codec.py" encode_torch + assemble_payload) of d_x[0..n)
 * with *d_codebook into d_payload[0..comp_bytes); writes *d_meta.  Any
 * codebook whose enc_lut entries are 0..15 or SZ_ESCAPE_CODE will do, such as
 * one calibrated on another tensor: the escapes follow from it.  Other
 * enc_lut values are not checked and give an unspecified payload (never a
 * fault).  If the payload would exceed
 * `capacity`, the payload is not valid and d_meta->status and the workspace
 * flags get SZ_FLAG_CAPACITY; no byte beyond capacity is written. */
SZ_API int sz_encode(const uint16_t* d_x, uint64_t n, const sz_codebook* d_codebook,
                     uint8_t* d_payload, uint64_t capacity, sz_meta* d_meta,
                     void* d_workspace, size_t workspace_bytes, sz_stream stream);

/* Decode ("splitzip_codec.py" decode_torch) of the payload described by
 * *d_meta (payload_bytes readable bytes at d_payload) with d_codebook->dec_lut
 * into d_out[0..n).  n must equal d_meta->n; a meta that disagrees with the
 * layout or with payload_bytes sets SZ_FLAG_META and leaves d_out unwritten;
 * an escape outside the tensor sets SZ_FLAG_ESCAPE and is skipped.  A meta
 * with SZ_META_GATED describes a tensor kept raw: nothing is written for it
 * and no flag is raised (the same holds in sz_decode_many). */
SZ_API int sz_decode(const uint8_t* d_payload, uint64_t payload_bytes, const sz_meta* d_meta,
                     const sz_codebook* d_codebook, uint16_t* d_out, uint64_t n,
                     void* d_workspace, size_t workspace_bytes, sz_stream stream);

/* ------------------------------------------------------------------ many tensors, one launch per step */

/* The same three operations over `count` (1..SZ_MANY_MAX_ITEMS) tensors of
 * any size, each with its own codebook and meta, described by the device
 * item table d_items (tile_begin filled as sz_items_prepare does;
 * total_tiles = its total).  Work is spread over all SMs tile by tile, so a
 * few large tensors and many mid-size ones run equally well.  A table whose
 * tensors average at most two tiles (16,384 elements, e.g. the blocks of a
 * paged KV cache) is encoded and decoded whole-tensor by whole-tensor in
 * shared memory instead: encode reads each input once and stages nothing,
 * decode copies each payload whole (at most 26 KiB) before decoding it.
 * Inside the same launches, encode hands the whole table to the tile-by-tile
 * kernels if one of its tensors is larger than two tiles, and decode leaves
 * them the tensors it cannot hold (more than two tiles, or a larger
 * payload).  Either way the results are the same bytes.  Calibration takes
 * the tile-by-tile kernel for every table.
 *   calibrate: reads x, n, tile_begin; writes *codebook.
 *   encode:    reads x, n, codebook, payload, capacity, tile_begin; writes payload, *meta.
 *   decode:    reads payload (capacity readable bytes), meta, codebook, n, tile_begin; writes out.
 * An inconsistent tile_begin chain sets SZ_FLAG_ITEMS; calibrate and encode
 * then write nothing, decode skips (and flags) the tiles it cannot place in
 * a consistent tensor and may decode the others -- never writing outside a
 * tensor's own output.  A tensor with n == 0 has nothing to decode, and decode
 * does not read its meta. */
SZ_API int sz_calibrate_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles,
                             void* d_workspace, size_t workspace_bytes, sz_stream stream);
SZ_API int sz_encode_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles,
                          void* d_workspace, size_t workspace_bytes, sz_stream stream);
SZ_API int sz_decode_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles,
                          void* d_workspace, size_t workspace_bytes, sz_stream stream);

/* ------------------------------------------------------------------ in-place slot decode */

/* Decode over the tensor's own buffer ("splitzip_codec.py"
 * GpuSplitZipDecoder.decode_slot_into; "docs/developer/splitzip.md", how a
 * compressed fault is served and the staging invariants): d_slot is the
 * BF16 destination, 2n bytes, 16-byte aligned, whose leading comp_bytes hold
 * the payload described by *d_meta (the bytes after it are ignored).  After
 * the call the slot holds the n decoded values.  The pages' decoder copies
 * the whole payload aside first; here the tiles are decoded in an order
 * that reads nearly everything in place (see sz_inplace_plan) and only the
 * pk bytes of about a quarter of the tiles and the escape streams (about
 * n / 8 + 7 n_esc bytes) are copied to the workspace; each tile is stored
 * once the tiles whose payload bytes lie under it have been read.
 * A payload larger than 2n bytes cannot be in the slot: SZ_FLAG_META, slot
 * untouched (as for a meta that disagrees with the layout).  A meta with
 * SZ_META_GATED means the slot already holds the raw tensor: nothing is
 * written.  Workspace: sz_decode_inplace_workspace_bytes(1, tiles(n))
 * (decode workspace + 4 bytes and 8 KiB per tile + 4352 bytes per tensor),
 * 256-byte aligned. */
SZ_API int sz_decode_inplace(uint16_t* d_slot, uint64_t n, const sz_meta* d_meta, const sz_codebook* d_codebook,
                             void* d_workspace, size_t workspace_bytes, sz_stream stream);
/* The same over an item table: item i's payload must equal its out (the
 * slot) and its payload may use at most min(capacity, 2n) bytes. */
SZ_API int sz_decode_inplace_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles,
                                  void* d_workspace, size_t workspace_bytes, sz_stream stream);
SZ_API size_t sz_decode_inplace_workspace_bytes(uint32_t count, uint64_t total_tiles);

/* The in-place schedule of one tile, for inspection (host only).  Tiles of a
 * tensor are decoded in three phases: A = [phase_a_first, tiles) from the
 * top down, B = [0, phase_b_end) from the top down, then C = [phase_b_end,
 * phase_a_first) from the bottom up; `rank` is the tile's position in that
 * order.  The payload bytes copied to the stash before the decode are the pk
 * bytes of phase C and the escape streams.  Before tile `tile` stores its
 * output, the tiles whose in-place payload bytes lie under it must have read
 * them (local tile indices, inclusive ranges, empty when lo > hi; the tile
 * itself may appear).  SZ_ERR_ARG for n == 0, n out of range, n_esc > n or
 * tile >= tiles(n); SZ_ERR_CAPACITY if the payload of (n, n_esc) is larger
 * than 2n bytes. */
typedef struct sz_inplace_tile {
  uint64_t tiles, phase_a_first, phase_b_end;  /* T, tA = ceil(off_sm / 8192), tB = off_sm / 16384 */
  uint64_t rank;                               /* position of `tile` in the decode order          */
  uint64_t stash_pk_from, stash_pk_to;         /* payload bytes stashed: pk of phase C             */
  uint64_t stash_esc_from, stash_esc_to;       /* payload bytes stashed: escape streams            */
  uint64_t stash_bytes, stash_budget;          /* stash bytes used / reserved for the tensor       */
  uint64_t pk_lo, pk_hi, pk2_lo, pk2_hi;       /* tiles whose pk bytes lie under this output       */
  uint64_t sm_lo, sm_hi;                       /* tiles whose sm bytes lie under it                */
} sz_inplace_tile;
SZ_API int sz_inplace_plan(uint64_t n, uint64_t n_esc, uint64_t tile, sz_inplace_tile* h_out);

/* ------------------------------------------------------------------ diagnostics */

/* Every wait inside the kernels is bounded: after about 2 s it gives up,
 * sets SZ_FLAG_TIMEOUT and lets the kernel end, so a stuck call reports an
 * error instead of hanging the device.  This call checks that on the device
 * it runs on: one CTA waits on an mbarrier phase that never completes, on a
 * word polled by one thread and on words polled by a warp (the three kinds
 * of waits the kernels use), none of which is ever satisfied.  Afterwards
 * the workspace flags hold SZ_FLAG_TIMEOUT and the uint32 words at byte
 * offsets 260, 264 and 268 of the workspace hold 1 (that wait gave up).
 * About 2 s of device time; asynchronous like the other calls.  Workspace:
 * SZ_CHECK_WAITS_WORKSPACE_BYTES, 256-byte aligned. */
#define SZ_CHECK_WAITS_WORKSPACE_BYTES 512u
SZ_API int sz_check_bounded_waits(void* d_workspace, size_t workspace_bytes, sz_stream stream);

/* ------------------------------------------------------------------ decode streamed from host memory */

/* Decode of tensors whose payloads are in pinned host memory
 * ("docs/developer/splitzip.md": a compressed fault is served by copying the
 * payload from pinned host memory to the GPU and decoding it there, on the
 * same stream).  h_items is a HOST array: payload = pinned host address
 * (16-byte aligned, h_metas[i].comp_bytes bytes read), out and codebook =
 * device addresses, n; meta, capacity and tile_begin are ignored.  h_metas
 * (host) are the tensors' metas.  The tensors go in groups that fit in half
 * of d_staging (device, 256-byte aligned, staging_bytes): copies of one group
 * on copy_stream overlap the decode of the previous group on `stream`
 * (the sz_decode_many kernels); payloads back to back in host memory (gaps
 * under 256 bytes) go in one copy.  d_scratch (device, 256-byte aligned) holds
 * the metas, the group tables and the decode workspace:
 * sz_decode_many_host_scratch_bytes bytes.  h_upload is a PINNED host buffer
 * of the caller's (cudaHostAlloc or cudaHostRegister; pageable memory is
 * refused with SZ_ERR_ARG) of at least sz_decode_many_host_upload_bytes(count)
 * bytes: the call writes the metas and the per-group tables there before it
 * returns and copies them to the device on `stream`, so the caller may write
 * to or free h_upload only once `stream` has passed the call (an event
 * recorded on `stream` after it); h_items and h_metas may be pageable and may
 * be reused as soon as the call returns.  Work on copy_stream follows the
 * caller's earlier work on `stream`, and `stream` waits for all of it, so the
 * call is ordered on `stream` like any other.  The call allocates no memory;
 * it creates three CUDA events and destroys them before it returns (the
 * runtime frees them once their work is done).  SZ_ERR_WORKSPACE if a
 * payload does not fit in half the staging buffer or if scratch_bytes or
 * upload_bytes is too small; SZ_ERR_CUDA if a CUDA call fails.
 * Device-visible conditions (a meta that disagrees with the layout, an escape
 * out of range) are reported as by sz_decode_many, through the workspace word
 * at the start of the decode workspace (see sz_decode_many_host_flags_offset). */
SZ_API size_t sz_decode_many_host_scratch_bytes(const sz_item* h_items, const sz_meta* h_metas, uint32_t count,
                                                uint64_t staging_bytes);
/* Bytes of the pinned upload buffer: round_up(count * 96, 256) + count * 64;
 * 0 if count is 0 or above SZ_MANY_MAX_ITEMS. */
SZ_API size_t sz_decode_many_host_upload_bytes(uint32_t count);
SZ_API int sz_decode_many_host(const sz_item* h_items, const sz_meta* h_metas, uint32_t count,
                               void* d_staging, uint64_t staging_bytes, void* d_scratch, size_t scratch_bytes,
                               void* h_upload, size_t upload_bytes, sz_stream stream, sz_stream copy_stream);
/* Offset (bytes) of the decode workspace, and so of its SZ_FLAG_* word, in the
 * scratch of sz_decode_many_host: pass d_scratch + this to sz_workspace_flags. */
SZ_API size_t sz_decode_many_host_flags_offset(uint32_t count);

/* ------------------------------------------------------------------ coverage gate */

/* sz_encode_many with the coverage gate of the pages' shard-cache builder
 * ("docs/developer/splitzip.md": tensors whose Top-16 exponent coverage is
 * below 0.99 are left uncompressed, so the worst case is parity; broad
 * exponent distributions would expand).  A tensor whose codebook coverage is
 * below min_coverage is not encoded: its meta gets status SZ_META_GATED, n,
 * its coverage and zeros elsewhere, and no payload byte is written; the
 * others are encoded exactly as by sz_encode_many.  *d_report (device, 16-byte
 * aligned) receives the build report of the call.  min_coverage < 0 gates
 * nothing.  Workspace: sz_encode_workspace_bytes. */
SZ_API int sz_encode_gated_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles,
                                double min_coverage, sz_gate_report* d_report,
                                void* d_workspace, size_t workspace_bytes, sz_stream stream);

/* ------------------------------------------------------------------ calibrate + encode in one call */

/* Calibration followed by encode ("splitzip_codec.py" calibrate_codebook,
 * then encode_torch + assemble_payload with the codebook it returns) in one
 * call.  A table of small tensors (as in sz_encode_many) is counted, ranked
 * and encoded one whole tensor at a time in shared memory, each input read
 * from HBM once.  Other tables go through one cooperative kernel (all its
 * CTAs resident at once; SZ_ERR_CUDA if the device cannot run it): the
 * tensors are taken in groups of about 32 MiB, and each group is counted and,
 * two groups later, encoded.  That second read was meant to hit L2, but the
 * traffic between the two passes is larger than L2, so on a GB300 it comes
 * from HBM (391 MB read for 201 MB of KV-cache input).  The codebooks,
 * payloads, metas and flags are those of sz_calibrate (or sz_calibrate_many)
 * followed by sz_encode (sz_encode_many), byte for byte; the table fields read
 * and written are the union of the two calls'.
 * On a GB300 with the input in HBM this call is the faster one for tables of
 * small tensors (8192 tensors of 16,384 elements: 164 against 171 us); for
 * large tensors the two separate calls are as fast or faster (0.95-0.98 x
 * on the KV-cache, weight and 4 GiB tables).  The pages calibrate offline,
 * one tensor at a time, and encode after a host round trip; this fusion has
 * no counterpart there. */
SZ_API int sz_calibrate_encode(const uint16_t* d_x, uint64_t n, sz_codebook* d_codebook,
                               uint8_t* d_payload, uint64_t capacity, sz_meta* d_meta,
                               void* d_workspace, size_t workspace_bytes, sz_stream stream);
SZ_API int sz_calibrate_encode_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles,
                                    void* d_workspace, size_t workspace_bytes, sz_stream stream);

/* ------------------------------------------------------------------ decode without a caller workspace */

#define SZ_NOALLOC_MAX_ELEMS 268435456ull  /* 2^28 elements (512 MiB of BF16) */

/* Decode for callers that cannot allocate device memory when they decode --
 * e.g. a host framework that owns all device memory and does not let
 * libraries allocate, or a latency-critical path that must not call
 * cudaMalloc (which may synchronise the device).  No counterpart in the
 * SplitZip pages: it is sz_decode with the workspace replaced by a fixed
 * scratch array inside the library (a file-scope __device__ array of 256
 * bytes, the decode's status header, present on every device that loads the
 * library until the process exits).  Nothing is allocated per call: no
 * cudaMalloc, cudaFree or allocating library routine.
 *   Arguments are those of sz_decode, without the workspace; n must not
 *   exceed SZ_NOALLOC_MAX_ELEMS (larger tensors: SZ_ERR_ARG, use sz_decode).
 *   d_flags: optional device pointer (4-byte aligned) that receives the
 *   call's SZ_FLAG_* word asynchronously (0 = no device-side problem).
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it.  All calls on a device share the one array
 * and each call starts
 * by resetting what it reads, but calls whose work may overlap on the GPU
 * (different streams without ordering) race on it: order them. */
SZ_API int sz_decode_noalloc(const uint8_t* d_payload, uint64_t payload_bytes, const sz_meta* d_meta,
                             const sz_codebook* d_codebook, uint16_t* d_out, uint64_t n, uint32_t* d_flags,
                             sz_stream stream);

/* ------------------------------------------------------------------ measurement */

/* Timing hook: `before` and `after` are cudaEvent_t handles (or NULL to
 * clear).  While set, every compute call made by the calling host thread
 * records `before` on its stream just before its main kernel (the streaming
 * pass: cal_hist, enc_main or small_main, ce_main or small_main, dec_flat or
 * dec_inplace) and `after` just after it, so the
 * caller can time that kernel alone with cudaEventElapsedTime.  The events are
 * borrowed, never destroyed. */
SZ_API int sz_set_timing_events(void* before, void* after);

#ifdef __cplusplus
}
#endif
#endif /* SPLITZIP_H */
