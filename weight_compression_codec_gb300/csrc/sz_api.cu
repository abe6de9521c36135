// C ABI of the SplitZip codec (declared in include/splitzip.h): host-side
// argument checks, workspace sizing and kernel dispatch.  No call allocates
// memory or synchronises the stream (except sz_workspace_flags, which exists
// to read the device status back).
#include <atomic>
#include <cstring>

#include "sz_internal.h"

namespace sz {

thread_local TimingHook g_timing = {nullptr, nullptr};

cudaError_t device_info(DeviceInfo* info) {
  // SM count per device, queried once; host threads may race to fill an
  // entry, all with the same value
  static std::atomic<int> cached_sms[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = cached_sms[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    cached_sms[dev].store(sms, std::memory_order_relaxed);
  }
  info->device = dev;
  info->num_sms = sms;
  return cudaSuccess;
}

}  // namespace sz

using namespace sz;

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_ws(const void* ws, size_t have, uint64_t need) {
  if (ws == nullptr || !aligned(ws, 256) || have < need) return SZ_ERR_WORKSPACE;
  return SZ_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? SZ_OK : SZ_ERR_CUDA; }

Items single(const sz_item& one) {
  Items it;
  it.table = nullptr;
  it.one = one;
  it.count = 1;
  it.total_tiles = tiles_of(one.n);
  return it;
}

Items table(const sz_item* d_items, uint32_t count, uint64_t total_tiles) {
  Items it;
  it.table = d_items;
  std::memset(&it.one, 0, sizeof(it.one));
  it.count = count;
  it.total_tiles = total_tiles;
  return it;
}

int check_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles) {
  if (d_items == nullptr || count == 0 || count > SZ_MANY_MAX_ITEMS) return SZ_ERR_ARG;
  if (!aligned(d_items, 16)) return SZ_ERR_ALIGN;
  if (total_tiles > uint64_t(count) * tiles_of(SZ_MAX_ELEMS)) return SZ_ERR_ARG;
  return SZ_OK;
}

}  // namespace

extern "C" {

SZ_API int sz_version(void) { return SZ_VERSION; }

SZ_API const char* sz_strerror(int status) {
  switch (status) {
    case SZ_OK: return "ok";
    case SZ_ERR_ARG: return "invalid argument (null pointer, size or count out of range)";
    case SZ_ERR_ALIGN: return "pointer alignment (data/payload/codebook/meta 16 bytes, workspace 256 bytes)";
    case SZ_ERR_CAPACITY: return "payload capacity too small";
    case SZ_ERR_META: return "meta disagrees with the wire layout";
    case SZ_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SZ_ERR_CUDA: return "CUDA runtime error";
    case SZ_ERR_DEVICE: return "device reported SZ_FLAG_* status bits";
    default: return "unknown status";
  }
}

SZ_API uint64_t sz_tiles(uint64_t n) { return tiles_of(n); }

SZ_API int sz_layout(uint64_t n, uint64_t n_esc, sz_meta* h_meta) {
  if (h_meta == nullptr || n > SZ_MAX_ELEMS || n_esc > n) return SZ_ERR_ARG;
  const Layout l = layout_of(n, n_esc);
  std::memset(h_meta, 0, sizeof(*h_meta));
  h_meta->n = n;
  h_meta->n_pairs = l.n_pairs;
  h_meta->n_esc = n_esc;
  h_meta->comp_bytes = l.comp_bytes;
  h_meta->off_pk = 0;
  h_meta->off_sm = l.off_sm;
  h_meta->off_cid = l.off_cid;
  h_meta->off_lpos = l.off_lpos;
  h_meta->off_ev = l.off_ev;
  h_meta->chunk_size = kChunk;
  return SZ_OK;
}

SZ_API uint64_t sz_payload_bytes(uint64_t n, uint64_t n_esc) { return layout_of(n, n_esc).comp_bytes; }

SZ_API uint64_t sz_max_payload_bytes(uint64_t n) { return layout_of(n, n).comp_bytes; }

SZ_API int sz_items_prepare(sz_item* h_items, uint32_t count, uint64_t* h_total_tiles) {
  if (h_items == nullptr || h_total_tiles == nullptr || count == 0) return SZ_ERR_ARG;
  uint64_t t = 0;
  for (uint32_t i = 0; i < count; ++i) {
    if (h_items[i].n > SZ_MAX_ELEMS) return SZ_ERR_ARG;
    h_items[i].tile_begin = t;
    t += tiles_of(h_items[i].n);
  }
  *h_total_tiles = t;
  return SZ_OK;
}

SZ_API size_t sz_calibrate_workspace_bytes(uint32_t count) { return size_t(cal_ws_bytes(count)); }

SZ_API size_t sz_encode_workspace_bytes(uint32_t count, uint64_t total_tiles) {
  return size_t(enc_ws_bytes(count, total_tiles));
}

SZ_API size_t sz_decode_workspace_bytes(uint32_t count, uint64_t total_tiles) {
  return size_t(dec_ws_bytes(count, total_tiles));
}

SZ_API size_t sz_decode_inplace_workspace_bytes(uint32_t count, uint64_t total_tiles) {
  return size_t(ip_ws_bytes(count, total_tiles));
}

SZ_API int sz_inplace_plan(uint64_t n, uint64_t n_esc, uint64_t tile, sz_inplace_tile* h_out) {
  if (h_out == nullptr || n == 0 || n > SZ_MAX_ELEMS || n_esc > n || tile >= tiles_of(n)) return SZ_ERR_ARG;
  const Layout l = layout_of(n, n_esc);
  if (l.comp_bytes > 2 * n) return SZ_ERR_CAPACITY;
  const IpStash st = ip_stash(n, n_esc, l.off_sm, l.off_cid, l.comp_bytes);
  const IpPhases ph = ip_phases(n, l.off_sm);
  const IpDeps d = ip_deps(n, l.off_sm, tile);
  h_out->tiles = ph.T;
  h_out->phase_a_first = ph.tA;
  h_out->phase_b_end = ph.tB;
  h_out->rank = ip_rank(ph, tile);
  h_out->stash_pk_from = st.pk_from;
  h_out->stash_pk_to = st.pk_to;
  h_out->stash_esc_from = st.esc_from;
  h_out->stash_esc_to = st.esc_to;
  h_out->stash_bytes = st.bytes;
  h_out->stash_budget = tiles_of(n) * kIpStashPerTile + kIpStashPerItem;
  h_out->pk_lo = d.pk_lo;
  h_out->pk_hi = d.pk_hi;
  h_out->pk2_lo = d.pk2_lo;
  h_out->pk2_hi = d.pk2_hi;
  h_out->sm_lo = d.sm_lo;
  h_out->sm_hi = d.sm_hi;
  return SZ_OK;
}

SZ_API size_t sz_calibrate_encode_workspace_bytes(uint32_t count, uint64_t total_tiles) {
  return size_t(ce_ws_bytes(count, total_tiles));
}

SZ_API int sz_workspace_flags(const void* d_workspace, uint32_t* h_flags, sz_stream stream) {
  if (d_workspace == nullptr || h_flags == nullptr) return SZ_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t f = 0;
  cudaError_t e = cudaMemcpyAsync(&f, d_workspace, sizeof(f), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return SZ_ERR_CUDA;
  *h_flags = f;
  return f ? SZ_ERR_DEVICE : SZ_OK;
}

// ---------------------------------------------------------------- single tensor

SZ_API int sz_calibrate(const uint16_t* d_x, uint64_t n, sz_codebook* d_codebook, void* d_workspace,
                        size_t workspace_bytes, sz_stream stream) {
  if (n > SZ_MAX_ELEMS || d_codebook == nullptr || (n > 0 && d_x == nullptr)) return SZ_ERR_ARG;
  if (!aligned(d_codebook, 16) || !aligned(d_x, 16)) return SZ_ERR_ALIGN;
  if (int rc = check_ws(d_workspace, workspace_bytes, cal_ws_bytes(1))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  sz_item one;
  std::memset(&one, 0, sizeof(one));
  one.x = d_x;
  one.codebook = d_codebook;
  one.n = n;
  return from_cuda(launch_calibrate(single(one), d_workspace, reinterpret_cast<cudaStream_t>(stream), dev));
}

SZ_API int sz_encode(const uint16_t* d_x, uint64_t n, const sz_codebook* d_codebook, uint8_t* d_payload,
                     uint64_t capacity, sz_meta* d_meta, void* d_workspace, size_t workspace_bytes,
                     sz_stream stream) {
  if (n > SZ_MAX_ELEMS || d_codebook == nullptr || d_meta == nullptr) return SZ_ERR_ARG;
  if (n > 0 && (d_x == nullptr || d_payload == nullptr)) return SZ_ERR_ARG;
  if (!aligned(d_x, 16) || !aligned(d_payload, 16) || !aligned(d_codebook, 16) || !aligned(d_meta, 16))
    return SZ_ERR_ALIGN;
  if (layout_of(n, 0).off_cid > capacity) return SZ_ERR_CAPACITY;
  if (int rc = check_ws(d_workspace, workspace_bytes, enc_ws_bytes(1, tiles_of(n)))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  sz_item one;
  std::memset(&one, 0, sizeof(one));
  one.x = d_x;
  one.payload = d_payload;
  one.codebook = const_cast<sz_codebook*>(d_codebook);
  one.meta = d_meta;
  one.n = n;
  one.capacity = capacity;
  return from_cuda(launch_encode(single(one), d_workspace, reinterpret_cast<cudaStream_t>(stream), dev));
}

SZ_API int sz_decode(const uint8_t* d_payload, uint64_t payload_bytes, const sz_meta* d_meta,
                     const sz_codebook* d_codebook, uint16_t* d_out, uint64_t n, void* d_workspace,
                     size_t workspace_bytes, sz_stream stream) {
  if (n > SZ_MAX_ELEMS || d_meta == nullptr || d_codebook == nullptr) return SZ_ERR_ARG;
  if (n > 0 && (d_out == nullptr || d_payload == nullptr)) return SZ_ERR_ARG;
  if (!aligned(d_payload, 16) || !aligned(d_out, 16) || !aligned(d_codebook, 16) || !aligned(d_meta, 16))
    return SZ_ERR_ALIGN;
  if (layout_of(n, 0).off_cid > payload_bytes) return SZ_ERR_CAPACITY;
  if (int rc = check_ws(d_workspace, workspace_bytes, dec_ws_bytes(1, tiles_of(n)))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  sz_item one;
  std::memset(&one, 0, sizeof(one));
  one.out = d_out;
  one.payload = const_cast<uint8_t*>(d_payload);
  one.codebook = const_cast<sz_codebook*>(d_codebook);
  one.meta = const_cast<sz_meta*>(d_meta);
  one.n = n;
  one.capacity = payload_bytes;
  return from_cuda(launch_decode(single(one), d_workspace, reinterpret_cast<cudaStream_t>(stream), dev));
}

SZ_API int sz_decode_inplace(uint16_t* d_slot, uint64_t n, const sz_meta* d_meta, const sz_codebook* d_codebook,
                             void* d_workspace, size_t workspace_bytes, sz_stream stream) {
  if (n > SZ_MAX_ELEMS || d_meta == nullptr || d_codebook == nullptr) return SZ_ERR_ARG;
  if (n > 0 && d_slot == nullptr) return SZ_ERR_ARG;
  if (!aligned(d_slot, 16) || !aligned(d_codebook, 16) || !aligned(d_meta, 16)) return SZ_ERR_ALIGN;
  if (int rc = check_ws(d_workspace, workspace_bytes, ip_ws_bytes(1, tiles_of(n)))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  sz_item one;
  std::memset(&one, 0, sizeof(one));
  one.out = d_slot;
  one.payload = reinterpret_cast<uint8_t*>(d_slot);
  one.codebook = const_cast<sz_codebook*>(d_codebook);
  one.meta = const_cast<sz_meta*>(d_meta);
  one.n = n;
  one.capacity = 2 * n;
  return from_cuda(launch_decode_inplace(single(one), d_workspace, reinterpret_cast<cudaStream_t>(stream), dev));
}

// ---------------------------------------------------------------- many tensors

SZ_API int sz_calibrate_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles, void* d_workspace,
                             size_t workspace_bytes, sz_stream stream) {
  if (int rc = check_many(d_items, count, total_tiles)) return rc;
  if (int rc = check_ws(d_workspace, workspace_bytes, cal_ws_bytes(count))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  return from_cuda(launch_calibrate(table(d_items, count, total_tiles), d_workspace,
                                    reinterpret_cast<cudaStream_t>(stream), dev));
}

SZ_API int sz_encode_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles, void* d_workspace,
                          size_t workspace_bytes, sz_stream stream) {
  if (int rc = check_many(d_items, count, total_tiles)) return rc;
  if (int rc = check_ws(d_workspace, workspace_bytes, enc_ws_bytes(count, total_tiles))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  return from_cuda(launch_encode(table(d_items, count, total_tiles), d_workspace,
                                 reinterpret_cast<cudaStream_t>(stream), dev));
}

SZ_API int sz_decode_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles, void* d_workspace,
                          size_t workspace_bytes, sz_stream stream) {
  if (int rc = check_many(d_items, count, total_tiles)) return rc;
  if (int rc = check_ws(d_workspace, workspace_bytes, dec_ws_bytes(count, total_tiles))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  return from_cuda(launch_decode(table(d_items, count, total_tiles), d_workspace,
                                 reinterpret_cast<cudaStream_t>(stream), dev));
}

SZ_API int sz_check_bounded_waits(void* d_workspace, size_t workspace_bytes, sz_stream stream) {
  if (int rc = check_ws(d_workspace, workspace_bytes, SZ_CHECK_WAITS_WORKSPACE_BYTES)) return rc;
  return from_cuda(launch_wait_selftest(d_workspace, reinterpret_cast<cudaStream_t>(stream)));
}

SZ_API int sz_decode_inplace_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles, void* d_workspace,
                                  size_t workspace_bytes, sz_stream stream) {
  if (int rc = check_many(d_items, count, total_tiles)) return rc;
  if (int rc = check_ws(d_workspace, workspace_bytes, ip_ws_bytes(count, total_tiles))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  return from_cuda(launch_decode_inplace(table(d_items, count, total_tiles), d_workspace,
                                         reinterpret_cast<cudaStream_t>(stream), dev));
}

// ---------------------------------------------------------------- coverage gate

SZ_API int sz_encode_gated_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles, double min_coverage,
                                sz_gate_report* d_report, void* d_workspace, size_t workspace_bytes,
                                sz_stream stream) {
  if (int rc = check_many(d_items, count, total_tiles)) return rc;
  if (d_report == nullptr || min_coverage != min_coverage) return SZ_ERR_ARG;  // NaN gate
  if (!aligned(d_report, 16)) return SZ_ERR_ALIGN;
  if (int rc = check_ws(d_workspace, workspace_bytes, enc_ws_bytes(count, total_tiles))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  return from_cuda(launch_encode(table(d_items, count, total_tiles), d_workspace,
                                 reinterpret_cast<cudaStream_t>(stream), dev, min_coverage, d_report));
}

// ---------------------------------------------------------------- calibrate + encode

SZ_API int sz_calibrate_encode(const uint16_t* d_x, uint64_t n, sz_codebook* d_codebook, uint8_t* d_payload,
                               uint64_t capacity, sz_meta* d_meta, void* d_workspace, size_t workspace_bytes,
                               sz_stream stream) {
  if (n > SZ_MAX_ELEMS || d_codebook == nullptr || d_meta == nullptr) return SZ_ERR_ARG;
  if (n > 0 && (d_x == nullptr || d_payload == nullptr)) return SZ_ERR_ARG;
  if (!aligned(d_x, 16) || !aligned(d_payload, 16) || !aligned(d_codebook, 16) || !aligned(d_meta, 16))
    return SZ_ERR_ALIGN;
  if (layout_of(n, 0).off_cid > capacity) return SZ_ERR_CAPACITY;
  if (int rc = check_ws(d_workspace, workspace_bytes, ce_ws_bytes(1, tiles_of(n)))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  sz_item one;
  std::memset(&one, 0, sizeof(one));
  one.x = d_x;
  one.payload = d_payload;
  one.codebook = d_codebook;
  one.meta = d_meta;
  one.n = n;
  one.capacity = capacity;
  return from_cuda(
      launch_calibrate_encode(single(one), d_workspace, reinterpret_cast<cudaStream_t>(stream), dev));
}

SZ_API int sz_calibrate_encode_many(const sz_item* d_items, uint32_t count, uint64_t total_tiles,
                                    void* d_workspace, size_t workspace_bytes, sz_stream stream) {
  if (int rc = check_many(d_items, count, total_tiles)) return rc;
  if (int rc = check_ws(d_workspace, workspace_bytes, ce_ws_bytes(count, total_tiles))) return rc;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  return from_cuda(launch_calibrate_encode(table(d_items, count, total_tiles), d_workspace,
                                           reinterpret_cast<cudaStream_t>(stream), dev));
}

// Timing hook used by the benchmark: events recorded around the next main
// kernels launched by this host thread (pass NULLs to clear).
SZ_API int sz_set_timing_events(void* before, void* after) {
  g_timing.before = reinterpret_cast<cudaEvent_t>(before);
  g_timing.after = reinterpret_cast<cudaEvent_t>(after);
  return SZ_OK;
}

}  // extern "C"
