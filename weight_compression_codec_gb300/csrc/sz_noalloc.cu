// sz_decode_noalloc: decode with a library-owned, fixed-size scratch area.
//
// The regular sz_decode takes a caller-allocated workspace.  Some callers
// cannot allocate device memory at the point where they decode: a host
// framework that owns every byte of device memory and does not let libraries
// allocate, or a latency-critical path that must not call cudaMalloc (it can
// synchronise the device and fragments memory).  For them this entry point
// keeps its scratch in a file-scope __device__ array that exists, once per
// device, for as long as the library is loaded; nothing is allocated per call.
#include <cstring>
#include <mutex>

#include "sz_internal.h"

namespace {

using namespace sz;

// The scratch holds the decode workspace of one tensor of up to
// SZ_NOALLOC_MAX_ELEMS elements (its size comes from the same function that
// sizes the workspace of sz_decode, and every call checks it before launch).
constexpr uint64_t kMaxTiles = (SZ_NOALLOC_MAX_ELEMS + kTile - 1) / kTile;
constexpr size_t kScratchBytes = size_t(dec_ws_bytes(1, kMaxTiles));
static_assert(kScratchBytes >= 256 && kScratchBytes % 256 == 0, "scratch holds at least the status header");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[64] = {nullptr};  // device address of the array, per device

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
cudaError_t scratch_for(int device, void** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" SZ_API int sz_decode_noalloc(const uint8_t* d_payload, uint64_t payload_bytes, const sz_meta* d_meta,
                                        const sz_codebook* d_codebook, uint16_t* d_out, uint64_t n,
                                        uint32_t* d_flags, sz_stream stream) {
  if (n > SZ_NOALLOC_MAX_ELEMS) return SZ_ERR_ARG;  // larger tensors need sz_decode and a workspace
  if (d_meta == nullptr || d_codebook == nullptr) return SZ_ERR_ARG;
  if (n > 0 && (d_out == nullptr || d_payload == nullptr)) return SZ_ERR_ARG;
  if (!aligned16(d_payload) || !aligned16(d_out) || !aligned16(d_codebook) || !aligned16(d_meta) ||
      (reinterpret_cast<uintptr_t>(d_flags) & 3))
    return SZ_ERR_ALIGN;
  if (layout_of(n, 0).off_cid > payload_bytes) return SZ_ERR_CAPACITY;
  // the decode workspace of this n must fit in the array
  if (dec_ws_bytes(1, tiles_of(n)) > sizeof(g_noalloc_scratch)) return SZ_ERR_ARG;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  void* scratch = nullptr;
  if (scratch_for(dev.device, &scratch) != cudaSuccess) return SZ_ERR_CUDA;

  Items items;
  std::memset(&items, 0, sizeof(items));
  items.table = nullptr;
  items.one.out = d_out;
  items.one.payload = const_cast<uint8_t*>(d_payload);
  items.one.codebook = const_cast<sz_codebook*>(d_codebook);
  items.one.meta = const_cast<sz_meta*>(d_meta);
  items.one.n = n;
  items.one.capacity = payload_bytes;
  items.count = 1;
  items.total_tiles = tiles_of(n);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // launch_decode zeroes the header (the status flags) itself, and the
  // decode reads nothing else of the array, so nothing an earlier call left
  // there is used.
  if (launch_decode(items, scratch, s, dev) != cudaSuccess) return SZ_ERR_CUDA;
  if (d_flags != nullptr &&
      cudaMemcpyAsync(d_flags, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return SZ_ERR_CUDA;
  return SZ_OK;
}
