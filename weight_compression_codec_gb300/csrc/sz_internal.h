// Internal launch interface between the C ABI (sz_api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "sz_device.cuh"

namespace sz {

struct DeviceInfo {
  int device;
  int num_sms;
};

// Cached per-device properties (SM count); also opts kernels into large
// dynamic shared memory once per device.
cudaError_t device_info(DeviceInfo* info);

cudaError_t launch_calibrate(const Items& items, void* ws, cudaStream_t stream, const DeviceInfo& dev);
// gate >= 0: tensors whose codebook coverage is below it are left uncompressed
// (meta status SZ_META_GATED); report (device) receives the build report
cudaError_t launch_encode(const Items& items, void* ws, cudaStream_t stream, const DeviceInfo& dev,
                          double gate = -1.0, sz_gate_report* report = nullptr);
// out-of-place decode; clear_header = false keeps the status flags of earlier
// launches on the same workspace (the groups of one host-streamed call)
cudaError_t launch_decode(const Items& items, void* ws, cudaStream_t stream, const DeviceInfo& dev,
                          bool clear_header = true);
// diagnostic: each kind of bounded wait, on something that never completes
cudaError_t launch_wait_selftest(void* ws, cudaStream_t stream);
// in-place slot decode (items with payload == out; ip_ws workspace)
cudaError_t launch_decode_inplace(const Items& items, void* ws, cudaStream_t stream, const DeviceInfo& dev);
// calibrate + encode in one streaming pass (CeWs workspace), then placement
cudaError_t launch_calibrate_encode(const Items& items, void* ws, cudaStream_t stream, const DeviceInfo& dev);
// escape placement, pads and metas after an encode pass (enc_place)
cudaError_t launch_place(const Items& items, const EncWs& ws, cudaStream_t stream, const DeviceInfo& dev);
// Small-tensor route: true for a table whose tensors average at most two
// tiles.  launch_small runs small_main over the table after the prepare pass
// (calibrate + encode when cal_done, the count pass's validity marks, is
// given; encode alone otherwise); it does the work only if the prepare pass
// found no tensor larger than kSmallMax.
bool small_route(const Items& items);
cudaError_t launch_small(const Items& items, const EncWs& ws, const uint32_t* cal_done, cudaStream_t stream,
                         const DeviceInfo& dev);

// Launches `kernel` on `stream` as a programmatic dependent of the kernel
// before it: it may be scheduled while that kernel drains, and waits for it
// in pdl_wait (every kernel launched this way calls pdl_wait before reading
// global memory).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Optional timing hook: when set (non-null), launchers record `before` just
// before and `after` just after their main kernel on the launch stream.
struct TimingHook {
  cudaEvent_t before;
  cudaEvent_t after;
};
extern thread_local TimingHook g_timing;

}  // namespace sz
