// Decode of payloads that live in pinned host memory, streamed to the device
// ("docs/developer/splitzip.md": a compressed fault is served by copying the
// payload from pinned host memory to the GPU and decoding it there, on the
// same stream, before the weight is handed to compute).
//
// The tensors go in groups that fit in half of a caller's device staging
// buffer.  A copy stream fills one half while the compute stream decodes the
// group in the other half with the sz_decode_many kernels; two events keep
// the halves apart.  Payloads that lie back to back in host memory (at most
// 255 bytes apart, as in a packed shard blob) go in one copy per run.  The
// metas (host copies, as a manifest holds them) and the per-group item
// tables go to the device in one copy per call, through a pinned host buffer
// of the caller's: a copy from pageable memory may wait for the stream, which
// would stall the pipeline between calls.  The call allocates nothing; its
// three events are created per call and released as soon as their work is
// done.
#include <cstring>
#include <vector>

#include "sz_internal.h"

namespace sz {
namespace {

struct Group {
  uint32_t first, count;  // items [first, first + count)
  uint64_t tiles;         // their tiles
};

struct Run {  // one host-to-device copy
  const uint8_t* src;
  uint64_t dst_off;  // within the group's staging half
  uint64_t bytes;
  uint32_t group;
};

struct Plan {
  std::vector<Group> groups;
  std::vector<Run> runs;
  std::vector<uint64_t> dst_off;  // per item: payload offset within its group's half
  uint64_t max_ws = 0;            // largest decode workspace of a group
};

// Groups of consecutive items whose staged payloads fit in `half` bytes.
int make_plan(const sz_item* h_items, const sz_meta* h_metas, uint32_t count, uint64_t half, Plan* plan) {
  plan->dst_off.assign(count, 0);
  uint64_t used = 0;
  Group g{0, 0, 0};
  for (uint32_t i = 0; i < count; ++i) {
    const sz_meta& m = h_metas[i];
    const sz_item& it = h_items[i];
    if (m.n != it.n || it.n > SZ_MAX_ELEMS) return SZ_ERR_META;
    if (m.comp_bytes > it.capacity) return SZ_ERR_CAPACITY;
    if (m.comp_bytes > 0 && (it.payload == nullptr || (reinterpret_cast<uintptr_t>(it.payload) & 15)))
      return SZ_ERR_ALIGN;
    const uint64_t bytes = m.comp_bytes;
    if (bytes > half) return SZ_ERR_WORKSPACE;  // a payload must fit in one half
    // where the payload goes: right after the previous one when the host
    // layout is back to back (same relative offset), else the next 256-byte
    // boundary
    uint64_t off = (used + 255) & ~uint64_t(255);
    bool extend = false;
    if (g.count > 0 && !plan->runs.empty() && bytes > 0) {
      const Run& r = plan->runs.back();
      const uint8_t* end = r.src + r.bytes;
      if (r.group == plan->groups.size() && it.payload >= end && uint64_t(it.payload - end) < 256) {
        off = r.dst_off + uint64_t(it.payload - r.src);
        extend = true;
      }
    }
    if (off + bytes > half) {  // the group is full: start the next one
      plan->groups.push_back(g);
      g = Group{i, 0, 0};
      off = 0;
      extend = false;
    }
    if (bytes > 0) {
      if (extend) {
        Run& r = plan->runs.back();
        r.bytes = off + bytes - r.dst_off;
      } else {
        plan->runs.push_back(Run{it.payload, off, bytes, uint32_t(plan->groups.size())});
      }
    }
    plan->dst_off[i] = off;
    used = off + bytes;
    g.count += 1;
    g.tiles += tiles_of(it.n);
  }
  if (g.count > 0) plan->groups.push_back(g);
  for (const Group& gr : plan->groups) {
    const uint64_t w = dec_ws_bytes(gr.count, gr.tiles);
    if (w > plan->max_ws) plan->max_ws = w;
  }
  return SZ_OK;
}

// device scratch: metas[count] | tables[count] | decode workspace
uint64_t scratch_bytes(uint32_t count, const Plan& plan) {
  return round_up256(uint64_t(count) * sizeof(sz_meta)) + round_up256(uint64_t(count) * sizeof(sz_item)) +
         plan.max_ws;
}

// bytes of the metas and tables as uploaded (and as laid out in the scratch)
uint64_t upload_size(uint32_t count) {
  return round_up256(uint64_t(count) * sizeof(sz_meta)) + uint64_t(count) * sizeof(sz_item);
}

// Events of one call, destroyed on every way out (a recorded event is
// released by the runtime once its work has completed).
struct CallEvents {
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  ~CallEvents() {
    for (cudaEvent_t e : ev)
      if (e != nullptr) cudaEventDestroy(e);
  }
  bool create() {
    for (cudaEvent_t& e : ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
};

}  // namespace
}  // namespace sz

using namespace sz;

SZ_API size_t sz_decode_many_host_upload_bytes(uint32_t count) {
  if (count == 0 || count > SZ_MANY_MAX_ITEMS) return 0;
  return size_t(upload_size(count));
}

SZ_API size_t sz_decode_many_host_flags_offset(uint32_t count) {
  return size_t(round_up256(uint64_t(count) * sizeof(sz_meta)) + round_up256(uint64_t(count) * sizeof(sz_item)));
}

SZ_API size_t sz_decode_many_host_scratch_bytes(const sz_item* h_items, const sz_meta* h_metas, uint32_t count,
                                                uint64_t staging_bytes) {
  if (h_items == nullptr || h_metas == nullptr || count == 0 || count > SZ_MANY_MAX_ITEMS) return 0;
  Plan plan;
  if (make_plan(h_items, h_metas, count, (staging_bytes / 2) & ~uint64_t(255), &plan) != SZ_OK) return 0;
  return size_t(scratch_bytes(count, plan));
}

SZ_API int sz_decode_many_host(const sz_item* h_items, const sz_meta* h_metas, uint32_t count, void* d_staging,
                               uint64_t staging_bytes, void* d_scratch, size_t scratch_size, void* h_upload,
                               size_t upload_bytes, sz_stream stream, sz_stream copy_stream) {
  if (h_items == nullptr || h_metas == nullptr || count == 0 || count > SZ_MANY_MAX_ITEMS) return SZ_ERR_ARG;
  if (d_staging == nullptr || d_scratch == nullptr || h_upload == nullptr) return SZ_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(d_staging) & 255) || (reinterpret_cast<uintptr_t>(d_scratch) & 255))
    return SZ_ERR_ALIGN;
  const uint64_t half = (staging_bytes / 2) & ~uint64_t(255);
  Plan plan;
  if (int rc = make_plan(h_items, h_metas, count, half, &plan)) return rc;
  if (scratch_size < scratch_bytes(count, plan) || upload_bytes < upload_size(count)) return SZ_ERR_WORKSPACE;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, h_upload) != cudaSuccess) {
    cudaGetLastError();  // clear it: an unknown pointer is the caller's error
    return SZ_ERR_ARG;
  }
  if (attr.type != cudaMemoryTypeHost) return SZ_ERR_ARG;  // pinned host memory only
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return SZ_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(copy_stream);
  char* scratch = static_cast<char*>(d_scratch);
  const uint64_t tables_off = round_up256(uint64_t(count) * sizeof(sz_meta));
  sz_meta* d_metas = reinterpret_cast<sz_meta*>(scratch);
  sz_item* d_tables = reinterpret_cast<sz_item*>(scratch + tables_off);
  void* d_ws = scratch + tables_off + round_up256(uint64_t(count) * sizeof(sz_item));
  uint8_t* stage[2] = {static_cast<uint8_t*>(d_staging), static_cast<uint8_t*>(d_staging) + half};

  // metas and tables, laid out as in the scratch, in the caller's pinned buffer
  char* pinned = static_cast<char*>(h_upload);
  std::memcpy(pinned, h_metas, uint64_t(count) * sizeof(sz_meta));
  sz_item* tables = reinterpret_cast<sz_item*>(pinned + tables_off);
  std::memcpy(tables, h_items, uint64_t(count) * sizeof(sz_item));
  // the per-group tables: payloads in the group's staging half, metas on the device
  for (size_t gi = 0; gi < plan.groups.size(); ++gi) {
    const Group& g = plan.groups[gi];
    uint64_t tb = 0;
    for (uint32_t i = g.first; i < g.first + g.count; ++i) {
      tables[i].payload = stage[gi & 1] + plan.dst_off[i];
      tables[i].meta = d_metas + i;
      tables[i].capacity = h_metas[i].comp_bytes;
      tables[i].tile_begin = tb;
      tb += tiles_of(h_items[i].n);
    }
  }
  // events: copy of group j done; decode of the group last in each half done
  CallEvents events;
  if (!events.create()) return SZ_ERR_CUDA;
  cudaEvent_t copied = events.ev[0], decoded[2] = {events.ev[1], events.ev[2]};
  cudaError_t e = cudaMemcpyAsync(d_metas, pinned, upload_size(count), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return SZ_ERR_CUDA;
  // nothing of this call starts on the copy stream before the caller's
  // earlier work on `stream` (e.g. the staging buffer's previous use)
  if ((e = cudaEventRecord(decoded[0], s)) != cudaSuccess) return SZ_ERR_CUDA;
  if ((e = cudaEventRecord(decoded[1], s)) != cudaSuccess) return SZ_ERR_CUDA;
  // one status word for the whole call: cleared once, each group's decode adds its flags
  if ((e = cudaMemsetAsync(d_ws, 0, sizeof(WsHeader), s)) != cudaSuccess) return SZ_ERR_CUDA;
  size_t r = 0;
  for (size_t gi = 0; gi < plan.groups.size(); ++gi) {
    const Group& g = plan.groups[gi];
    const int h = int(gi & 1);
    // the half is free once the decode of the group before last is done
    if ((e = cudaStreamWaitEvent(cs, decoded[h], 0)) != cudaSuccess) return SZ_ERR_CUDA;
    for (; r < plan.runs.size() && plan.runs[r].group == gi; ++r) {
      const Run& run = plan.runs[r];
      e = cudaMemcpyAsync(stage[h] + run.dst_off, run.src, run.bytes, cudaMemcpyHostToDevice, cs);
      if (e != cudaSuccess) return SZ_ERR_CUDA;
    }
    if ((e = cudaEventRecord(copied, cs)) != cudaSuccess) return SZ_ERR_CUDA;
    if ((e = cudaStreamWaitEvent(s, copied, 0)) != cudaSuccess) return SZ_ERR_CUDA;
    Items items;
    items.table = d_tables + g.first;
    std::memset(&items.one, 0, sizeof(items.one));
    items.count = g.count;
    items.total_tiles = g.tiles;
    if ((e = launch_decode(items, d_ws, s, dev, false)) != cudaSuccess) return SZ_ERR_CUDA;
    if ((e = cudaEventRecord(decoded[h], s)) != cudaSuccess) return SZ_ERR_CUDA;
  }
  // the copy stream has no work left that `stream` does not wait for
  return SZ_OK;
}
