// decode_noalloc.cu -- decode attention for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code running inside another runtime's memory arena, embedders whose
// allocator is owned by a host framework, or a loop that must not touch the
// driver's allocator (an allocation can synchronise the device or fail under
// memory pressure at the worst moment). kvarn_decode_attention needs a
// caller-provided workspace; this entry point instead uses a fixed scratch
// array that lives in the library's own device memory, so the caller passes
// only inputs and outputs.
//
// The scratch array is a file-scope __device__ array: every GPU that loads
// this library holds it (KVARN_NOALLOC_SCRATCH_BYTES) until the process exits.
// Host code cannot use the array's name as a device address, so on the first
// call on each device (with that device current) the address is fetched with
// cudaGetSymbolAddress and cached per device.
#include <mutex>

#include "kvarn_common.cuh"

namespace {

constexpr size_t kScratchBytes = KVARN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, or NULL.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int kvarn_decode_attention_noalloc(const float* q, const uint8_t* tiles,
                                              int64_t tiles_bytes, const int64_t* tile_table,
                                              const int32_t* n_tiles, const float* win_k,
                                              const float* win_v, const int32_t* win_start,
                                              const int32_t* win_len, int win_capacity, int B,
                                              int Hq, int Hkv, int head_dim, int max_tiles,
                                              float softmax_scale, const kvarn_layout_t* layout,
                                              float* out, unsigned launch_flags,
                                              kvarn_stream_t stream) {
  // argument errors are reported before the scratch array is looked up
  if ((launch_flags & ~(KVARN_LAUNCH_PDL | KVARN_LAUNCH_PREFETCH)) ||
      ((launch_flags & KVARN_LAUNCH_PREFETCH) && !(launch_flags & KVARN_LAUNCH_PDL)) ||
      tiles_bytes < 0)
    return KVARN_ERR_BAD_ARG;
  size_t need = 0;
  int rc = kvarn_decode_workspace_bytes(B, Hq, Hkv, head_dim, max_tiles, win_capacity, &need);
  if (rc != KVARN_OK) return rc;
  if (need > kScratchBytes) return KVARN_ERR_WORKSPACE;  // the request is larger than the array
  void* ws = scratch_on_current_device();
  if (!ws) return KVARN_ERR_CUDA;
  return kvarn_decode_attention(q, tiles, tiles_bytes, tile_table, n_tiles, win_k, win_v,
                                win_start, win_len, win_capacity, B, Hq, Hkv, head_dim, max_tiles,
                                softmax_scale, layout, ws, kScratchBytes, out, launch_flags,
                                stream);
}
