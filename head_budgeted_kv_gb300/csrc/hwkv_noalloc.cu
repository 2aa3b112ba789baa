// Decode attention for callers that must not allocate device memory.
//
// hwkv_decode_attn takes its split-K scratch (the per-split partial results) from a
// workspace the caller allocates.  Some callers cannot do that at the point where they run
// attention: code that runs while a CUDA graph is being captured (a cudaMalloc there breaks
// or invalidates the capture), runtimes whose memory is entirely owned by a pool allocator
// that must not be bypassed, and plugin hosts that forbid device allocation once inference
// has started.  hwkv_decode_attn_noalloc gives them the same computation with the scratch
// taken from a fixed array compiled into this library, so the call itself allocates
// nothing.  Inputs and outputs are still passed in by the caller.
#include <cstdint>
#include <mutex>

#include "hwkv_internal.h"
#include "../../include/hwkv.h"

namespace {

// The scratch array.  It lives in this file's own device module.  Under CUDA's lazy module
// loading (the default) that module is loaded on a device -- and the 4 MiB committed there --
// by the first address lookup below, i.e. the first call of the entry point on that device;
// with eager loading, when the library is loaded.  Either way the bytes stay committed until
// the process exits.
constexpr uint64_t kScratchBytes = HWKV_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};  // device address of g_decode_scratch, per device

// Device address of the scratch array on the current device.  The array's name is only a
// host-side stand-in for the symbol; the address the kernels need comes from the runtime,
// looked up once per device with that device current.
int scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return hwkv::set_error(HWKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return hwkv::set_error(HWKV_ERR_UNSUPPORTED, "device %d: only devices 0..%d are supported", dev, kMaxDevices - 1);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess)
      return hwkv::set_error(HWKV_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return HWKV_OK;
}

}  // namespace

extern "C" int hwkv_decode_attn_noalloc(hwkv_pool_t pool, int layer, const void* q, int q_heads, float scale,
                                        const int32_t* lens_dev, void* out, void* stream) {
  uint64_t need = 0;
  int rc = hwkv_decode_workspace_bytes(pool, q_heads, &need);
  if (rc != HWKV_OK) return rc;
  if (need > kScratchBytes)
    return hwkv::set_error(HWKV_ERR_WORKSPACE_TOO_SMALL,
                           "this decode configuration needs %llu bytes of scratch; the static scratch of "
                           "hwkv_decode_attn_noalloc holds %llu bytes (use hwkv_decode_attn with a workspace)",
                           (unsigned long long)need, (unsigned long long)kScratchBytes);
  // the address is cached per device: look it up only with the pool's own device current
  if (!pool) return hwkv::set_error(HWKV_ERR_INVALID_ARG, "pool is NULL");
  rc = hwkv::check_pool_device(pool);
  if (rc != HWKV_OK) return rc;
  void* scratch = nullptr;
  rc = scratch_on_current_device(&scratch);
  if (rc != HWKV_OK) return rc;
  return hwkv_decode_attn(pool, layer, q, q_heads, scale, lens_dev, out, scratch, kScratchBytes, stream);
}
