// attn_fwd_noalloc: the forward pass for callers that cannot allocate device
// memory themselves.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run attention: code embedded in a host framework that owns every byte
// of device memory through its own pool and forbids raw allocations, or a
// latency-critical path where an allocation's implicit device-wide
// synchronisation is not acceptable.  attn_fwd needs a small scratch buffer
// (the tile plan and the device status word); this variant takes it from a
// fixed-size array in the library's own device memory instead of from the
// caller.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds its kAttnNoAllocScratchBytes until the process exits.  In
// host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, with the caller's device
// current, on every call.  Once the library's module is loaded on a device
// that lookup allocates nothing; repeating it instead of caching the pointer
// keeps the address right after a cudaDeviceReset or a primary-context
// teardown, which load the module again at a new address.
#include "internal.h"

namespace {

constexpr size_t kAttnNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) uint8_t g_fwd_scratch[kAttnNoAllocScratchBytes];

// Device address of g_fwd_scratch on the current device, or null.
void* scratch_on_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess) return nullptr;
  return p;
}

}  // namespace

extern "C" GB300ATTN_API int attn_fwd_noalloc(const attn_fwd_params* p, attn_stream_t stream) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  attn_fwd_params q = *p;
  const size_t need = attn_fwd_workspace_bytes(p);
  if (need == 0) {
    // invalid or unsupported problem: attn_fwd reports which, launching nothing
    q.workspace = nullptr;
    q.workspace_bytes = 0;
    return attn_fwd(&q, stream);
  }
  if (need > kAttnNoAllocScratchBytes) return ATTN_ERR_UNSUPPORTED;
  void* ws = scratch_on_current_device();
  if (!ws) return ATTN_ERR_CUDA;
  q.workspace = ws;
  q.workspace_bytes = kAttnNoAllocScratchBytes;
  return attn_fwd(&q, stream);
}

// The status word of the scratch above on the current device: ATTN_OK, or
// ATTN_ERR_TIMEOUT when a bounded device-side wait of the last
// attn_fwd_noalloc on this device gave up (its outputs are then undefined).
extern "C" GB300ATTN_API int attn_fwd_noalloc_status(attn_stream_t stream) {
  void* ws = scratch_on_current_device();
  if (!ws) return ATTN_ERR_CUDA;
  return attn_read_device_status(ws, stream);
}
