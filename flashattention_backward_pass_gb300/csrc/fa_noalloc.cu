// fa_noalloc.cu — fa_bwd_noalloc: the backward with library-owned scratch, for callers
// that cannot allocate device memory.
//
// Who needs it: code that must not call cudaMalloc (or any allocator) at the point where
// it runs the backward — for example inside a serving or real-time loop where a device
// allocation would synchronize the device and stall other work, inside a region that is
// being recorded into a CUDA graph (cudaMalloc is not a capturable operation), or in an
// embedding that has a fixed device-memory budget and no allocator to hand the library.
// fa_bwd asks such callers for a workspace buffer; this entry point instead uses a
// fixed-size scratch array that lives in the library's own device memory.
//
// The scratch is one file-scope __device__ array of FA_NOALLOC_SCRATCH_BYTES (32 MiB).
// Every GPU that loads the library holds it until the process exits.  Problems whose
// workspace (fa_bwd_workspace_size) is larger are rejected with FA_ERR_WORKSPACE before
// anything is launched.  A bounded device-side wait that runs out records its code in the
// array's status word; fa_bwd_noalloc_status reads and clears it.
//
// Host code may not use the array's name as a device address (on the host it is only a
// stand-in symbol).  The first call on each device therefore looks the address up with
// cudaGetSymbolAddress while that device is current, checks the result and caches it;
// later calls on that device reuse the cached pointer.  Make that first call on a device
// outside any stream capture.
//
// Every call on a device shares the one array and leaves its contents behind.  The parts
// that must start at zero (dQ accumulator, ordering counters, status word, tile ticket)
// are cleared by the preprocess kernel at the start of every call, and the other parts
// are fully rewritten, so a call never reads a previous call's values.  Two calls whose
// kernels overlap on the GPU (different streams without ordering between them) race on
// the array: order them on one stream, or use fa_bwd with separate workspaces.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k,
                              const fa_tensor* v, const fa_tensor* out, const fa_tensor* lse,
                              fa_tensor* dq, fa_tensor* dk, fa_tensor* dv, float softmax_scale,
                              int causal, int window_left, int window_right, float softcap,
                              int deterministic, void* stream) {
  // fa_bwd validates every argument and returns FA_ERR_WORKSPACE, before any launch, for a
  // problem whose workspace does not fit the FA_NOALLOC_SCRATCH_BYTES it is given.
  void* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, causal, window_left,
                window_right, softcap, deterministic, scratch, (size_t)FA_NOALLOC_SCRATCH_BYTES,
                stream);
}

// The status word of the last fa_bwd_noalloc on the current device lives in the scratch
// array's header, where fa_bwd_status finds it once it has the array's device address.
extern "C" int fa_bwd_noalloc_status(void* stream, int* device_status) {
  if (!device_status) return FA_ERR_NULL;
  void* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd_status(scratch, stream, device_status);
}
