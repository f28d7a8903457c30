// ar_execute_noalloc: the all-reduce for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain the workspace that ar_execute asks for:
// their device memory belongs to another allocator (a framework's caching
// pool, or a fixed budget handed out by a host application) and they are not
// allowed to call cudaMalloc themselves, or they sit on a latency-sensitive
// path where cudaMalloc may implicitly synchronise the device. The bf16
// step-by-step executors are the only plans that need scratch memory (their
// fp32 partial sums). This entry point gives those callers a workspace that
// already exists: a fixed array in the library's own device memory, of
// AR_STATIC_WORKSPACE_BYTES bytes, which every GPU that loads the library
// holds until the process exits.
//
// It runs exactly the same kernels as ar_execute; only the workspace pointer
// differs. The first call on a device that needs the array looks up its
// address there; with lazy module loading that is when the module is loaded
// on the device and the array reserved, so callers make one warm-up call at
// start-up, before a pool takes the device's memory and before any capture.
#include <mutex>

#include "internal.h"

namespace {

// The shared scratch array. In host code this name is a host-side stand-in,
// not a device address: host code must look up its device address with
// cudaGetSymbolAddress (done once per device below) and pass that on.
static __device__ __align__(256) unsigned char g_noalloc_workspace[AR_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};  // device address of the array, per device

// Look up the array's device address on the current device, once.
ar_status workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AR_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return AR_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_workspace);
    if (err != cudaSuccess || ptr == nullptr) return AR_ECUDA;
    g_addr[dev] = ptr;
  }
  *out = g_addr[dev];
  return AR_OK;
}

}  // namespace

extern "C" ar_status ar_execute_noalloc(const ar_plan_t* plan, void* const* bufs, void* const* outs,
                                        void* stream) {
  if (plan == nullptr) return AR_EINVAL;
  ar_stats st;
  if (ar_plan_stats(plan, &st) != AR_OK) return AR_EINVAL;
  if (st.workspace_bytes > AR_STATIC_WORKSPACE_BYTES) return AR_EINVAL;  // too large for the array
  void* ws = nullptr;
  if (st.workspace_bytes > 0) {
    const ar_status s = workspace_address(&ws);
    if (s != AR_OK) return s;
  }
  return ar_execute(plan, bufs, outs, ws, stream);
}
