// gns_gram_ns_batched_noalloc: Gram Newton-Schulz for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where they
// orthogonalize: code running inside a framework's memory pool that forbids allocations it
// does not own, real-time or embedded loops that must not allocate after start-up, and
// plug-ins that are handed device pointers but no allocator. For them this entry point
// takes the scratch memory that gns_gram_ns_batched needs from a fixed array compiled into
// the library instead of from a caller-provided workspace.
//
// The array lives in device global memory: every GPU on which the library's code is loaded
// reserves GNS_NOALLOC_SCRATCH_BYTES for it until the process exits. In host code its name
// is only a stand-in, not a device address, so its address is looked up once per device
// (cudaGetSymbolAddress, with that device current) on the first call made on that device;
// make that first call before any stream capture. All calls share the array and it keeps
// whatever the last call left there: the completion counters that must start at zero are
// reset by every call (a memset on the stream), and every other scratch value is written
// before it is read. Calls whose executions overlap on the GPU (different streams, or
// different host threads) race on the array and give wrong results: serialise them.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/gns.h"

namespace {

constexpr size_t kScratchBytes = GNS_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

}  // namespace

namespace gns {
int set_error(int code, const std::string& msg);  // sets gns_last_error(); defined with the C ABI
}

extern "C" {

GNS_API int gns_gram_ns_batched_noalloc(const gns_batch* x, const gns_batch* out, int ngroups, gns_dtype dtype,
                                        const gns_ns_params* ns, int32_t* dev_status, void* stream) {
  const size_t need = gns_workspace_size(GNS_OP_GRAM_NS, x, ngroups, dtype, ns, nullptr);
  if (need == 0) return GNS_ERR_INVALID;  // argument error, message already set
  if (need > kScratchBytes)
    return gns::set_error(GNS_ERR_WORKSPACE,
                          "gns_gram_ns_batched_noalloc: these batches need " + std::to_string(need) +
                              " bytes of scratch, more than the fixed " + std::to_string(kScratchBytes) +
                              " bytes (GNS_NOALLOC_SCRATCH_BYTES); split the batch or call gns_gram_ns_batched "
                              "with a workspace");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return gns::set_error(GNS_ERR_CUDA, "gns_gram_ns_batched_noalloc: no usable current device");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p)
        return gns::set_error(GNS_ERR_CUDA, std::string("gns_gram_ns_batched_noalloc: cudaGetSymbolAddress of "
                                                        "the scratch array failed: ") +
                                                cudaGetErrorString(e));
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return gns_gram_ns_batched(x, out, ngroups, dtype, ns, scratch, kScratchBytes, dev_status, stream);
}

}  // extern "C"
