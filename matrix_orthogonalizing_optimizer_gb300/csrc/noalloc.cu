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
// is only a stand-in, not a device address, so every call outside stream capture looks its
// address up (cudaGetSymbolAddress, with the call's device current) and remembers it per
// device; a call recorded by stream capture, which may not make that query, uses the
// remembered address, so the first call on a device must come before any capture (a first
// call under capture is refused with a message saying so). Looking the address up again on
// every uncaptured call keeps it valid after a cudaDeviceReset, which unloads the module and
// may place the array elsewhere when it is loaded again. All calls share the array and it keeps
// whatever the last call left there: the completion counters that must start at zero are
// reset by every call (a memset on the stream, or the norm pass enqueued just before the
// GEMM), and every other scratch value is written before it is read. Calls whose executions overlap on the GPU (different streams, or
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
int plan_workspace(gns_op op, const gns_batch* x, int ngroups, gns_dtype dtype, const gns_ns_params* ns,
                   const gns_muon_params* muon, size_t* need);
}

extern "C" {

GNS_API int gns_gram_ns_batched_noalloc(const gns_batch* x, const gns_batch* out, int ngroups, gns_dtype dtype,
                                        const gns_ns_params* ns, int32_t* dev_status, void* stream) {
  size_t need = 0;
  const int prc = gns::plan_workspace(GNS_OP_GRAM_NS, x, ngroups, dtype, ns, nullptr, &need);
  if (prc) return prc;  // invalid or unsupported request, message already set
  if (need > kScratchBytes)
    return gns::set_error(GNS_ERR_WORKSPACE,
                          "gns_gram_ns_batched_noalloc: these batches need " + std::to_string(need) +
                              " bytes of scratch, more than the fixed " + std::to_string(kScratchBytes) +
                              " bytes (GNS_NOALLOC_SCRATCH_BYTES); split the batch or call gns_gram_ns_batched "
                              "with a workspace");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return gns::set_error(GNS_ERR_CUDA, "gns_gram_ns_batched_noalloc: no usable current device");
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap) != cudaSuccess)
    return gns::set_error(GNS_ERR_CUDA, "gns_gram_ns_batched_noalloc: cudaStreamIsCapturing failed on the stream");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (cap == cudaStreamCaptureStatusNone) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p)
        return gns::set_error(GNS_ERR_CUDA, std::string("gns_gram_ns_batched_noalloc: cudaGetSymbolAddress of "
                                                        "the scratch array failed: ") +
                                                cudaGetErrorString(e));
      g_scratch_ptr[dev] = p;
    } else if (!g_scratch_ptr[dev]) {
      return gns::set_error(GNS_ERR_INVALID,
                            "gns_gram_ns_batched_noalloc: the first call on a device must run outside stream "
                            "capture (it looks up the scratch array's device address, which a capture cannot)");
    }
    scratch = g_scratch_ptr[dev];
  }
  return gns_gram_ns_batched(x, out, ngroups, dtype, ns, scratch, kScratchBytes, dev_status, stream);
}

}  // extern "C"
