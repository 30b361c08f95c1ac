// kda_fwd_noalloc: the forward pass with its scratch memory inside the library.
//
// kda_fwd needs a caller-provided device workspace.  Some callers cannot
// allocate device memory at the point where they run the forward pass: code
// running inside a host callback or a plugin with no allocator handle, host
// code that must not touch the caching allocator of the framework that owns
// the device, or deployments with a fixed memory budget that forbid runtime
// cudaMalloc.  For them this entry point takes the workspace from a
// fixed-size buffer compiled into the library (a file-scope __device__ array),
// so the call allocates nothing.  The buffer exists once per GPU that loads
// the library and stays allocated until the process exits.
#include <mutex>

#include "../../include/kda.h"

namespace {

// The built-in scratch.  In host code `g_noalloc_scratch` names a host-side
// stand-in, not device memory: its device address is obtained with
// cudaGetSymbolAddress once per device (below) and only that address is
// handed to the kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call per device), or nullptr on failure.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" int kda_fwd_noalloc(const kda_fwd_args* args, void* stream) {
  const size_t need = kda_fwd_workspace_bytes(args);
  if (need == 0)  // invalid arguments (reported by kda_fwd), or no scratch needed
    return kda_fwd(args, nullptr, 0, stream);
  if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_NOALLOC_LIMIT;
  void* scratch = scratch_address();
  if (!scratch) return KDA_ERR_LAUNCH;
  return kda_fwd(args, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}
