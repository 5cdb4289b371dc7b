// match_pair_noalloc: match_pair for callers that may not allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a host application
// which owns every device allocation (a plugin handed only its inputs and outputs),
// real-time loops where an allocation's implicit device synchronisation or its
// failure mid-run is not allowed, and tools that must keep their device footprint
// fixed from load time.  This entry point gives them matching with no workspace
// argument: the scratch lives in one file-scope __device__ array of fixed size that
// every GPU which loads the library holds until the process exits.
//
// The array's name in host code is a host-side stand-in, not a device address, so
// the device address is looked up with cudaGetSymbolAddress once per device (on the
// first call made with that device current) and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "serac.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SERAC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device (set-up on first use).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SERAC_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return SERAC_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SERAC_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SERAC_OK;
}

}  // namespace

extern "C" int match_pair_noalloc(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b,
                                  const serac_params* params, const serac_out* out, void* cuda_stream) {
  if (n_a < 0 || n_b < 0) return SERAC_EINVAL;
  if (serac_pair_workspace_size(n_a, n_b) > static_cast<size_t>(SERAC_NOALLOC_SCRATCH_BYTES))
    return SERAC_EWORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != SERAC_OK) return st;
  return match_pair(desc_a, n_a, desc_b, n_b, params, out, scratch, SERAC_NOALLOC_SCRATCH_BYTES, cuda_stream);
}
