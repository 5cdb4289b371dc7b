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
// the device address is looked up with cudaGetSymbolAddress, with the device current,
// the first time a call runs in a CUDA context, and cached for that context.  The
// cache is keyed by the context's unique ID, not by the device ordinal: after
// cudaDeviceReset, or in another context on the same device, the module is loaded
// again at another address, and the new context's first call looks it up afresh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "serac.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SERAC_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

constexpr int kMaxDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id = 0;  // context the address belongs to (0: none yet)
  void* ptr = nullptr;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

template <typename Fn>
Fn driver_fn(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(f);
}

// Unique ID of the calling thread's current context; false if none is current yet.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// Device address of g_noalloc_scratch in the current context (set-up on first use in
// each context).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SERAC_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return SERAC_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& e = g_scratch[dev];
  unsigned long long id = 0;
  if (current_context_id(&id) && e.ptr && e.ctx_id == id) {
    *out = e.ptr;
    return SERAC_OK;
  }
  // look the address up (this also makes the runtime's context current on a thread
  // that has made no CUDA call yet), then record the context it belongs to
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SERAC_ECUDA;
  if (!current_context_id(&id)) return SERAC_ECUDA;
  e.ctx_id = id;
  e.ptr = p;
  *out = p;
  return SERAC_OK;
}

}  // namespace

extern "C" int match_pair_noalloc(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b,
                                  const serac_params* params, const serac_out* out, void* cuda_stream) {
  if (n_a < 0 || n_b < 0 || n_a > SERAC_MAX_N || n_b > SERAC_MAX_N || !params || params->max_features < 0)
    return SERAC_EINVAL;
  // the scratch must hold the workspace of the pair as it is matched (under the cap)
  const int32_t k = params->max_features;
  const int32_t ca = (k > 0 && n_a > k) ? k : n_a, cb = (k > 0 && n_b > k) ? k : n_b;
  if (serac_pair_workspace_size(ca, cb) > static_cast<size_t>(SERAC_NOALLOC_SCRATCH_BYTES))
    return SERAC_EWORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != SERAC_OK) return st;
  return match_pair(desc_a, n_a, desc_b, n_b, params, out, scratch, SERAC_NOALLOC_SCRATCH_BYTES, cuda_stream);
}
