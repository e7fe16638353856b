// Backward entry point that allocates nothing: the identity-STE backward with
// its scratch memory (the per-chunk state-gradient buffer and, for grouped
// heads, the per-value-head dq/dk partials) taken from a fixed array that the
// library owns, instead of a workspace the caller must allocate.
//
// Why: some callers cannot allocate device memory when they call the
// backward — for example a runtime that reserved the device's memory up front
// for its own pool and forbids further allocations, or code running where an
// allocation would have to synchronize the device.  Such callers can still
// pass their inputs and outputs, but not a workspace.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// this library holds GDN_NOALLOC_SCRATCH_BYTES of device memory for it until
// the process exits.  In host code its name is only a host-side stand-in, so
// the device address is looked up with cudaGetSymbolAddress (with the device
// current) on the first call made in each CUDA context, and kept per context:
// a context created later on the same device (e.g. after cudaDeviceReset) gets
// its own lookup.  Make the first call on a device before any stream capture.
// All calls share the one array, and it keeps the last call's contents: every
// scratch byte a call reads it has written first (each state-gradient slot and
// each dq/dk partial row is stored before it is loaded), so nothing needs
// clearing; calls that overlap on the GPU (e.g. on two streams) race.
#include <cuda.h>

#include <mutex>

#include "../../include/gdn_qdq.h"
#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[GDN_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point query (no link-time
// dependency on the driver library)
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

constexpr int kMaxContexts = 64;
std::mutex g_mu;
CUcontext g_ctx[kMaxContexts];  // contexts seen so far ...
void* g_addr[kMaxContexts];     // ... and the scratch array's device address in each
int g_n = 0;

// Device address of the scratch array in the current context (looked up once
// per context).
gdn_status scratch_address(void** out) {
  const CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return GDN_ERR_CUDA;
  if (!ctx) {
    // no context is current yet: the runtime makes the device's primary
    // context current on its first call, here the symbol lookup
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return GDN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_n; ++i)
    if (g_ctx[i] == ctx) {
      *out = g_addr[i];
      return GDN_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
  if (g_n < kMaxContexts) {
    g_ctx[g_n] = ctx;
    g_addr[g_n] = p;
    ++g_n;
  }
  *out = p;
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_chunk_bwd_ste_noalloc(const gdn_problem* p, const void* q, const void* k,
                                                const void* v, const float* beta, const float* g,
                                                const void* ctx, const void* dO, const float* dht,
                                                float* dq, float* dk, float* dv, float* dbeta,
                                                float* dg, float* dh0, void* stream) {
  const gdn_status s = gdn_validate(p);
  if (s != GDN_OK) return s;
  // Problems whose scratch exceeds the fixed array are rejected before any launch.
  if (gdn_bwd_workspace_bytes(p) > (size_t)GDN_NOALLOC_SCRATCH_BYTES)
    return GDN_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const gdn_status a = scratch_address(&scratch);
  if (a != GDN_OK) return a;
  return gdn_chunk_bwd_ste(p, q, k, v, beta, g, ctx, dO, dht, dq, dk, dv, dbeta, dg, dh0, scratch,
                           (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}
