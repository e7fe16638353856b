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
// the device address is looked up with cudaGetSymbolAddress once per device
// (with that device current) on the first call made on that device; make that
// first call before any stream capture.  All calls share the one array, and it
// keeps the last call's contents: the launch path clears what must start at
// zero, and calls that overlap on the GPU (e.g. on two streams) race.
#include <mutex>

#include "../../include/gdn_qdq.h"
#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices];  // device address of g_bwd_scratch, per device

// Device address of the scratch array on the current device (looked up once).
gdn_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
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
