// decode_attn_forward_static: the whole forward pass (plan, split kernel,
// combine) for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: code loaded as a plugin into
// a host process that owns every device allocation and forbids its plugins
// from making their own, or latency-critical paths that cannot afford the
// implicit device synchronisation a cudaMalloc may cause.  They still own q,
// the caches, the index tables and the outputs; only the scratch workspace
// (plan arrays and split partials) is taken from the fixed array below.
#include <mutex>

#include "common.cuh"

// The scratch workspace of this entry point.  Every device on which this
// module is loaded holds it (with CUDA's lazy module loading: from the first
// call of the entry point on that device) until the process exits.
static __device__ __align__(256) unsigned char g_static_workspace[DA_STATIC_WORKSPACE_BYTES];

namespace {

std::mutex g_mu;
void* g_addr[64];

// Device address of g_static_workspace on the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in,
// so the address must come from the runtime.  The cached address belongs to
// the device's current context: after cudaDeviceReset it is stale, and this
// entry point must not be called again in that process.
int static_workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return DA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DA_OK;
}

}  // namespace

extern "C" int decode_attn_forward_static(const da_problem* prob, int32_t policy, const void* q,
                                          const void* k, const void* v, const int32_t* table,
                                          const int32_t* lengths, void* out, float* lse,
                                          void* stream, da_plan* plan_out) {
  size_t need = 0;
  int rc = decode_attn_workspace_bytes(prob, &need);
  if (rc != DA_OK) return rc;
  if (need > (size_t)DA_STATIC_WORKSPACE_BYTES) return DA_ERR_WORKSPACE;
  void* ws = nullptr;
  rc = static_workspace_address(&ws);
  if (rc != DA_OK) return rc;
  da_plan plan;
  rc = decode_attn_plan(prob, policy, lengths, ws, (size_t)DA_STATIC_WORKSPACE_BYTES, &plan,
                        stream);
  if (rc != DA_OK) return rc;
  rc = decode_attn_run(&plan, q, k, v, table, lengths, out, lse, stream);
  if (rc != DA_OK) return rc;
  rc = decode_attn_combine(&plan, out, lse, stream);
  // The plan names the array's device address, so decode_attn_read_error can
  // read this call's error word from it (until the next call overwrites it).
  if (rc == DA_OK && plan_out) *plan_out = plan;
  return rc;
}
