// static_workspace.cu -- decode_attn_static_workspace(): decode attention
// for callers that cannot allocate device memory.
//
// decode_attn() asks the caller for a workspace (the fp32 partial outputs and
// log-sum-exps of the KV chunks).  Some callers have no way to provide one:
// plugin hosts that hand the library only the input and output buffers,
// runtimes whose device memory is owned end to end by another allocator, and
// deployments that forbid any device allocation after start-up.  This entry
// point takes the same inputs and outputs and keeps the partials in a
// fixed-size array that lives in this library's own device memory instead.
//
// Limits and sharing:
//   * the array holds DECODE_ATTN_STATIC_WORKSPACE_BYTES (16 MiB); every GPU
//     that loads the library holds it until the process exits;
//   * a call whose partials need more than that is rejected with
//     DA_ERR_STATIC_WORKSPACE_LIMIT before anything is launched;
//   * every call on a device uses the same array, so calls whose work
//     overlaps on the GPU (different streams, or other host threads) race on
//     it and must be serialised by the caller;
//   * the array keeps whatever the previous call left in it; nothing needs
//     clearing, because the combine step reads only partials that the split
//     pass of the same call has just written;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture on that device.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.

#include <cuda_runtime.h>

#include <mutex>

#include "decode_attn.h"

namespace {

constexpr size_t kStaticBytes = DECODE_ATTN_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The partials of one call: fp32 [rows, splits, 128] then [rows, splits].
static __device__ __align__(256) unsigned char g_static_workspace[kStaticBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices];  // device address of g_static_workspace, per device

// Device address of the array on the current device (looked up once).
int static_workspace_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return DA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr)
      return DA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DA_OK;
}

}  // namespace

extern "C" int decode_attn_static_workspace(const decode_attn_params* p, const void* q,
                                            const void* k_cache, const void* v_cache,
                                            const int32_t* block_table,
                                            const int32_t* seq_lens, void* out, float* lse,
                                            int32_t num_splits, int32_t* status,
                                            void* stream) {
  if (p == nullptr) return DA_ERR_NULL_POINTER;
  void* ws = nullptr;
  int rc = static_workspace_address(&ws);  // first call on a device: the lookup
  if (rc != DA_OK) return rc;
  int32_t splits = num_splits;
  if (splits <= 0) {
    int32_t chunk = 0;
    rc = decode_attn_plan(p, nullptr, &splits, &chunk);
    if (rc != DA_OK) return rc;
  }
  size_t need = 0;
  rc = decode_attn_workspace_bytes(p, splits, &need);
  if (rc != DA_OK) return rc;
  if (need > kStaticBytes) return DA_ERR_STATIC_WORKSPACE_LIMIT;
  return decode_attn(p, q, k_cache, v_cache, block_table, seq_lens, out, lse, splits, ws,
                     kStaticBytes, status, stream);
}
