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
//   * the array's device address is looked up (cudaGetSymbolAddress, with
//     the device current) by the first call in each CUDA context and cached
//     under that context's unique id: normally once per device, again after
//     cudaDeviceReset (the module is reloaded, possibly elsewhere) or when a
//     driver-API caller makes another context current.  Make that first call
//     before any stream capture in that context.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "decode_attn.h"

namespace {

constexpr size_t kStaticBytes = DECODE_ATTN_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The partials of one call: fp32 [rows, splits, 128] then [rows, splits].
static __device__ __align__(256) unsigned char g_static_workspace[kStaticBytes];

// Driver entry points (fetched through the runtime: the library does not
// link libcuda) that name the current context and its process-unique id.
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_entry_once;

void load_entry_points() {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  f = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
}

// Unique id of the calling thread's current context (0: none or unknown).
unsigned long long current_context_id() {
  std::call_once(g_entry_once, load_entry_points);
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct Cached {
  unsigned long long ctx_id;  // context the address belongs to (0: none)
  void* addr;
};
std::mutex g_mu;
Cached g_addr[kMaxDevices];

// Device address of the array in the current context, looked up (with the
// device current) on the first call in each context.
int static_workspace_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return DA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  const unsigned long long id = current_context_id();
  Cached& c = g_addr[dev];
  if (id == 0 || c.ctx_id != id || c.addr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr)
      return DA_ERR_CUDA;
    // the lookup made the runtime's context current if none was: name it now
    c.ctx_id = id != 0 ? id : current_context_id();
    c.addr = p;
  }
  *out = c.addr;
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
  int rc = static_workspace_address(&ws);  // first call in a context: the lookup
  if (rc != DA_OK) return rc;
  int32_t splits = num_splits;
  if (splits <= 0) {
    int32_t chunk = 0;
    rc = decode_attn_plan(p, nullptr, &splits, &chunk);
    if (rc != DA_OK) return rc;
  }
  // only a call that writes partials (two launches: split + combine) uses
  // the array; a single-chunk or cluster-merged call is never rejected
  const int launches = decode_attn_launch_count(p, splits);
  if (launches < 0) return launches;
  size_t need = 0;
  if (launches == 2) {
    rc = decode_attn_workspace_bytes(p, splits, &need);
    if (rc != DA_OK) return rc;
    if (need > kStaticBytes) return DA_ERR_STATIC_WORKSPACE_LIMIT;
  }
  return decode_attn(p, q, k_cache, v_cache, block_table, seq_lens, out, lse, splits, ws,
                     kStaticBytes, status, stream);
}
