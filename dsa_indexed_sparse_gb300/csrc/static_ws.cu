// dsa_decode_step_static_ws: the decode step with its scratch memory in a
// library-owned device array, for callers that cannot allocate device memory.
//
// Who needs it: host code that has no way to call cudaMalloc for the step's
// scratch -- for example a plugin running inside an engine that owns all device
// memory and hands plugins no allocator, or a caller whose memory pool is fixed
// once at start-up and may not grow afterwards.  Such a caller still owns every
// input and output buffer; only the scratch (the score rows, the selected
// indices when idx_out is NULL, and the attention partials of split rows) lives
// in the array below.
//
// Costs and rules:
//  * DSA_STATIC_WORKSPACE_BYTES (32 MiB) of device memory is reserved on every GPU
//    that loads this library, for as long as the process lives.
//  * The first call on a device looks up that device's address of the array
//    (cudaGetSymbolAddress, with that device current); make this first call
//    before any stream capture is started on the device.
//  * All calls share the one array and it keeps whatever the last call wrote.
//    Nothing in it needs to start at zero: the step writes every scratch value
//    before reading it.  Calls whose work overlaps on the GPU (two streams, or
//    two host threads) race on the array; serialise them.
//  * Requests beyond DSA_STATIC_WORKSPACE_BYTES fail with DSA_ERR_WORKSPACE; the call
//    never allocates (no cudaMalloc / cudaFree, no allocating library routine).
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "dsa.h"
#include "dsa_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = DSA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mu;
void* g_ws_ptr[kMaxDevices] = {nullptr};

// Device address of the array on the current device (looked up once per device).
dsa_status_t static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    dsa::set_last_error(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    dsa::set_last_error("device ordinal out of range for the static workspace table");
    return DSA_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ws_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr) {
      dsa::set_last_error(std::string("cudaGetSymbolAddress(static workspace): ") + cudaGetErrorString(e));
      return DSA_ERR_CUDA;
    }
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" {

dsa_status_t dsa_decode_step_static_ws(const dsa_seq_desc_t* seq, const dsa_indexer_desc_t* idx,
                                       const dsa_mla_desc_t* mla, int32_t K, void* out, float* lse,
                                       int32_t* idx_out, dsa_stream_t stream) {
  size_t need = 0;
  const dsa_status_t chk = dsa::decode_workspace_need(seq, mla, K, &need);
  if (chk != DSA_OK) return chk;   // the same status (and dsa_last_error text) dsa_decode_step gives
  if (need > kStaticWorkspaceBytes) {
    char buf[160];
    snprintf(buf, sizeof(buf),
             "static workspace too small: this step needs %zu bytes, the library reserves %zu; "
             "use dsa_decode_step with a caller-provided workspace",
             need, kStaticWorkspaceBytes);
    dsa::set_last_error(buf);
    return DSA_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  const dsa_status_t st = static_workspace(&ws);
  if (st != DSA_OK) return st;
  return dsa_decode_step(seq, idx, mla, K, out, lse, idx_out, ws, kStaticWorkspaceBytes, stream);
}

}  // extern "C"
