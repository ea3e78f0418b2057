// noalloc.cu -- vsa_bwd_no_alloc: the backward for callers that cannot allocate device memory.
//
// Its scratch (the workspace vsa_bwd otherwise receives from the caller) is a file-scope static
// device array of VSA_BWD_NO_ALLOC_MAX_WORKSPACE_BYTES.  The array exists on every GPU that loads
// the library, from module load until the process exits.  Host code cannot use the symbol as a
// device address, so the first call on each device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and caches it; every call then runs the normal
// backward with that address as its workspace.  Nothing here allocates: no cudaMalloc, cudaFree
// or allocating library routine is called.
//
// All calls share the one array and the array keeps whatever the last call left in it.  The
// backward already clears, at its start, everything that must begin at zero (the error word,
// the per-head maxima; its preprocess zeroes the dQ accumulator), so stale contents do not leak
// into results.  Calls whose GPU work overlaps (different streams, or host threads racing) would
// write the same scratch at the same time: they race, and must be ordered by the caller.
#include <mutex>

#include "vsa_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[VSA_BWD_NO_ALLOC_MAX_WORKSPACE_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[MAX_DEVICES] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
vsa_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return vsa::record_cuda_failure(e);
  if (dev < 0 || dev >= MAX_DEVICES) return VSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_bwd_scratch);
    if (e != cudaSuccess || addr == nullptr) return vsa::record_cuda_failure(e);
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return VSA_OK;
}

}  // namespace

extern "C" vsa_status vsa_bwd_no_alloc(const void* dout, const void* q, const void* k,
                                       const void* v, const void* o, const float* lse,
                                       const int32_t* k2q_idx, const int32_t* k2q_num,
                                       int32_t max_q_blocks, const int32_t* vbs, float sm_scale,
                                       vsa_shape shape, void* dq, void* dk, void* dv,
                                       void* stream) {
  const size_t need = vsa_bwd_workspace_bytes(shape);
  if (need == 0)  // an invalid shape: vsa_bwd reports which check it fails, before any launch
    return vsa_bwd(dout, q, k, v, o, lse, k2q_idx, k2q_num, max_q_blocks, vbs, sm_scale, shape,
                   dq, dk, dv, nullptr, 0, stream);
  if (need > VSA_BWD_NO_ALLOC_MAX_WORKSPACE_BYTES) return VSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const vsa_status st = scratch_address(&scratch);
  if (st != VSA_OK) return st;
  return vsa_bwd(dout, q, k, v, o, lse, k2q_idx, k2q_num, max_q_blocks, vbs, sm_scale, shape, dq,
                 dk, dv, scratch, VSA_BWD_NO_ALLOC_MAX_WORKSPACE_BYTES, stream);
}

extern "C" vsa_status vsa_bwd_no_alloc_device_error(uint32_t* bits, void* stream) {
  if (!bits) return VSA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  vsa_status st = scratch_address(&scratch);
  if (st != VSA_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return vsa::record_cuda_failure(e);
  e = cudaMemcpy(bits, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? VSA_OK : vsa::record_cuda_failure(e);
}
