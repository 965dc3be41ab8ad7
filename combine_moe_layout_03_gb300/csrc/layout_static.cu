// layout_static.cu -- moe_layout_noalloc: the routing layout without a
// caller-supplied workspace.
//
// Some callers of this library cannot hand it device memory for scratch: a
// plugin running inside a host program that owns every device allocation
// through its own pool and forbids direct cudaMalloc, or a service that fixes
// its device footprint at start-up and must not allocate afterwards (a
// cudaMalloc/cudaFree can also stall the device at the wrong moment). For
// them this file keeps the layout's scratch in a fixed array that lives in
// the library's own device image: it is reserved on every GPU that loads the
// library and held until the process exits, and no call here allocates.
//
// The scratch is shared by every call. The layout kernels overwrite every
// scratch word they later read (per-chunk counts, flags and the status word),
// so nothing has to be cleared between calls. Calls that overlap on the GPU
// (on different streams, or from different host threads without ordering)
// race on the array and give wrong results.
#include <mutex>

#include "moe_internal.cuh"

namespace {

// The layout's scratch: status word, per-chunk expert counts [C][E], per-chunk
// rank counts [C][R] and flags [C], with C = ceil(N / 128).
static __device__ __align__(256) uint8_t g_layout_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device, looked up once
// per device (the host-side name of the array is not a device address) and
// kept for the life of the process: a cudaDeviceReset while the library is
// loaded would leave a stale address here, so it is not supported.
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_layout_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_layout_noalloc(const moe_desc_t* desc, const int32_t* topk_idx,
                                  int32_t* tokens_per_expert, int32_t* tokens_per_rank,
                                  uint8_t* is_token_in_rank, int32_t* expert_offset,
                                  int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot,
                                  int32_t* status, moe_stream_t stream) {
  if (!desc) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_workspace_size(desc);
  if (need == 0) return MOE_ERR_SHAPE;
  if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_TOO_LARGE;
  if (status && ((uintptr_t)status & 3)) return MOE_ERR_ALIGNMENT;
  void* scratch = nullptr;
  int rc = scratch_on_current_device(&scratch);
  if (rc != MOE_OK) return rc;
  rc = moe_layout(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank,
                  expert_offset, rank_offset, slot_of, src_of_slot, scratch,
                  (size_t)MOE_NOALLOC_SCRATCH_BYTES, stream);
  if (rc != MOE_OK || !status) return rc;
  // the status word is the first word of the scratch
  cudaError_t e = cudaMemcpyAsync(status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                  (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
