// kda_noalloc.cu -- kda_chunk_prefill_noalloc: the chunked prefill for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the prefill:
// plug-in hosts whose device allocator is owned by someone else, and real-time
// paths that forbid allocation after start-up.
// This entry point gives them the prefill with its scratch (the device status
// word, the work counter and the longest-first sequence order) taken from a
// fixed array that lives in the library's own device memory instead of a
// workspace they would have to allocate.  It allocates nothing: no cudaMalloc,
// no cudaFree, no allocating library routine.
#include <mutex>

#include "kda_internal.cuh"

namespace {

// Scratch shared by every call on a device; each GPU that loads the library holds
// it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device.  Host code may not
// use the symbol itself (it is a host-side stand-in, not a device address), so the
// address is looked up once per device, with that device current.
kda_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status_t kda_chunk_prefill_noalloc(const kda_desc_t* desc, const void* q,
                                                  const void* k, const void* v, const float* g,
                                                  const float* beta, const int32_t* cu_seqlens,
                                                  void* state, const int32_t* state_indices,
                                                  void* final_state, void* o,
                                                  cudaStream_t stream) {
  const size_t need = kda_chunk_prefill_min_workspace_size(desc);
  if (need == 0) return KDA_ERR_INVALID_ARGUMENT;
  if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const kda_status_t st = scratch_for_current_device(&scratch);
  if (st != KDA_OK) return st;
  return kda_chunk_prefill(desc, q, k, v, g, beta, cu_seqlens, state, state_indices, final_state,
                           o, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}
