// pda_noalloc.cu -- pda_decode_static: the decode call for callers that
// cannot give the library any device memory of its own.
//
// pda_decode needs a split_scratch buffer from its caller. Some callers have
// no way to make one: a plugin that its host framework hands only input and
// output pointers (the framework owns every device allocation and exposes no
// allocator to it), or a caller that must not call cudaMalloc at that point
// because its host enforces a fixed device-memory budget or forbids
// allocation on that path. For them this entry point keeps the split scratch
// in a fixed array that is part of the library's own device image, so the
// call allocates nothing.
//
// The array is PDA_STATIC_SCRATCH_BYTES long. Every GPU that loads the
// library holds it until the process exits. All calls share it and it keeps
// whatever the last call wrote: each call clears its status word first, and
// calls whose GPU work overlaps (two streams, or two host threads) race on
// it, so the caller must order them on one stream or otherwise serialise
// them. The first call on a device looks up the array's device address (with
// that device current) and caches it; make that first call before any
// stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "pda_internal.h"

namespace {

// The shared split scratch: status header, partial LSEs and partial outputs.
static __device__ __align__(256) unsigned char g_static_scratch[PDA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up once
// per device; host code cannot use the symbol itself as a device address).
int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return PDA_ERR_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return PDA_OK;
}

}  // namespace

extern "C" int pda_decode_static(const pda_plan_t* plan, const void* q, const void* k_pages,
                                 const void* v_pages, const int32_t* page_table,
                                 const int32_t* kv_indptr, const int32_t* kv_len,
                                 const int32_t* qo_indptr, int32_t max_q_len,
                                 const int32_t* window, float sm_scale, const float* k_scale,
                                 const float* v_scale, void* out, float* lse,
                                 pda_stream_t stream) {
  if (!plan) return PDA_ERR_NULL;
  if (plan->magic != PDA_PLAN_MAGIC) return PDA_ERR_PLAN;
  if (plan->scratch_bytes > (int64_t)PDA_STATIC_SCRATCH_BYTES) return PDA_ERR_TOO_LARGE;
  void* scratch = nullptr;
  int rc = static_scratch(&scratch);
  if (rc != PDA_OK) return rc;
  // The status word is the only part that must start at zero.
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  return pda_decode(plan, q, k_pages, v_pages, page_table, kv_indptr, kv_len, qo_indptr,
                    max_q_len, window, sm_scale, k_scale, v_scale, out, lse, scratch, stream);
}
