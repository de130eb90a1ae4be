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
// them. The status word of the array is read and cleared by pda_get_status
// and pda_reset_status with split_scratch = NULL.
//
// Host code cannot use the array's symbol as a device address: its device
// address is looked up with the plan's device current, on every call whose
// stream is not capturing a graph (so a device reset, which may move the
// array, is followed). A call made while its stream is capturing reuses the
// address of the last lookup on that device, so the first call on a device
// must come before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "pda_internal.h"

namespace {

// The shared split scratch: status header, partial LSEs and partial outputs.
static __device__ __align__(256) unsigned char g_static_scratch[PDA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_addr[kMaxDevices] = {};

}  // namespace

namespace pda {

int static_scratch(int device, cudaStream_t s, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  // the array is per device: the plan's device must be the current one
  if (dev != device || dev < 0 || dev >= kMaxDevices) return PDA_ERR_INVALID;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> guard(g_lock);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return PDA_ERR_CUDA;
    }
    g_addr[dev] = p;
  } else if (!g_addr[dev]) {
    return PDA_ERR_CUDA;  // never looked up outside a capture
  }
  *out = g_addr[dev];
  return PDA_OK;
}

}  // namespace pda

extern "C" int pda_decode_static(const pda_plan_t* plan, const void* q, const void* k_pages,
                                 const void* v_pages, const int32_t* page_table,
                                 const int32_t* kv_indptr, const int32_t* kv_len,
                                 const int32_t* qo_indptr, int32_t max_q_len,
                                 const int32_t* window, float sm_scale, const float* k_scale,
                                 const float* v_scale, void* out, float* lse,
                                 pda_stream_t stream) {
  // every host-side check first: a refused call touches nothing on the device
  int rc = pda::check_decode_args(plan, q, k_pages, v_pages, page_table, kv_indptr, kv_len,
                                  qo_indptr, max_q_len, k_scale, v_scale, out, lse);
  if (rc != PDA_OK) return rc;
  if (plan->scratch_bytes > (int64_t)PDA_STATIC_SCRATCH_BYTES) return PDA_ERR_TOO_LARGE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  rc = pda::static_scratch(plan->device, s, &scratch);
  if (rc != PDA_OK) return rc;
  // The status word is the only part that must start at zero.
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  return pda_decode(plan, q, k_pages, v_pages, page_table, kv_indptr, kv_len, qo_indptr,
                    max_q_len, window, sm_scale, k_scale, v_scale, out, lse, scratch, stream);
}
