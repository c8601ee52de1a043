// mla_noalloc.cu -- a decode entry point for callers that cannot allocate device
// memory.
//
// mla_decode needs a caller-owned workspace (the sticky error word plus the
// fp32 split partials).  Some callers have no way to provide one: code that runs
// inside a host framework that owns every device allocation, or a plug-in that
// is handed only input and output pointers and may not call cudaMalloc itself.
// For them, mla_decode_noalloc runs the same two kernels with the workspace
// placed in a fixed-size array that lives in this library's device image.
//
// Limits and rules (also stated in include/mla_decode.h):
//   * The array holds MLA_NOALLOC_SCRATCH_BYTES (32 MiB).  Every GPU that loads
//     the library keeps that much device memory reserved until the process exits.
//   * A plan whose workspace_bytes exceeds it is rejected with
//     MLA_ERR_WORKSPACE_TOO_SMALL before anything is launched; plan with fewer
//     splits (force_splits) to fit.  A one-split plan needs only the header.
//   * All calls on a device share the one array.  Calls that can overlap on the
//     GPU (different streams without ordering) race on it; keep them ordered.
//   * The first call on a device looks up the array's device address and caches
//     it; make that first call before any stream capture begins.
//   * The error word is cleared at the start of each call, so a device-side input
//     error or a bounded wait that ran out is visible only as NaN rows of the
//     affected request.
//   * The cached address belongs to the device's context; after
//     cudaDeviceReset it is stale.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "mla_decode.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch workspace.  On the host this name is only a stand-in for the
// device symbol: its device address must come from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once.
mla_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_noalloc(const mla_decode_plan_t* plan, const void* q_nope,
                                           int64_t q_nope_row_stride, const void* q_pe,
                                           int64_t q_pe_row_stride, const void* kv_cache, int num_pages,
                                           const int32_t* block_table, int block_table_stride,
                                           const int32_t* seq_lens, float softmax_scale,
                                           const float* kv_scale, void* out, mla_out_dtype_t out_dtype,
                                           float* lse, void* cuda_stream) {
  // The plan is checked before anything touches the GPU: the scratch array's
  // bounds are only as good as the plan's byte counts.
  if (!mla::plan_valid(plan)) return MLA_ERR_INVALID_ARG;
  if (plan->workspace_bytes > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  mla_status_t st = scratch_for_current_device(&ws);
  if (st != MLA_OK) return st;
  // The previous call's error word must not leak into this one.
  if (cudaMemsetAsync(ws, 0, MLA_WORKSPACE_HEADER_BYTES, (cudaStream_t)cuda_stream) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return mla_decode(plan, q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_pages, block_table,
                    block_table_stride, seq_lens, softmax_scale, kv_scale, out, out_dtype, lse, ws,
                    (size_t)MLA_NOALLOC_SCRATCH_BYTES, cuda_stream);
}
