// noalloc.cu -- paged_attention_forward_noalloc: the attention entry point for callers that
// cannot allocate device memory at the point of the call.
//
// paged_attention_forward needs a caller-provided workspace (launch plan + fp32 split-KV
// partials).  Some callers have no way to provide one: a plugin whose host framework owns all
// device memory and offers no workspace hook, or a latency-critical serving loop in which an
// allocator call (with its locks and possible implicit synchronisation) is not allowed.  For
// them this file keeps one fixed scratch buffer in device global memory, declared at file scope,
// and runs the unchanged attention path on it.
//
// Cost and rules of use:
//   * the buffer is PKV_NOALLOC_SCRATCH_BYTES (64 MiB) and exists on every GPU that loads this
//     library, until the process exits;
//   * a batch that needs more scratch than that is rejected with PKV_ERR_WORKSPACE before
//     anything is launched;
//   * the host cannot use the array's name as a device address, so the first call on each
//     device looks the address up with cudaGetSymbolAddress (with that device current) and
//     caches it; make that first call before any stream capture;
//   * every call shares the one buffer and leaves its contents behind.  Nothing in it has to
//     start at zero (the plan kernel rewrites every field the later kernels read), but two
//     calls whose kernels overlap on the GPU (different streams, or several threads) race on
//     it: serialise them on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "paged_kv.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return PKV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int paged_attention_forward_noalloc(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads,
                                               const void* q_rot, int64_t q_row_stride, void* out,
                                               float softmax_scale, int32_t* d_error, pkv_stream_t stream) {
  const size_t need = paged_attention_workspace_size(pool, batch, num_q_heads);
  if (need == 0) {
    // invalid arguments (or an empty batch): let the regular entry point report or no-op
    return paged_attention_forward(pool, batch, num_q_heads, q_rot, q_row_stride, out, softmax_scale, nullptr, 0,
                                   d_error, stream);
  }
  if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
  return paged_attention_forward(pool, batch, num_q_heads, q_rot, q_row_stride, out, softmax_scale, scratch,
                                 PKV_NOALLOC_SCRATCH_BYTES, d_error, stream);
}
