// bwd_noalloc.cu -- attn_chunk_bwd_noalloc: the chunk-pair backward for
// callers that cannot allocate device memory at the point of the call.
//
// attn_chunk_bwd needs a caller-provided workspace for the per-row dot
// products delta_i = <dO_i, O_i>.  Some callers cannot obtain one: a plugin
// or extension running inside a host application that owns the device
// memory pool and gives its extensions no way to request more, or a
// latency-critical loop whose rules forbid any allocation once it has
// started.  This entry point takes the same tensors and uses a fixed array
// compiled into the library instead, so the caller supplies only inputs and
// outputs.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (16 MiB: delta for up to 4,194,304 query rows, e.g. 32 heads x 131,072
// tokens).  Every GPU that loads the library keeps it until the process
// exits.  When the row statistics and the fp32 dQ accumulator (or the
// sequence-contiguous copy of K) that attn_chunk_bwd uses for its faster
// path also fit, they go into the same array.  It is shared by all calls on
// a device and keeps the last call's contents.  What a call reads is
// written by that call first: the row-dot kernel rewrites the delta rows,
// the row statistics and the selector tiles; the K copy is rewritten by the
// transpose kernel; the dQ accumulator is cleared on the call's stream by
// the backward itself (cudaMemsetAsync, which allocates nothing) before the
// fused kernel adds into it.  Two calls whose work overlaps on the GPU (e.g.
// on two streams without an ordering between them) race on the array and
// produce wrong gradients.
//
// Set-up: the first call made on a device (with that device current) looks
// up the device address of the array with cudaGetSymbolAddress and caches
// it; that first call should come before any stream capture.  Under CUDA's
// default lazy module loading, that look-up (or the first kernel of this
// library run on the device) is also when the driver loads the library's
// module on that device and reserves the 16 MiB; a caller that must not
// take device memory after its start-up makes one small call during start-up.
// No call allocates: no cudaMalloc, cudaFree or allocating library routine.
#include <mutex>

#include "internal.h"

namespace lsx {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return LSX_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return LSX_ERR_DEVICE;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return LSX_OK;
}

}  // namespace
}  // namespace lsx

extern "C" size_t attn_chunk_bwd_noalloc_max_bytes(void) {
  return lsx::kNoAllocScratchBytes;
}

extern "C" int attn_chunk_bwd_noalloc(const lsx_tensor* q, const lsx_tensor* k,
                                      const lsx_tensor* v, const lsx_tensor* o,
                                      const lsx_tensor* lse, const lsx_tensor* d_o,
                                      int64_t q_off, int64_t kv_off, int causal,
                                      float scale, const lsx_tensor* dq,
                                      const lsx_tensor* dk, const lsx_tensor* dv,
                                      int accumulate, lsx_stream_t stream) {
  if (q == nullptr || k == nullptr) return LSX_ERR_NULL;
  const size_t need = attn_chunk_bwd_min_workspace_size(q, k);
  if (need > lsx::kNoAllocScratchBytes) return LSX_ERR_WORKSPACE;  // beyond the fixed array
  void* scratch = nullptr;
  const int rc = lsx::noalloc_scratch(&scratch);
  if (rc != LSX_OK) return rc;
  return attn_chunk_bwd(q, k, v, o, lse, d_o, q_off, kv_off, causal, scale, dq, dk, dv,
                        accumulate, scratch, lsx::kNoAllocScratchBytes, stream);
}
