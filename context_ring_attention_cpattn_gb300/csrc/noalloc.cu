// cpattn_prefill_noalloc: CP prefill whose workspace is a fixed buffer inside
// the library instead of memory the caller allocates.
//
// Some callers cannot call cudaMalloc: code embedded in a host framework that
// owns every byte of device memory through its own pool and forbids raw
// allocations, or a latency-critical loop where cudaMalloc's implicit device
// synchronisation and allocator locking are not acceptable.  Such callers
// still pass inputs and outputs; the Pass-KV accumulator or the Pass-Q partial
// stack lives in the file-scope array below.  The paper has no counterpart:
// this is an interface convenience of this library.
//
// The array is ordinary static device memory: every GPU on which this code
// is loaded holds CPATTN_NOALLOC_SCRATCH_BYTES until the process exits.  In
// host code its name is only a host-side stand-in, so its device address is
// obtained with cudaGetSymbolAddress (with the device current) on the first
// call in each CUDA context of a device, and passed on as the workspace
// pointer.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "cpattn.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[CPATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// The driver's cuCtxGetCurrent, looked up once (no link-time dependency on
// the driver library).
CtxGetCurrentFn ctx_get_current_fn() {
  static const CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(ptr);
    return nullptr;
  }();
  return fn;
}

// Device address of the scratch array on the current device.  It is looked
// up (cudaGetSymbolAddress, with the device current) on the first call in
// each CUDA context of the device and cached for that context: after a
// cudaDeviceReset the module is loaded again, the context changes and the
// address is looked up again.  nullptr on failure.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) return nullptr;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (ctx == nullptr || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    // (Also makes the device's primary context current if none was.)
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" cpattn_status cpattn_prefill_noalloc(const cpattn_tensor *q, const cpattn_tensor *k,
                                                const cpattn_tensor *v, int64_t q_base,
                                                int n_chunks, int mode, int causal, float scale,
                                                cpattn_tensor *o, float *lse, void *stream) {
  size_t need = 0;
  cpattn_status s = cpattn_prefill_workspace_size(q, k, q_base, n_chunks, mode, causal, &need);
  if (s != CPATTN_OK) return s;
  if (need > (size_t)CPATTN_NOALLOC_SCRATCH_BYTES) return CPATTN_ERR_UNSUPPORTED;
  void *ws = nullptr;
  if (need > 0) {
    ws = scratch_on_current_device();
    if (ws == nullptr) return CPATTN_ERR_CUDA;
  }
  // Nothing in the workspace has to start at zero: the first contribution to
  // each accumulator row and every Pass-Q partial overwrite their slots.
  return cpattn_prefill(q, k, v, q_base, n_chunks, mode, causal, scale, o, lse, ws,
                        (size_t)CPATTN_NOALLOC_SCRATCH_BYTES, stream);
}
