// fa_noalloc.cu -- fa_bwd_noalloc: the backward for callers that cannot
// allocate device memory.  Its workspace (the fp32 dQ accumulator and the
// -D and -LSE vectors) lives in a static device array of this translation
// unit, so the array belongs to a module of its own: under lazy module
// loading (the CUDA runtime's default) a device reserves it only once this
// entry point is first called there, not when libfa.so is merely loaded.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_common.cuh"

namespace {

constexpr int kMaxDevices = 64;

// File-scope device array: in host code its name is only a stand-in, so the
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

struct ScratchState {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchState g_scratch[kMaxDevices];

// Device address of the scratch array on the current device (looked up the
// first time this device asks, with the device current).
int scratch_ready(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  ScratchState& st = g_scratch[dev];
  std::call_once(st.once, [&] { st.err = cudaGetSymbolAddress(&st.ptr, g_noalloc_scratch); });
  if (st.err != cudaSuccess || st.ptr == nullptr) return FA_ERR_CUDA;
  *out = st.ptr;
  return FA_OK;
}

// The scratch array and the kernels belong to the current device, so the
// tensors must live there too.
int on_current_device(const void* p) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_INVALID;
  }
  return (a.type == cudaMemoryTypeDevice && a.device == dev) ? FA_OK : FA_ERR_INVALID;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                              float scale, int causal, fa_stream_t stream) {
  int rc;
  if ((rc = fa::api_check_shape(B, H, N, d)) != FA_OK) return rc;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0) return FA_ERR_INVALID;
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH;
  if ((rc = fa::api_check_bwd_args(q, k, v, o, dout, lse, dq, dk, dv, scale)) != FA_OK) return rc;
  if ((rc = fa::api_device_ready()) != FA_OK) return rc;
  if ((rc = on_current_device(q)) != FA_OK) return rc;
  void* ws = nullptr;
  if ((rc = scratch_ready(&ws)) != FA_OK) return rc;
  return fa::api_bwd(q, k, v, o, dout, lse, dq, dk, dv, ws, B, H, N, d, scale, causal,
                     reinterpret_cast<cudaStream_t>(stream));
}
