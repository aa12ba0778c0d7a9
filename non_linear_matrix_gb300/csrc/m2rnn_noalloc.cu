// m2rnn_noalloc.cu -- m2rnn_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or an allocating library routine at
// the point where they need gradients: code running while a memory pool is
// frozen or exhausted, code inside a framework whose allocator must not be
// re-entered from this call, or a runtime that only hands out pre-registered
// buffers.  m2rnn_bwd needs a caller-provided workspace when it has to
// recompute checkpoints; this entry point instead keeps them in a fixed
// buffer compiled into the library, so it performs no allocation at all.
//
// The buffer is a file-scope static __device__ array of
// M2RNN_NOALLOC_SCRATCH_BYTES (64 MiB).  Every GPU that loads this part of the
// library holds it until the process exits.  Host code must not use the
// array's name as a device address (in host code it is only a stand-in); the
// device address is obtained once per device with cudaGetSymbolAddress,
// with that device current, on the first call made on that device, and kept
// for the life of the process (a cudaDeviceReset of that device would make
// it stale: the library must not be used on a device again after a reset).
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "m2rnn.h"
#include "m2rnn_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = M2RNN_NOALLOC_SCRATCH_BYTES;  // per GPU

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device, with that device current).  Returns nullptr on failure.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

int m2rnn_bwd_noalloc(const m2rnn_shape* s, const void* q, const void* k, const void* v,
                      const void* f, const void* W, const void* w_r, const float* H0,
                      const void* dy, const float* dH_T, float* dq, float* dk, float* dv,
                      float* df, float* dW, float* dw_r, float* dH0, void* stream) {
  // Host-side checks first, so that a bad argument is refused before any
  // CUDA call (the scratch set-up below may load the module on the device).
  const int rc = m2rnn::validate_shape(s);
  if (rc != M2RNN_OK) return rc;
  if (s->ckpt_every <= 0) return M2RNN_ERR_INVALID_ARG;
  // Checkpoints are recomputed into the built-in buffer: refuse problems
  // whose checkpoints do not fit.
  const size_t need = m2rnn_bwd_workspace_size(s, 0);
  if (need > kNoAllocScratchBytes) return M2RNN_ERR_WORKSPACE;
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return M2RNN_ERR_CUDA;
  return m2rnn_bwd(s, q, k, v, f, W, w_r, H0, nullptr, dy, dH_T, dq, dk, dv, df, dW, dw_r, dH0,
                   nullptr, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
