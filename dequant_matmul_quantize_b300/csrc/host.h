// Host-side error reporting and kernel launch shared by every entry point.
//
// Every CUDA runtime or driver call the library makes goes through
// cuda_check / cu_check: a failure becomes NF4Q_ERR_CUDA and its text (the
// call and the error's name) is kept per thread for nf4q_last_cuda_error.
// Kernels are launched with cudaLaunchKernelEx, whose return value is that
// launch's own status: the library never reads the thread's sticky "last
// error", which another call on the same thread may have left behind.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>

#include "nf4q.h"

namespace nf4q {

inline char* last_error_text() {
  static thread_local char text[256] = {0};
  return text;
}

inline nf4q_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return NF4Q_OK;
  std::snprintf(last_error_text(), 256, "%s: %s (%d): %s", what, cudaGetErrorName(e),
                static_cast<int>(e), cudaGetErrorString(e));
  return NF4Q_ERR_CUDA;
}

inline nf4q_status cu_check(CUresult r, const char* what) {
  if (r == CUDA_SUCCESS) return NF4Q_OK;
  std::snprintf(last_error_text(), 256, "%s: CUresult %d", what, static_cast<int>(r));
  return NF4Q_ERR_CUDA;
}

inline nf4q_status cuda_fail(const char* what) {
  std::snprintf(last_error_text(), 256, "%s", what);
  return NF4Q_ERR_CUDA;
}

// Make the current device's primary context current on the calling thread.
// The tensor-map encoder is a driver call and needs a current context; a
// thread whose CUDA calls so far did not bind one (another library's runtime
// may only have asked for the device number, as on a fresh autograd worker
// thread) has none, and the encoder would fail with an invalid-context
// error.  cudaSetDevice binds the primary context; it is called only when
// no context is current.
inline nf4q_status ensure_context() {
  using CtxGetCurrentFn = CUresult (*)(CUcontext*);
  static const CtxGetCurrentFn get_current = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return static_cast<CtxGetCurrentFn>(nullptr);
  }();
  if (!get_current) return cuda_fail("cuCtxGetCurrent: driver entry point not found");
  CUcontext ctx = nullptr;
  nf4q_status st = cu_check(get_current(&ctx), "cuCtxGetCurrent");
  if (st != NF4Q_OK || ctx) return st;
  int dev = 0;
  if ((st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) != NF4Q_OK) return st;
  return cuda_check(cudaSetDevice(dev), "cudaSetDevice (bind the primary context)");
}

// Unique id of the calling thread's current context (cuCtxGetId: unique over
// the process lifetime, unlike the CUcontext handle, whose value may be
// reused after a context is destroyed).  *id = 0 when no context is current.
inline nf4q_status current_context_id(unsigned long long* id) {
  using CtxGetCurrentFn = CUresult (*)(CUcontext*);
  using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static const CtxGetCurrentFn get_current = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return static_cast<CtxGetCurrentFn>(nullptr);
  }();
  static const CtxGetIdFn get_id = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetIdFn>(p);
    return static_cast<CtxGetIdFn>(nullptr);
  }();
  if (!get_current || !get_id) return cuda_fail("cuCtxGetCurrent/cuCtxGetId: driver entry point not found");
  CUcontext ctx = nullptr;
  nf4q_status st = cu_check(get_current(&ctx), "cuCtxGetCurrent");
  if (st != NF4Q_OK) return st;
  *id = 0;
  if (!ctx) return NF4Q_OK;
  return cu_check(get_id(ctx, id), "cuCtxGetId");
}

// One launch of `kernel` on `stream`; `attrs` (may be null) are passed on as
// cudaLaunchKernelEx launch attributes.
template <typename... KArgs, typename... Args>
inline nf4q_status launch(const char* what, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                          size_t smem, cudaStream_t stream, cudaLaunchAttribute* attrs,
                          unsigned n_attrs, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = n_attrs;
  return cuda_check(cudaLaunchKernelEx(&cfg, kernel, args...), what);
}

}  // namespace nf4q
