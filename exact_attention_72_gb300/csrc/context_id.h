// Identity of the CUDA context current on the calling thread.
//
// Device addresses of the library's file-scope device variables, and the streams and events it
// keeps, belong to one context. After cudaDeviceReset the runtime builds a new primary context on
// the same device and loads the library's module again, so anything cached for the old context
// must be looked up again: a cached address would point into memory this process no longer owns.
// Caches in this library are therefore keyed on the context's unique id (cuCtxGetId), not on the
// device index. The driver entry points are looked up through the runtime, as for the tensor-map
// encoder, so the library needs no link-time dependency on the driver library.
#pragma once
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300 {

// Unique id of the current context, or 0 when there is none yet or it cannot be read.
inline unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace gb300
