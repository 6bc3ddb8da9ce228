// attn_fwd_splitkv_static: split-KV decode for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc, or must not: a plugin running inside a framework
// that owns all device memory through its own pool, a server working under a fixed memory budget
// it has already committed, or a latency-critical path where an allocation (which may synchronize
// the device) is not acceptable. attn_fwd_splitkv needs a workspace for its partial results; this
// variant keeps that workspace in a fixed device array that is part of the library instead.
//
// The array is file-scope device memory of ATTN_SPLITKV_STATIC_SCRATCH_BYTES (16 MiB). Every GPU
// that loads the library holds it until the process exits. In host code the array's name is only a
// host-side stand-in, so its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) on the first call made on that device, and
// passed to the kernels from then on.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"

static_assert(ATTN_SPLITKV_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// Partial results (normalized O and LSE per split) of attn_fwd_splitkv_static; shared by all calls.
static __device__ __align__(256) unsigned char g_splitkv_scratch[ATTN_SPLITKV_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct ScratchAddress {
  std::once_flag once;
  void* ptr = nullptr;
};
ScratchAddress g_scratch[kMaxDevices];

// Device address of the scratch array on the current device (nullptr if it cannot be found).
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  ScratchAddress& s = g_scratch[dev];
  std::call_once(s.once, [&s] {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitkv_scratch) == cudaSuccess) s.ptr = p;
  });
  return s.ptr;
}

}  // namespace

extern "C" attn_status_t attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                                                 int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                                                 int num_splits, attn_dtype_t dtype, const float* descale_q,
                                                 const float* descale_k, const float* descale_v,
                                                 cudaStream_t stream) {
  const size_t need = attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, num_splits);
  if (need > (size_t)ATTN_SPLITKV_STATIC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;
  void* scratch = scratch_on_current_device();
  if (!scratch) return ATTN_ERR_CUDA;
  // Argument checks (including need == 0 for invalid shapes) happen in attn_fwd_splitkv.
  return attn_fwd_splitkv(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, num_splits, dtype, descale_q, descale_k,
                          descale_v, scratch, (size_t)ATTN_SPLITKV_STATIC_SCRATCH_BYTES, stream);
}
