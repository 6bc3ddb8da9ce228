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
// host-side stand-in, so its device address is looked up with cudaGetSymbolAddress (with the device
// current) on the first call made in a CUDA context, and passed to the kernels from then on. The
// address is kept per context, not per device index: after cudaDeviceReset the next call finds a
// new context and looks the address up again. A lookup that fails is not kept, so the next call
// tries again.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"
#include "context_id.h"

static_assert(ATTN_SPLITKV_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// Partial results (normalized O and LSE per split) of attn_fwd_splitkv_static; shared by all calls.
static __device__ __align__(256) unsigned char g_splitkv_scratch[ATTN_SPLITKV_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct ScratchAddress {
  std::mutex mu;
  unsigned long long ctx = 0;   // context id the address belongs to (0: none yet)
  void* ptr = nullptr;
};
ScratchAddress g_scratch[kMaxDevices];

// Device address of the scratch array in the current context (nullptr if it cannot be found).
void* scratch_in_current_context() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  ScratchAddress& s = g_scratch[dev];
  const unsigned long long id = gb300::current_context_id();
  std::lock_guard<std::mutex> lock(s.mu);
  if (id != 0 && id == s.ctx) return s.ptr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || p == nullptr) return nullptr;
  // The lookup initialises the context if there was none yet: key the address on it.
  s.ctx = gb300::current_context_id();
  s.ptr = p;
  return p;
}

}  // namespace

extern "C" attn_status_t attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                                                 int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                                                 int num_splits, attn_dtype_t dtype, const float* descale_q,
                                                 const float* descale_k, const float* descale_v,
                                                 cudaStream_t stream) {
  // attn_fwd_splitkv runs min(num_splits, ceil(Nk / 128)) splits, so the footprint is that of the
  // splits that run: a large request over few keys still fits.
  if (Nk >= 1 && num_splits >= 1) {
    const int n_kvt = (int)(((long long)Nk + 127) / 128);
    if (num_splits > n_kvt) num_splits = n_kvt;
  }
  const size_t need = attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, num_splits);
  if (need > (size_t)ATTN_SPLITKV_STATIC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;
  void* scratch = scratch_in_current_context();
  if (!scratch) return ATTN_ERR_CUDA;
  // Argument checks (including need == 0 for invalid shapes) happen in attn_fwd_splitkv.
  return attn_fwd_splitkv(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, num_splits, dtype, descale_q, descale_k,
                          descale_v, scratch, (size_t)ATTN_SPLITKV_STATIC_SCRATCH_BYTES, stream);
}
