// Launchers of the backward pass: preprocess (D, -LSE log2 e), then dK/dV, then dQ, all on one stream.
#include <algorithm>

#include "launch.h"

namespace gb300 {
namespace {

template <class K>
cudaError_t launch_persistent(K kernel, int smem, int threads, const BwdLaunchArgs& a, BwdParams p,
                              cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.n_tiles, a.num_sms);
  kernel<<<grid, threads, smem, s>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, p);
  return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd(BwdLaunchArgs& a, cudaStream_t s) {
  using C = BwdCfg<D, CAUSAL>;
  const BwdParams& p = a.params;
  const long long rows = (long long)p.B * p.H * p.Np;
  attn_bwd_preprocess_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.nlse2, a.dd, p.B,
      p.H, p.N, p.Np);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  BwdParams p1 = p;
  p1.n_tiles = p.n_t * p.B * p.Hkv;
  if ((e = launch_persistent(attn_bwd_dkdv_kernel<C>, C::SMEM_BYTES, C::THREADS, a, p1, s)) != cudaSuccess) return e;
  BwdParams p2 = p;
  p2.n_tiles = p.n_t * p.B * p.H;
  return launch_persistent(attn_bwd_dq_kernel<C>, C::DQ_SMEM_BYTES, C::THREADS, a, p2, s);
}

}  // namespace

cudaError_t launch_attn_bwd(BwdLaunchArgs& a, int d, bool causal, cudaStream_t stream) {
  switch (d) {
    case 64: return causal ? launch_bwd<64, true>(a, stream) : launch_bwd<64, false>(a, stream);
    case 128: return causal ? launch_bwd<128, true>(a, stream) : launch_bwd<128, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gb300
