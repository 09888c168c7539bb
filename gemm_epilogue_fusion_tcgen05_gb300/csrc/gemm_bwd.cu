// Reverse-fused backward GEMM-plus-epilogue kernels. Both multiply an
// activation gradient by a transposed weight: A K-major [M, K], B K-major
// (the weight stored [N, K]).
#include "core/launch.cuh"

namespace coda {

cudaError_t launch_swiglu_bwd(const SwiGLUBwdArgs& a, const LaunchCtx& lc) {
  using E = EpiSwiGLUBwd;
  using T = Gemm2Traits<kTileN, false, false, E>;
  E::Params p;
  p.tm_y = a.tm_y;
  p.tm_dy = a.tm_dy;
  p.r = a.r;
  p.spart = a.spart;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

cudaError_t launch_norm_bwd(const NormBwdArgs& a, const LaunchCtx& lc) {
  using E = EpiNormBwd;
  using T = Gemm2Traits<kTileN, false, false, E>;
  E::Params p;
  p.tm_h = a.tm_h;
  p.tm_dres = a.tm_dres;
  p.tm_dh = a.tm_dh;
  p.gamma = a.gamma;
  p.r = a.r;
  p.s = a.s;
  p.dgpart = a.dgpart;
  p.has_dres = a.has_dres;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

}  // namespace coda
