// Forward GEMM-plus-epilogue kernels: residual + RMSNorm weight + row
// statistics, delayed row scale + SwiGLU, row scale + RoPE, LM head + CE.
// All take A K-major (activations [M, K]) and B MN-major (weights [K, N]).
#include "core/launch.cuh"

namespace coda {

template <bool LN, int MS>
static cudaError_t resid_norm_stats_impl(const ResidNormStatsArgs& a, const LaunchCtx& lc) {
  using E = EpiResidNormStats<LN>;
  using T = Gemm2Traits<256, false, true, E, MS>;
  typename E::Params p{};
  p.z = a.z;
  p.tm_h = a.tm_h;
  p.tm_hg = a.tm_hg;
  p.gamma = a.gamma;
  p.part = a.part;
  p.part2 = a.part2;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

template <bool LN>
static cudaError_t resid_norm_stats_shape(const ResidNormStatsArgs& a, const LaunchCtx& lc) {
  // long K (e.g. the down projection feeding the next norm): two-slab tiles
  if (prefer_two_slabs(a.M, a.N, a.K, 256, lc.num_sms / 2, kEpiKbLoads))
    return resid_norm_stats_impl<LN, 2>(a, lc);
  return resid_norm_stats_impl<LN, 1>(a, lc);
}

cudaError_t launch_resid_norm_stats(const ResidNormStatsArgs& a, const LaunchCtx& lc) {
  return a.ln ? resid_norm_stats_shape<true>(a, lc) : resid_norm_stats_shape<false>(a, lc);
}

template <bool LN>
static cudaError_t rowscale_swiglu_impl(const RowScaleSwiGLUArgs& a, const LaunchCtx& lc) {
  using E = EpiRowScaleSwiGLU<LN>;
  using T = Gemm2Traits<256, false, true, E>;
  typename E::Params p{};
  p.tm_a = a.tm_a;
  p.tm_y = a.tm_y;
  p.r = a.r;
  p.save_y = a.save_y;
  p.mu = a.mu;
  p.w1 = a.w1;
  p.b1 = a.b1;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

cudaError_t launch_rowscale_swiglu(const RowScaleSwiGLUArgs& a, const LaunchCtx& lc) {
  return a.ln ? rowscale_swiglu_impl<true>(a, lc) : rowscale_swiglu_impl<false>(a, lc);
}

cudaError_t launch_rope(const RopeArgs& a, const LaunchCtx& lc) {
  using E = EpiRope;
  using T = Gemm2Traits<256, false, true, E>;
  E::Params p{};
  p.tm_out = a.tm_out;
  p.tm_save = a.tm_save;
  p.save = a.save;
  p.r = a.r;
  p.cs = a.cs;
  p.seq_len = a.seq_len;
  p.head_dim = a.head_dim;
  p.n_rope = a.n_rope;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

cudaError_t launch_ce(const CEArgs& a, const LaunchCtx& lc) {
  using E = EpiCE;
  using T = Gemm2Traits<256, false, true, E>;
  E::Params p{};
  p.targets = a.targets;
  p.part = a.part;
  p.tlogit = a.tlogit;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

cudaError_t launch_ce_grad(const CEGradArgs& a, const LaunchCtx& lc) {
  using E = EpiCEGrad;
  using T = Gemm2Traits<256, false, true, E>;
  E::Params p{};
  p.tm_g = a.tm_g;
  p.targets = a.targets;
  p.lse = a.lse;
  p.dloss = a.dloss;
  p.v0 = a.v0;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

}  // namespace coda
