// Reverse-fused backward GEMM-plus-epilogue kernels. Both multiply an
// activation gradient by a transposed weight: A K-major [M, K], B K-major
// (the weight stored [N, K]). Each has an RMSNorm and a LayerNorm form.
#include "core/launch.cuh"

namespace coda {

template <bool LN, int EW = 4, bool HOIST = false>
static cudaError_t swiglu_bwd_impl(const SwiGLUBwdArgs& a, const LaunchCtx& lc) {
  // with eight epilogue warps, one y load slot per warp (no load ahead of its
  // chunk; the other warp of the lane quarter covers the wait) keeps four
  // pipeline stages
  using E = EpiSwiGLUBwd<LN, EW == 8 ? 1 : 2, HOIST>;
  using T = Gemm2Traits<256, false, false, E, 1, EW>;
  typename E::Params p{};
  p.tm_y = a.tm_y;
  p.tm_dy = a.tm_dy;
  p.r = a.r;
  p.spart = a.spart;
  p.w1 = a.w1;
  p.b1 = a.b1;
  p.spart_w = a.spart_w;
  p.spart_b = a.spart_b;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

cudaError_t launch_swiglu_bwd(const SwiGLUBwdArgs& a, const LaunchCtx& lc) {
  // RMSNorm form: at short K the epilogue outlasts the mainloop, and reading
  // each chunk's y ahead of its stores ran 4 % faster (M = 8192, f = 8192,
  // K = 2048); at K = 4096 the epilogue hides behind the mainloop and the
  // form measured no better
  if (!a.ln) return a.K <= 2048 ? swiglu_bwd_impl<false, 4, true>(a, lc)
                                : swiglu_bwd_impl<false>(a, lc);
  // the LayerNorm form's epilogue (two more n-vectors and two more row
  // partials per chunk) is the one long enough for eight warps
  return pick_epi_warps(a.K, true) == 8 ? swiglu_bwd_impl<true, 8>(a, lc)
                                        : swiglu_bwd_impl<true>(a, lc);
}

template <bool LN, int MS, int EW = 4>
static cudaError_t norm_bwd_impl(const NormBwdArgs& a, const LaunchCtx& lc) {
  using E = EpiNormBwd<LN>;
  using T = Gemm2Traits<256, false, false, E, MS, EW>;
  typename E::Params p{};
  p.h = a.h;
  p.dres = a.dres;
  p.tm_dh = a.tm_dh;
  p.tm_hhat = a.tm_hhat;
  p.gamma = a.gamma;
  p.r = a.r;
  p.s = a.s;
  p.dgpart = a.dgpart;
  p.mu = a.mu;
  p.sa = a.sa;
  p.beta = a.beta;
  p.dbpart = a.dbpart;
  p.save_hhat = a.save_hhat;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

cudaError_t launch_norm_bwd(const NormBwdArgs& a, const LaunchCtx& lc) {
  // K = 2f is long: two-slab tiles where the wave count allows. A two-slab
  // tile fills TMEM with one accumulator, so its epilogue does not overlap
  // the next tile's MMAs; in the RMSNorm form eight epilogue warps (column
  // halves) shorten it and still leave four pipeline stages (2-3 % at
  // M = 16384, d = 4096, K = 28672; 1 % at M = 8192, d = 2048, K = 16384).
  // The one-slab form, whose epilogue overlaps, measured no better with
  // eight; the LayerNorm form's registers do not fit eight.
  if (prefer_two_slabs(a.M, a.N, a.K, 256, lc.num_sms / 2, kEpiKbLoads))
    return a.ln ? norm_bwd_impl<true, 2>(a, lc) : norm_bwd_impl<false, 2, 8>(a, lc);
  return a.ln ? norm_bwd_impl<true, 1>(a, lc) : norm_bwd_impl<false, 1>(a, lc);
}

}  // namespace coda
