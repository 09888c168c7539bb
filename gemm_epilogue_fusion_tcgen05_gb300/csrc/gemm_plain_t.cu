// Plain GEMM instantiations for transposed operands: the data-gradient
// (A K-major, B K-major) and weight-gradient (A MN-major, B MN-major) shapes.
#include "core/launch.cuh"

namespace coda {

template <bool AMN, bool BMN, bool F32, bool R = false, int MS = 1>
static cudaError_t plain_t_impl(const PlainArgs& a, const LaunchCtx& lc) {
  using E = EpiPlain<F32, R, false>;
  using T = Gemm2Traits<256, AMN, BMN, E, MS>;
  typename E::Params p{};
  p.tm_c = a.tmC;
  p.resid = a.resid_ptr;
  p.ld_res = a.ld_res;
  p.rowsq = nullptr;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

cudaError_t launch_plain_other(const PlainArgs& a, const LaunchCtx& lc) {
  if (a.rowsq) return cudaErrorNotSupported;
  if (a.resid) {
    // C (+)= A B^T in fp32: e.g. a gradient accumulated over several launches
    if (!a.a_mn && !a.b_mn && a.out_f32) {
      if (prefer_two_slabs(a.M, a.N, a.K, 256, lc.num_sms / 2))
        return plain_t_impl<false, false, true, true, 2>(a, lc);
      return plain_t_impl<false, false, true, true>(a, lc);
    }
    return cudaErrorNotSupported;
  }
  if (!a.a_mn && !a.b_mn)
    return a.out_f32 ? plain_t_impl<false, false, true>(a, lc) : plain_t_impl<false, false, false>(a, lc);
  if (a.a_mn && a.b_mn) {
    // the weight-gradient shape: K = tokens, usually long
    if (prefer_two_slabs(a.M, a.N, a.K, 256, lc.num_sms / 2))
      return a.out_f32 ? plain_t_impl<true, true, true, false, 2>(a, lc)
                       : plain_t_impl<true, true, false, false, 2>(a, lc);
    return a.out_f32 ? plain_t_impl<true, true, true>(a, lc) : plain_t_impl<true, true, false>(a, lc);
  }
  return a.out_f32 ? plain_t_impl<true, false, true>(a, lc) : plain_t_impl<true, false, false>(a, lc);
}

}  // namespace coda
