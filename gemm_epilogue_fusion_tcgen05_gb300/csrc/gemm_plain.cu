// Plain GEMM instantiations: C = op(A) op(B) (+ residual, + row sums of
// squares), bf16 or fp32 output, every operand majorness.
#include "core/launch.cuh"

namespace coda {

template <bool AMN, bool BMN, bool F32, bool R, bool Q, int MS = 1>
static cudaError_t plain_impl(const PlainArgs& a, const LaunchCtx& lc) {
  using E = EpiPlain<F32, R, Q>;
  using T = Gemm2Traits<256, AMN, BMN, E, MS>;
  typename E::Params p{};
  p.tm_c = a.tmC;
  p.resid = a.resid_ptr;
  p.ld_res = a.ld_res;
  p.rowsq = a.rowsq_part;
  return launch_gemm2<T>(a.tmA, a.tmB, p, a.M, a.N, a.K, lc);
}

cudaError_t launch_plain_other(const PlainArgs& a, const LaunchCtx& lc);

cudaError_t launch_plain(const PlainArgs& a, const LaunchCtx& lc) {
  if (!a.a_mn && a.b_mn) {
    const bool two = prefer_two_slabs(a.M, a.N, a.K, 256, lc.num_sms / 2);
    if (a.out_f32) {
      if (a.resid) return plain_impl<false, true, true, true, false>(a, lc);
      return two ? plain_impl<false, true, true, false, false, 2>(a, lc)
                 : plain_impl<false, true, true, false, false>(a, lc);
    }
    if (a.resid && a.rowsq) return plain_impl<false, true, false, true, true>(a, lc);
    if (a.resid) return plain_impl<false, true, false, true, false>(a, lc);
    if (a.rowsq) return plain_impl<false, true, false, false, true>(a, lc);
    return two ? plain_impl<false, true, false, false, false, 2>(a, lc)
               : plain_impl<false, true, false, false, false>(a, lc);
  }
  return launch_plain_other(a, lc);
}

}  // namespace coda
