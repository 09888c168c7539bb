// Host-side launcher for the persistent tcgen05 GEMM: grid = min(tiles, SMs),
// one CTA per SM, tile order chosen so the larger operand streams from HBM
// once while the smaller one stays resident in L2.
#pragma once
#include <atomic>
#include "../internal.h"
#include "epilogues.cuh"

namespace coda {

template <class T>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const typename T::Epi::Params& ep, int M, int N, int K, const LaunchCtx& lc) {
  static std::atomic<unsigned long long> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_acq_rel);
  }
  GemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.tiles_m = (M + kBM - 1) / kBM;
  g.tiles_n = (N + T::BN - 1) / T::BN;
  g.num_tiles = g.tiles_m * g.tiles_n;
  g.num_kb = (K + kBK - 1) / kBK;
  // B much larger than A (e.g. an LM head): walk all row blocks of one column
  // block before the next, so each B panel is read from HBM once.
  g.n_fast = M > N ? 1 : 0;
  g.err = lc.err;
  g.timeout_ns = lc.timeout_ns;
  const int grid = g.num_tiles < lc.num_sms ? g.num_tiles : lc.num_sms;
  gemm_kernel<T><<<grid, T::kThreads, T::SMEM_BYTES, lc.stream>>>(tmA, tmB, ep, g);
  return cudaGetLastError();
}

}  // namespace coda
