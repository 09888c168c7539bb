// Host-side launcher for the persistent tcgen05 GEMM: grid = min(tiles, SMs),
// one CTA per SM, tile order chosen so the larger operand streams from HBM
// once while the smaller one stays resident in L2.
#pragma once
#include <atomic>
#include <cmath>
#include "../internal.h"
#include "epilogues.cuh"
#include "gemm2.cuh"

namespace coda {

// Tile order for an M x N x K GEMM with bm x bn tiles and `conc` tiles in
// flight at a time. Tiles go in bands of `group` row blocks (or column
// blocks); the estimate of HBM traffic for a band size G is:
//   * if the band's stationary panels (G of them) fit an L2 budget, they
//     are read once and the moving operand's panels stream once per band;
//   * otherwise nothing survives from one wave of `conc` tiles to the next,
//     and each wave reads the distinct panels it touches.
// The direction and G with the smallest estimate win. Small operands that
// fit the budget whole simply stay resident (G = all blocks).
inline void choose_tile_order(GemmArgs& g, int bm, int bn, int K, int conc) {
  const double budget = 48.0 * 1024 * 1024;
  const double pa = 2.0 * bm * K, pb = 2.0 * bn * K;  // bytes of one row / column panel
  double best = -1.0;
  for (int dir = 0; dir < 2; ++dir) {
    const int ts = dir == 0 ? g.tiles_m : g.tiles_n;  // blocks of the stationary operand
    const int to = dir == 0 ? g.tiles_n : g.tiles_m;  // blocks of the moving operand
    const double ps = dir == 0 ? pa : pb, po = dir == 0 ? pb : pa;
    for (int G = 1; G <= ts; ++G) {
      const int bands = (ts + G - 1) / G;
      double band_cost;
      if (G * ps <= budget) {
        band_cost = G * ps + to * po;
      } else {
        const double waves = std::ceil((double)G * to / conc);
        const double gs = G < conc ? G : conc;
        const double os = std::ceil((double)conc / G) < to ? std::ceil((double)conc / G) : to;
        band_cost = waves * (gs * ps + os * po);
      }
      const double cost = bands * band_cost;
      if (best < 0 || cost < best * 0.999) {
        best = cost;
        g.along_m = dir == 0 ? 1 : 0;
        g.group = G;
      }
    }
  }
}

// Whether the two-slab pair tile (512 x bn, see gemm2.cuh) should beat the
// one-slab tile (256 x bn) on an M x N x K GEMM with `pairs` co-resident CTA
// pairs. Two slabs move a quarter fewer operand bytes per FLOP (measured
// 1.25x the throughput on weight-gradient shapes with K = 16384 at equal wave
// counts), but they halve the tile count (coarser waves) and the epilogue no
// longer overlaps the next tile's MMA (about `epi_kb` K-blocks of MMA time
// per tile for a 256 x 256 fp32 output per CTA). Estimated time in units of
// one 256-row tile's mainloop of K:
//   one slab   ceil(T1 / P)
//   two slabs  ceil(T2 / P) * (2 * kTwoSlabCost + epi_kb / kblocks)
// Two slabs are taken only when the estimate is at least 3 % lower (at
// K = 8192 with 7 one-slab waves against 4 two-slab waves they measured even).
constexpr int kTwoSlabMinK = 8192;
constexpr double kTwoSlabCost = 0.80;
constexpr double kEpiKbLoads = 24.0;  // epilogues that also read tiles (residual, h)
constexpr int kTwoSlabMinKLoads = 12288;  // ... which measured no gain at K = 8192
inline bool prefer_two_slabs(int M, int N, int K, int bn, int pairs, double epi_kb = 16.0) {
  if (K < (epi_kb > 16.0 ? kTwoSlabMinKLoads : kTwoSlabMinK) || pairs <= 0) return false;
  const double tn = (double)((N + bn - 1) / bn);
  const double t1 = (double)((M + 255) / 256) * tn, t2 = (double)((M + 511) / 512) * tn;
  const double w1 = std::ceil(t1 / pairs), w2 = std::ceil(t2 / pairs);
  const double kblocks = (double)((K + kBK - 1) / kBK);
  return w2 * (2.0 * kTwoSlabCost + epi_kb / kblocks) < 0.97 * w1;
}

// Epilogue warps of a one-slab launch: four (one per TMEM lane quarter, each
// on the whole 256-column tile) or eight (two per quarter, each on one
// 128-column half). Eight hide more of an epilogue's latency but leave fewer
// pipeline stages (their staging comes out of the same shared memory). They
// paid off only where the epilogue is much longer than a short-K mainloop:
// the LayerNorm form of the SwiGLU backward at K = 2048 (0.226 against
// 0.265 ms at M = 8192, f = 8192); the RMSNorm forms and the plain GEMMs ran
// 1-3 % slower with eight, and the RMSNorm SwiGLU backward at K = 4096 20 %
// slower.
inline int pick_epi_warps(int K, bool heavy) { return heavy && K <= 2048 ? 8 : 4; }

// Launch of the CTA-pair kernel: clusters of 2, grid = 2 x min(tiles,
// co-resident pairs).
template <class T>
cudaError_t launch_gemm2(const CUtensorMap& tmA, const CUtensorMap& tmB,
                         const typename T::Epi::Params& ep, int M, int N, int K, const LaunchCtx& lc) {
  static std::atomic<int> max_pairs[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  dev &= 63;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the kernel's prologue may overlap the
  // previous kernel's drain (the kernel waits in grid_dep_wait())
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(T::kThreads, 1, 1);
  cfg.dynamicSmemBytes = T::SMEM_BYTES;
  cfg.stream = lc.stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
  int pairs_max = max_pairs[dev].load(std::memory_order_acquire);
  if (pairs_max <= 0) {
    e = cudaFuncSetAttribute(gemm2_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2, 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm2_kernel<T>, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    pairs_max = n;
    max_pairs[dev].store(n, std::memory_order_release);
  }
  GemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  constexpr int kPairRows = 2 * T::MS * kBM;
  g.tiles_m = (M + kPairRows - 1) / kPairRows;
  g.tiles_n = (N + T::BN - 1) / T::BN;
  g.num_tiles = g.tiles_m * g.tiles_n;
  g.num_kb = (K + kBK - 1) / kBK;
  const int pairs = g.num_tiles < pairs_max ? g.num_tiles : pairs_max;  // clusters
  choose_tile_order(g, kPairRows, T::BN, K, pairs);
  g.err = lc.err;
  g.timeout_ns = lc.timeout_ns;
  g.skip_kb = lc.skip_kb;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, gemm2_kernel<T>, tmA, tmB, ep, g);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace coda
