// Host-only check of the GEMM form choices in core/launch.cuh: for each shape
// given on the command line as "M N K loads" (loads = 1 for epilogues that
// read tiles, which charge a larger epilogue term), prints one JSON line with
// the two-slab decision on 76 CTA pairs (152 SMs). Also prints the epilogue
// warp choice for K = 2048 and K = 4096. No GPU is touched.
#include <cstdio>
#include <cstdlib>

#include "core/launch.cuh"

int main(int argc, char** argv) {
  const int pairs = 76;
  for (int i = 1; i + 3 < argc; i += 4) {
    const int M = std::atoi(argv[i]), N = std::atoi(argv[i + 1]), K = std::atoi(argv[i + 2]);
    const bool loads = std::atoi(argv[i + 3]) != 0;
    const bool two = loads ? coda::prefer_two_slabs(M, N, K, 256, pairs, coda::kEpiKbLoads)
                           : coda::prefer_two_slabs(M, N, K, 256, pairs);
    std::printf("{\"M\": %d, \"N\": %d, \"K\": %d, \"loads\": %d, \"two_slabs\": %d}\n", M, N, K,
                loads ? 1 : 0, two ? 1 : 0);
  }
  std::printf("{\"warps_heavy_k2048\": %d, \"warps_heavy_k4096\": %d, \"warps_light_k2048\": %d}\n",
              coda::pick_epi_warps(2048, true), coda::pick_epi_warps(4096, true),
              coda::pick_epi_warps(2048, false));
  return 0;
}
