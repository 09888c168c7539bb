// Pieces shared by the tcgen05 GEMM-plus-epilogue kernels (gemm2.cuh): tile
// and pipeline constants, the launch arguments, the epilogue warps' context
// and the tile order.
//
//   C[M, N] = A[M, K] * B[K, N]    (bf16 operands, fp32 accumulation in TMEM)
//
// The mainloop is fixed; an epilogue class decides what happens to each
// accumulator tile while it is still on chip ("CODA: Rewriting Transformer
// Blocks as GEMM-Epilogue Programs", Fig. 3 caption; "Reading notes on
// CODA", s1 "The Epilogue Concept"). Operands may be K-major or MN-major
// (the tcgen05 transpose bits), both with the 128-byte swizzle; out-of-range
// rows and columns are zero-filled by TMA on load and clipped by TMA on store.
#pragma once
#include "ptx.cuh"

namespace coda {

constexpr int kBM = 128;        // tile rows (TMEM lanes)
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kUK = 16;         // K per tcgen05.mma (kind::f16)
constexpr int kSmemMax = 232448;
constexpr int kEpiBars = 8;     // mbarriers per epilogue warp (tile loads)
// Row partials (sums over a row's columns, e.g. of h^2) are written per
// kPartCols columns, whatever the tile width: the partial buffers of the C
// ABI are [ceil(N / kPartCols), M].
constexpr int kPartCols = 128;

struct GemmArgs {
  int M, N, K;
  int tiles_m, tiles_n, num_tiles, num_kb;
  int group;                      // tiles are ordered in bands of `group` row (or column) blocks
  int along_m;                    // 1: bands of row blocks (row index fastest inside a band)
  int* err;                       // device error word
  unsigned long long timeout_ns;  // bound on every wait
  int skip_kb;                    // failure-detection tests only (normally -1): the
                                  // producers do not load this k-block of their
                                  // first tile, so the waits for it run out
};

// Per-epilogue-warp context: staging buffers, the warp's mbarriers for
// epilogue tile loads, their phase bits, and a running chunk counter.
struct EpiCtx {
  uint32_t buf;      // shared address of this warp's staging area
  uint32_t bar0;     // first of this warp's kEpiBars mbarriers (8 bytes apart)
  uint32_t phase;    // parity bit per barrier
  uint32_t pending;  // barriers with a load issued and not yet waited on
  uint32_t cnt;      // chunks processed so far (selects the staging set)
  int lane, q;       // lane; TMEM lane quarter = row block of 32 inside the tile
  uint64_t pol;      // L2 policy for data touched once (epilogue tile loads and stores)
  DevError e;

  __device__ __forceinline__ uint32_t bar(int j) const { return bar0 + 8u * j; }
  // issue (lane 0): expect `bytes` on barrier j and load box (x, y) into dst
  __device__ __forceinline__ void load(const CUtensorMap* m, int j, uint32_t dst, int x, int y,
                                       uint32_t bytes) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(j), bytes);
      tma_load_2d_hint(m, dst, bar(j), x, y, pol);
    }
    pending |= 1u << j;
  }
  // wait (all lanes) for the load on barrier j; warp-uniform result
  __device__ __forceinline__ bool wait(int j, int where) {
    bool ok = mbar_wait(bar(j), (phase >> j) & 1u, e, where);
    ok = __all_sync(0xffffffffu, ok);
    phase ^= 1u << j;
    pending &= ~(1u << j);
    return ok;
  }
  __device__ __forceinline__ void drain() {
    for (int j = 0; j < kEpiBars; ++j)
      if (pending & (1u << j)) mbar_drain(bar(j), (phase >> j) & 1u, 50000000ull);
    pending = 0;
  }
  // store one staged box (lane 0 issues)
  __device__ __forceinline__ void store(const CUtensorMap* m, uint32_t src, int x, int y) {
    tma_store_2d_hint(m, src, x, y, pol);
  }
  // lane 0 makes sure every earlier TMA store has finished reading its smem
  __device__ __forceinline__ void stores_read_done() {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }
  // ... every earlier store except the most recent group (the previous
  // chunk's): enough before reusing a staging set two chunks later
  __device__ __forceinline__ void stores_read_but_last() {
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
  }
};

// Grouped tile order. With along_m, the tiles form bands of `group` row
// blocks; inside a band the row block varies fastest, then the column block.
// The concurrently running tiles then share a few operand panels: the
// band's A panels stay in L2 while B panels stream past, each read from HBM
// once per band. (along_m = 0 is the same with rows and columns swapped.)
__device__ __forceinline__ void tile_coords(const GemmArgs& g, int t, int& mb, int& nb) {
  if (g.along_m) {
    const int per = g.group * g.tiles_n;
    const int band = t / per, r = t - band * per;
    const int m0 = band * g.group;
    const int gs = min(g.group, g.tiles_m - m0);
    mb = m0 + r % gs;
    nb = r / gs;
  } else {
    const int per = g.group * g.tiles_m;
    const int band = t / per, r = t - band * per;
    const int n0 = band * g.group;
    const int gs = min(g.group, g.tiles_n - n0);
    nb = n0 + r % gs;
    mb = r / gs;
  }
}

}  // namespace coda
