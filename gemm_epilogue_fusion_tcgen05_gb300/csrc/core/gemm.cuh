// Persistent, warp-specialised tcgen05 GEMM with a pluggable epilogue.
//
//   C[M, N] = A[M, K] * B[K, N]    (bf16 operands, fp32 accumulation in TMEM)
//
// This is the fixed "mainloop" of a GEMM-plus-epilogue program: the epilogue
// class decides what happens to each 128 x BN accumulator tile while it is
// still on chip ("CODA: Rewriting Transformer Blocks as GEMM-Epilogue
// Programs", Fig. 3 caption; "Reading notes on CODA", s1 "The Epilogue
// Concept"). The pages' mainloop is a Hopper PingPong template; on sm_103a
// the same overlap of epilogue and tensor-core work comes from two TMEM
// accumulator buffers: the MMA warp fills buffer b^1 while the epilogue warps
// drain buffer b.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: A and B tiles into a ring of shared-memory stages
//   warp 1      TMEM allocator and MMA issuer (one thread issues tcgen05.mma)
//   warps 2..5  epilogue: TMEM -> registers -> epilogue math -> smem -> TMA store
// Operands may be K-major or MN-major (the tcgen05 transpose bits), both with
// the 128-byte swizzle; out-of-range rows and columns are zero-filled by TMA
// on load and clipped by TMA on store.
#pragma once
#include "ptx.cuh"

namespace coda {

constexpr int kBM = 128;        // tile rows (TMEM lanes)
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kUK = 16;         // K per tcgen05.mma (kind::f16)
constexpr int kSmemMax = 232448;
constexpr int kEpiWarps = 4;
constexpr int kEpiBars = 8;     // mbarriers per epilogue warp (tile loads)

struct GemmArgs {
  int M, N, K;
  int tiles_m, tiles_n, num_tiles, num_kb;
  int group;                      // tiles are ordered in bands of `group` row (or column) blocks
  int along_m;                    // 1: bands of row blocks (row index fastest inside a band)
  int* err;                       // device error word
  unsigned long long timeout_ns;  // bound on every wait
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

template <int BN_, bool A_MN_, bool B_MN_, class Epi_>
struct GemmTraits {
  static constexpr int BN = BN_;
  static constexpr bool A_MN = A_MN_;
  static constexpr bool B_MN = B_MN_;
  using Epi = Epi_;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_BYTES = Epi::kSmemPerWarp * kEpiWarps;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int kFit = (kSmemMax - 1024 - EPI_BYTES - BAR_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = kFit > 6 ? 6 : kFit;
  static_assert(STAGES >= 2, "not enough shared memory for two pipeline stages");
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= kSmemMax, "shared memory budget");
  static constexpr int TMEM_COLS = 2 * BN;
  static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM columns must be a power of two");
  static_assert(BN % 64 == 0 && BN <= 256, "BN");
  static constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN, A_MN, B_MN);
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

template <class T>
__global__ void __launch_bounds__(T::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ typename T::Epi::Params ep, const GemmArgs g) {
  constexpr int S = T::STAGES;
  constexpr int BN = T::BN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + S * T::A_BYTES;
  const uint32_t sEpi = sbase + S * T::STAGE_BYTES;
  uint8_t* barp = smem + S * T::STAGE_BYTES + T::EPI_BYTES;
  const uint32_t bars = smem_u32(barp);
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (S + s); };
  auto tfull = [&](int i) { return bars + 8u * (2 * S + i); };
  auto tempty = [&](int i) { return bars + 8u * (2 * S + 2 + i); };
  const uint32_t epibar = bars + 8u * (2 * S + 4);      // 4 warps x kEpiBars barriers
  const uint32_t drainbar = bars + 8u * (2 * S + 4 + kEpiBars * kEpiWarps);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(barp + 8 * (2 * S + 5 + kEpiBars * kEpiWarps));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull(i), 1);
      mbar_init(tempty(i), kEpiWarps);
    }
    for (int j = 0; j < kEpiBars * kEpiWarps; ++j) mbar_init(epibar + 8u * j, 1);
    mbar_init(drainbar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), T::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const DevError e{g.err, abort_flag, g.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(g, t, mb, nb);
        const int m0 = mb * kBM, n0 = nb * BN;
        for (int kb = 0; kb < g.num_kb; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, e, 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full(stage), T::STAGE_BYTES);
          const uint32_t a_dst = sA + stage * T::A_BYTES;
          const uint32_t b_dst = sB + stage * T::B_BYTES;
          const int k0 = kb * kBK;
          if constexpr (!T::A_MN) {
            tma_load_2d(&tmA, a_dst, full(stage), k0, m0);
          } else {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j) tma_load_2d(&tmA, a_dst + j * 8192, full(stage), m0 + j * 64, k0);
          }
          if constexpr (!T::B_MN) {
            tma_load_2d(&tmB, b_dst, full(stage), k0, n0);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_2d(&tmB, b_dst + j * 8192, full(stage), n0 + j * 64, k0);
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // the MMA warp may never consume what is in flight: wait for it to land
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s)) mbar_drain(full(s), (issued_par >> s) & 1u, 50000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, li = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < g.num_tiles && ok; t += gridDim.x, ++li) {
        const int acc = li & 1;
        if (!mbar_wait(tempty(acc), ((li >> 1) & 1) ^ 1u, e, 2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < g.num_kb; ++kb) {
          if (!mbar_wait(full(stage), phase, e, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_s = sA + stage * T::A_BYTES;
          const uint32_t b_s = sB + stage * T::B_BYTES;
#pragma unroll
          for (int k = 0; k < kBK / kUK; ++k) {
            const uint64_t ad = T::A_MN ? smem_desc_sw128(a_s + k * 2048, 8192, 1024)
                                        : smem_desc_sw128(a_s + k * 32, 16, 1024);
            const uint64_t bd = T::B_MN ? smem_desc_sw128(b_s + k * 2048, 8192, 1024)
                                        : smem_desc_sw128(b_s + k * 32, 16, 1024);
            mma_bf16(d_tmem, ad, bd, T::IDESC, (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit(empty(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull(acc));
      }
      // every MMA issued so far must finish before TMEM is released
      mma_commit(drainbar);
      mbar_drain(drainbar, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    EpiCtx ctx;
    ctx.buf = sEpi + ew * T::Epi::kSmemPerWarp;
    ctx.bar0 = epibar + 8u * kEpiBars * ew;
    ctx.phase = 0;
    ctx.pending = 0;
    ctx.cnt = 0;
    ctx.lane = lane;
    ctx.q = warp & 3;
    ctx.pol = l2_policy_evict_first();
    ctx.e = e;
    int li = 0;
    for (int t = blockIdx.x; t < g.num_tiles; t += gridDim.x, ++li) {
      int mb, nb;
      tile_coords(g, t, mb, nb);
      const int m0 = mb * kBM, n0 = nb * BN;
      const int acc = li & 1;
      T::Epi::template prefetch<BN>(ep, ctx, g, m0, n0);
      bool ok = mbar_wait(tfull(acc), (li >> 1) & 1, e, 4);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * ctx.q) << 16) + acc * BN;
      ok = T::Epi::template tile<BN>(ep, ctx, g, m0, n0, nb, taddr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(acc));
      if (!ok) break;
    }
    if (lane == 0) bulk_wait<0>();
    ctx.drain();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, T::TMEM_COLS);
  }
}

}  // namespace coda
