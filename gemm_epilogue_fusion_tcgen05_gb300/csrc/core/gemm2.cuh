// Persistent tcgen05 GEMM on CTA pairs (cta_group::2): each cluster of two
// CTAs on neighbouring SMs computes a 256 x BN tile with one
// tcgen05.mma.cta_group::2 (M = 256) per K step, issued by the even CTA.
// Each CTA stages its own 128 rows of A and half (BN/2 columns) of B, so per
// SM the shared-memory traffic per MMA and the operand bytes fetched from L2
// are half those of a single-CTA 128 x BN tile; TMEM of each CTA holds its
// 128 accumulator rows; every CTA's epilogue warps drain their own
// 128 x BN slice. Two TMEM accumulator buffers let the MMA warp fill buffer
// b^1 while the epilogue warps drain buffer b (the sm_103a counterpart of the
// pages' Hopper PingPong overlap). BN is 256 or 128: the narrower tile gives
// twice the tiles, for outputs whose 256-wide tiles fill the SMs in too few
// waves.
//
// Warp roles (64 + 32 EW threads, one CTA per SM):
//   warp 0      TMA producer: this CTA's A rows and B half into a ring of stages
//   warp 1      TMEM allocator; in the even CTA, the single thread issuing tcgen05.mma
//   warps 2..   EW epilogue warps: TMEM -> registers -> epilogue math -> smem ->
//               TMA store. A warp may read only its own 32-lane TMEM quarter
//               (warp index mod 4), so with EW = 4 each warp drains 32 rows x
//               BN columns; with EW = 8 two warps share a quarter and each
//               takes one 128-column half: twice the warps to hide the
//               latency of an epilogue whose instruction stream outlasts a
//               short-K mainloop.
//
// Synchronisation across the pair:
//   full[s]   (even CTA)  both CTAs' TMA loads complete_tx here; the even
//                          CTA's producer arms it with both CTAs' bytes
//   empty[s]  (both)      MMA commit multicast to both CTAs frees stage s
//   tfull[b]  (both)      MMA commit multicast: accumulator b is ready
//   tempty[b] (even CTA)  2 EW arrivals (every epilogue warp of both CTAs)
//   drain     (both)      last MMA commit: nothing reads shared memory or
//                          TMEM any more, so both CTAs may leave
//
// Two-slab form (MS = 2): each CTA holds 2 x 128 rows of A and the pair
// computes a 512 x BN tile with two MMAs per K step that share the B half, so
// every byte of B staged in shared memory feeds twice the tensor-core work
// and the operand bytes per FLOP drop by a quarter; the same bytes in flight
// then cover a third more MMA time. Both slabs' accumulators fill TMEM, so
// there is one accumulator buffer and the epilogue does not overlap the next
// tile's MMA: the form pays off for long K, where the epilogue is rare.
#pragma once
#include "gemm.cuh"

namespace coda {

template <int BN_, bool A_MN_, bool B_MN_, class Epi_, int MS_ = 1, int EW_ = 4>
struct Gemm2Traits {
  static constexpr int BN = BN_;
  static constexpr bool A_MN = A_MN_;
  static constexpr bool B_MN = B_MN_;
  using Epi = Epi_;
  static constexpr int MS = MS_;                          // 128-row slabs of A per CTA
  static constexpr int NACC = MS == 1 ? 2 : 1;            // accumulator buffers in TMEM
  static_assert(MS == 1 || MS == 2, "MS");
  static constexpr int EW = EW_;                          // epilogue warps
  static_assert(EW == 4 || EW == 8, "EW");
  static constexpr int ECOLS = BN / (EW / 4);             // columns per epilogue warp
  static_assert(ECOLS % kPartCols == 0, "an epilogue warp covers whole row-partial groups");
  static constexpr int kThreads = 64 + 32 * EW;
  static constexpr int SLAB_BYTES = kBM * kBK * 2;        // one 128-row slab of A
  static constexpr int A_BYTES = MS * SLAB_BYTES;         // this CTA's 128 * MS rows
  static constexpr int B_BYTES = (BN / 2) * kBK * 2;     // this CTA's half of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_BYTES = Epi::kSmemPerWarp * EW;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int kFit = (kSmemMax - 1024 - EPI_BYTES - BAR_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = kFit > 8 ? 8 : kFit;
  static_assert(STAGES >= 3, "not enough shared memory for three pipeline stages");
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= kSmemMax, "shared memory budget");
  static constexpr int TMEM_COLS = NACC * MS * BN;
  static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM columns must be a power of two");
  static_assert(BN % 128 == 0 && BN <= 256, "BN");
  static constexpr uint32_t IDESC = idesc_bf16_f32(2 * kBM, BN, A_MN, B_MN);
};

template <class T>
__global__ void __launch_bounds__(T::kThreads, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
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
  const uint32_t epibar = bars + 8u * (2 * S + 4);      // EW warps x kEpiBars barriers
  const uint32_t drainbar = bars + 8u * (2 * S + 4 + kEpiBars * T::EW);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(barp + 8 * (2 * S + 5 + kEpiBars * T::EW));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = issues the pair's MMA, 1 = peer
  const bool leader = rank == 0;
  const uint32_t lead = 0;                   // the pair's even CTA
  const uint16_t pair_mask = 3u;
  const int pair = blockIdx.x / 2;           // cluster index: one tile at a time
  const int npairs = gridDim.x / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);  // the pair's MMA commit frees the stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull(i), 1);
      mbar_init(tempty(i), 2 * T::EW);
    }
    for (int j = 0; j < kEpiBars * T::EW; ++j) mbar_init(epibar + 8u * j, 1);
    mbar_init(drainbar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), T::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const DevError e{g.err, abort_flag, g.timeout_ns};
  // everything above (barriers, TMEM, descriptor prefetch) may overlap the
  // previous kernel's drain; no global memory is touched before this wait.
  // All of this grid's CTAs are resident (grid <= co-resident clusters), so
  // the next kernel's CTAs, once released, only take SMs ours have left.
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      const uint64_t pol_keep = l2_policy_evict_last();
      for (int t = pair; t < g.num_tiles && ok; t += npairs) {
        int mb, nb;
        tile_coords(g, t, mb, nb);
        const int m0 = (mb * 2 + (int)rank) * T::MS * kBM;
        const int n0 = nb * BN + (int)rank * (BN / 2);
        for (int kb = 0; kb < g.num_kb; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, e, 21)) {
            ok = false;
            break;
          }
          if (kb == g.skip_kb && t == pair) {
            // test hook: leave this stage unarmed and unloaded; the MMA
            // issuer's wait for it, and every wait behind that, runs out
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (leader) mbar_arrive_expect_tx(full(stage), 2 * T::STAGE_BYTES);
          const uint32_t fb = mapa_shared(full(stage), lead);
          const uint32_t a_dst = sA + stage * T::A_BYTES;
          const uint32_t b_dst = sB + stage * T::B_BYTES;
          const int k0 = kb * kBK;
          // the band's stationary operand stays in L2 (evict_last); the
          // other streams past with the default policy
#pragma unroll
          for (int i = 0; i < T::MS; ++i) {
            const uint32_t ad = a_dst + i * T::SLAB_BYTES;
            const int mi = m0 + i * kBM;
            if constexpr (!T::A_MN) {
              if (g.along_m) tma_load_2d_pair_hint(&tmA, ad, fb, k0, mi, pol_keep);
              else tma_load_2d_pair(&tmA, ad, fb, k0, mi);
            } else {
#pragma unroll
              for (int j = 0; j < kBM / 64; ++j) {
                if (g.along_m) tma_load_2d_pair_hint(&tmA, ad + j * 8192, fb, mi + j * 64, k0, pol_keep);
                else tma_load_2d_pair(&tmA, ad + j * 8192, fb, mi + j * 64, k0);
              }
            }
          }
          if constexpr (!T::B_MN) {
            // 64-row boxes (the map does not depend on the tile width); two
            // stacked boxes have the layout of one 128-row box
#pragma unroll
            for (int j = 0; j < BN / 128; ++j) {
              if (!g.along_m) tma_load_2d_pair_hint(&tmB, b_dst + j * 8192, fb, k0, n0 + j * 64, pol_keep);
              else tma_load_2d_pair(&tmB, b_dst + j * 8192, fb, k0, n0 + j * 64);
            }
          } else {
#pragma unroll
            for (int j = 0; j < BN / 128; ++j) {
              if (!g.along_m) tma_load_2d_pair_hint(&tmB, b_dst + j * 8192, fb, n0 + j * 64, k0, pol_keep);
              else tma_load_2d_pair(&tmB, b_dst + j * 8192, fb, n0 + j * 64, k0);
            }
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s)) mbar_drain(full(s), (issued_par >> s) & 1u, 50000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0) {
      if (leader) {
        int stage = 0, li = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = pair; t < g.num_tiles && ok; t += npairs, ++li) {
          const int acc = li % T::NACC;
          if (!mbar_wait_cluster(tempty(acc), ((li / T::NACC) & 1) ^ 1u, e, 22)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * T::MS * BN;
          for (int kb = 0; kb < g.num_kb; ++kb) {
            if (!mbar_wait_cluster(full(stage), phase, e, 23)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_s = sA + stage * T::A_BYTES;
            const uint32_t b_s = sB + stage * T::B_BYTES;
#pragma unroll
            for (int k = 0; k < kBK / kUK; ++k) {
              const uint64_t bd = T::B_MN ? smem_desc_sw128(b_s + k * 2048, 8192, 1024)
                                          : smem_desc_sw128(b_s + k * 32, 16, 1024);
#pragma unroll
              for (int i = 0; i < T::MS; ++i) {
                const uint32_t as = a_s + i * T::SLAB_BYTES;
                const uint64_t ad = T::A_MN ? smem_desc_sw128(as + k * 2048, 8192, 1024)
                                            : smem_desc_sw128(as + k * 32, 16, 1024);
                mma_bf16_pair(d_tmem + i * BN, ad, bd, T::IDESC, (kb | k) != 0 ? 1u : 0u);
              }
            }
            // the stage is free for both CTAs' producers once these MMAs
            // have read it
            mma_commit_pair(empty(stage), pair_mask);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_pair(tfull(acc), pair_mask);
        }
        // both CTAs learn when every MMA (which reads both CTAs' smem and
        // writes both CTAs' TMEM) has finished
        mma_commit_pair(drainbar, pair_mask);
        mbar_drain(drainbar, 0, 200000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    constexpr int EC = T::ECOLS;
    const int ew = warp - 2;
    const int cpart = ew >> 2;  // column part of the tile (EW = 8: two 128-column halves)
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
    for (int t = pair; t < g.num_tiles; t += npairs, ++li) {
      int mb, nb;
      tile_coords(g, t, mb, nb);
      const int m_cta = (mb * 2 + (int)rank) * T::MS * kBM;
      const int n_w = nb * BN + cpart * EC;  // this warp's first column
      const bool live = n_w < g.N;           // a part wholly past N has nothing to do
      const int acc = li % T::NACC;
      if (live) T::Epi::template prefetch<EC>(ep, ctx, g, m_cta, n_w);
      bool ok = mbar_wait_cluster(tfull(acc), (li / T::NACC) & 1, e, 24);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int i = 0; i < T::MS && ok && live; ++i) {
        const int m0 = m_cta + i * kBM;
        if (i > 0) T::Epi::template prefetch<EC>(ep, ctx, g, m0, n_w);
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * ctx.q) << 16) +
                               (acc * T::MS + i) * BN + cpart * EC;
        ok = T::Epi::template tile<EC>(ep, ctx, g, m0, n_w, nb, taddr);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty(acc), lead));
      if (!ok) break;
    }
    if (lane == 0) bulk_wait<0>();
    ctx.drain();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // copies issued before giving up may still be landing: let them finish
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) {
    }
  }
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, T::TMEM_COLS);
  }
}

}  // namespace coda
