// Internal declarations shared by the translation units of libcoda.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "core/ptx.cuh"

namespace coda {

using bf16 = __nv_bfloat16;

// Launch context passed from the C-ABI layer to the GEMM launchers.
struct LaunchCtx {
  cudaStream_t stream;
  int* err;                        // device error word
  unsigned long long timeout_ns;   // bound on every wait
  int num_sms;
  int skip_kb;                     // coda_debug_skip_kblock (normally -1)
};

// Plain GEMM: C = op(A) op(B) (+ resid), optional per-row sum of squares.
struct PlainArgs {
  CUtensorMap tmA, tmB, tmC;
  bool a_mn, b_mn, out_f32, resid, rowsq;
  const void* resid_ptr;   // [M, N] with the output's type (read by the epilogue without TMA)
  size_t ld_res;           // its row stride in bytes
  float* rowsq_part;
  int M, N, K;
};
cudaError_t launch_plain(const PlainArgs& a, const LaunchCtx& lc);

struct ResidNormStatsArgs {
  CUtensorMap tmA, tmB, tm_h, tm_hg;
  const bf16* z;   // [M, N] residual (read by the epilogue without TMA)
  const bf16* gamma;
  float* part;
  int M, N, K;
  int ln;        // LayerNorm variant: also per-tile sums of h into part2
  float* part2;
};
cudaError_t launch_resid_norm_stats(const ResidNormStatsArgs& a, const LaunchCtx& lc);

struct RowScaleSwiGLUArgs {
  CUtensorMap tmA, tmB, tm_a, tm_y;
  const float* r;
  int save_y;
  int M, N, K;
  int ln;        // LayerNorm variant: y = r acc - (r mu) w1 + b1
  const float* mu;
  const float* w1;
  const float* b1;
};
cudaError_t launch_rowscale_swiglu(const RowScaleSwiGLUArgs& a, const LaunchCtx& lc);

struct RopeArgs {
  CUtensorMap tmA, tmB, tm_out, tm_save;
  const float* r;
  const float2* cs;
  int seq_len, head_dim, n_rope, save;
  int M, N, K;
};
cudaError_t launch_rope(const RopeArgs& a, const LaunchCtx& lc);

struct CEArgs {
  CUtensorMap tmA, tmB;
  const int* targets;
  float2* part;
  float* tlogit;
  int M, N, K;
};
cudaError_t launch_ce(const CEArgs& a, const LaunchCtx& lc);

struct CEGradArgs {
  CUtensorMap tmA, tmB, tm_g;
  const int* targets;
  const float* lse;
  const float* dloss;
  int v0;
  int M, N, K;
};
cudaError_t launch_ce_grad(const CEGradArgs& a, const LaunchCtx& lc);

struct SwiGLUBwdArgs {
  CUtensorMap tmA, tmB, tm_y, tm_dy;
  const float* r;
  float* spart;
  int M, N, K;
  int ln;        // LayerNorm variant: also sum dy w1 and sum dy b1 partials
  const float* w1;
  const float* b1;
  float* spart_w;
  float* spart_b;
};
cudaError_t launch_swiglu_bwd(const SwiGLUBwdArgs& a, const LaunchCtx& lc);

struct NormBwdArgs {
  CUtensorMap tmA, tmB, tm_dh, tm_hhat;
  const bf16* h;      // [M, N] (read by the epilogue without TMA)
  const bf16* dres;   // nullable [M, N]
  const bf16* gamma;
  const float* r;
  const float* s;
  float* dgpart;
  int M, N, K;
  int ln;        // LayerNorm variant (s is s_b)
  const float* mu;
  const float* sa;
  const bf16* beta;
  float* dbpart;
  int save_hhat;
};
cudaError_t launch_norm_bwd(const NormBwdArgs& a, const LaunchCtx& lc);

// text returned by coda_last_error_string() for this thread
void set_last_error(const char* msg);

// Rows of an A box (one CTA's slab); columns of the per-tile (max, sum-exp)
// partials of the LM-head cross-entropy (its GEMM always runs 256-wide tiles);
// columns per row partial of every other epilogue (kPartCols in core/gemm.cuh).
constexpr int kTileM = 128;
constexpr int kCeTileN = 256;
constexpr int kRowPartCols = 128;

// auxiliary kernels
cudaError_t launch_row_rms(const float* part, int nparts, int M, float inv_d, float eps, float* r,
                           cudaStream_t st);
cudaError_t launch_row_sum_scale(const float* part, int nparts, int M, float scale, float* out,
                                 cudaStream_t st);
cudaError_t launch_col_reduce(const float* part, int nparts, int N, float* out, cudaStream_t st);
cudaError_t launch_ce_combine(const float2* part, int nparts, const float* tlogit, const int* targets,
                              int M, int V, float* lse, float* loss, int* err, cudaStream_t st);
cudaError_t launch_rope_table(float2* cs, int seq_len, int head_dim, double theta, cudaStream_t st);
cudaError_t launch_rope_bwd(const bf16* d, const __half* q, const float* r, const float2* cs,
                            int seq_len, int head_dim, int n_rope, bf16* out, float* s, int M, int N,
                            float inv_d, cudaStream_t st);
cudaError_t launch_ln_stats(const float* part_sq, const float* part_sum, int nparts, int M, float inv_d,
                            float eps, float* r, float* mu, cudaStream_t st);
cudaError_t launch_ln_bwd_stats(const float* spart, const float* spart_w, const float* spart_b,
                                int nparts, int M, float inv_d, float* sa, float* sb, cudaStream_t st);
cudaError_t launch_bounded_wait_probe(int* err, unsigned long long timeout_ns, cudaStream_t st);

}  // namespace coda
