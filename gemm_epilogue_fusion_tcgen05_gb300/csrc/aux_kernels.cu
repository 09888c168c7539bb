// Auxiliary reductions and the RoPE backward pairwise map.
//
// "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs", Fig. 4
// caption: a small auxiliary kernel reduces the GEMM epilogue's tile partials
// to the row statistic r, reading a few values per tile rather than the whole
// activation. The same two-level scheme gives s (backward), the LM-head
// log-sum-exp (combine of per-tile max / sum-exp), and the RMSNorm weight
// gradient (column sums of per-32-row partials). Partials are laid out
// [nparts][M] (or [nparts][N]) so that neighbouring threads read neighbouring
// rows: every load is coalesced.
#include <cuda_runtime.h>
#include <cstdint>
#include <cuda_bf16.h>
#include "internal.h"

namespace coda {

// r[m] = 1 / sqrt(sum_j part[j, m] * inv_d + eps)
__global__ void row_rms_kernel(const float* __restrict__ part, int nparts, int M, float inv_d,
                               float eps, float* __restrict__ r) {
  grid_dep_wait();  // the producer of our inputs has finished (no-op without PDL)
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  float acc = 0.f;
  int j = 0;
  for (; j + 4 <= nparts; j += 4) {
    const float a = __ldg(part + (size_t)j * M + m);
    const float b = __ldg(part + (size_t)(j + 1) * M + m);
    const float c = __ldg(part + (size_t)(j + 2) * M + m);
    const float d = __ldg(part + (size_t)(j + 3) * M + m);
    acc += (a + b) + (c + d);
  }
  for (; j < nparts; ++j) acc += __ldg(part + (size_t)j * M + m);
  r[m] = 1.0f / sqrtf(fmaf(acc, inv_d, eps));
}

// out[m] = scale * sum_j part[j, m]
__global__ void row_sum_scale_kernel(const float* __restrict__ part, int nparts, int M, float scale,
                                     float* __restrict__ out) {
  grid_dep_wait();  // the producer of our inputs has finished (no-op without PDL)
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  float acc = 0.f;
  for (int j = 0; j < nparts; ++j) acc += __ldg(part + (size_t)j * M + m);
  out[m] = acc * scale;
}

// out[n] = sum_j part[j, n]; a block of 32 x 8 threads covers 32 columns,
// the 8 rows of threads stride over j, then combine through shared memory.
__global__ void col_reduce_kernel(const float* __restrict__ part, int nparts, int N,
                                  float* __restrict__ out) {
  grid_dep_wait();  // the producer of our inputs has finished (no-op without PDL)
  __shared__ float sm[8][33];
  const int n = blockIdx.x * 32 + threadIdx.x;
  float acc = 0.f;
  if (n < N)
    for (int j = threadIdx.y; j < nparts; j += 8) acc += __ldg(part + (size_t)j * N + n);
  sm[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y == 0 && n < N) {
    float t = 0.f;
#pragma unroll
    for (int y = 0; y < 8; ++y) t += sm[y][threadIdx.x];
    out[n] = t;
  }
}

// LSE = M* + log sum_j s_j exp(m_j - M*), loss = LSE - target logit.
// A block of 32 x 8 threads handles 32 rows; 8 lanes of j per row.
__global__ void ce_combine_kernel(const float2* __restrict__ part, int nparts,
                                  const float* __restrict__ tlogit, const int* __restrict__ targets,
                                  int M, int V, float* __restrict__ lse, float* __restrict__ loss,
                                  int* err) {
  grid_dep_wait();  // the producer of our inputs has finished (no-op without PDL)
  __shared__ float smax[8][33], ssum[8][33];
  const int m = blockIdx.x * 32 + threadIdx.x;
  float mx = -INFINITY, sm = 0.f;
  if (m < M) {
    for (int j = threadIdx.y; j < nparts; j += 8) {
      const float2 p = __ldg(part + (size_t)j * M + m);
      const float nm = fmaxf(mx, p.x);
      sm = sm * expf(mx - nm) + p.y * expf(p.x - nm);
      mx = nm;
    }
  }
  smax[threadIdx.y][threadIdx.x] = mx;
  ssum[threadIdx.y][threadIdx.x] = sm;
  __syncthreads();
  if (threadIdx.y == 0 && m < M) {
    float gm = -INFINITY;
#pragma unroll
    for (int y = 0; y < 8; ++y) gm = fmaxf(gm, smax[y][threadIdx.x]);
    float s = 0.f;
#pragma unroll
    for (int y = 0; y < 8; ++y) {
      const float my = smax[y][threadIdx.x];
      if (my != -INFINITY) s += ssum[y][threadIdx.x] * expf(my - gm);
    }
    const float l = gm + logf(s);
    lse[m] = l;
    const int t = targets[m];
    if (t < 0 || t >= V) {
      loss[m] = __int_as_float(0x7fc00000);  // NaN: the target index is out of range
      if (err) atomicCAS(err, 0, kErrInvalid | (20 << 8));
    } else {
      loss[m] = l - tlogit[m];
    }
  }
}

// cos_sin[p, i] = (cos(p theta_i), sin(p theta_i)), theta_i = theta^(-2i/hd),
// evaluated in fp64 and rounded to fp32.
__global__ void rope_table_kernel(float2* __restrict__ cs, int seq_len, int head_dim, double theta) {
  grid_dep_wait();  // the producer of our inputs has finished (no-op without PDL)
  const int half = head_dim / 2;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= seq_len * half) return;
  const int p = idx / half, i = idx % half;
  const double inv = pow(theta, -2.0 * (double)i / (double)head_dim);
  double s, c;
  sincos((double)p * inv, &s, &c);
  cs[idx] = make_float2((float)c, (float)s);
}

// RoPE backward with the delayed row scale and the relocated RMSNorm
// statistic (the GEMM producing this gradient, attention backward, is not
// part of this library, so this pairwise map runs on its own):
//   dhat = r[m] * R(pos)^T d   (pairs of the q and k columns; v unrotated)
//   s[m] = inv_d * sum_n d[m, n] * q[m, n]   (rotation keeps dot products;
//          q is the fp16 copy of the forward output kept for this purpose)
// One block of 128 threads per row; vectors of 8 columns (4 pairs).
__global__ void rope_bwd_kernel(const __nv_bfloat16* __restrict__ d, const __half* __restrict__ q,
                                const float* __restrict__ r, const float2* __restrict__ cs,
                                int seq_len, int head_dim, int n_rope, __nv_bfloat16* __restrict__ out,
                                float* __restrict__ s, int M, int N, float inv_d) {
  grid_dep_wait();  // the producer of our inputs has finished (no-op without PDL)
  const int m = blockIdx.x;
  if (m >= M) return;
  const float rr = r ? __ldg(r + m) : 1.f;
  const int pos = m % seq_len;
  const uint4* drow = reinterpret_cast<const uint4*>(d + (size_t)m * N);
  const uint4* qrow = reinterpret_cast<const uint4*>(q + (size_t)m * N);
  uint4* orow = reinterpret_cast<uint4*>(out + (size_t)m * N);
  const float2* csr = cs + (size_t)pos * (head_dim / 2);
  float acc = 0.f;
  const int nvec = N / 8;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint4 du = __ldg(drow + v);
    const uint4 qu = __ldg(qrow + v);
    const uint32_t dw[4] = {du.x, du.y, du.z, du.w};
    const uint32_t qw[4] = {qu.x, qu.y, qu.z, qu.w};
    float qv[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&qw[t]));
      qv[2 * t] = f.x;
      qv[2 * t + 1] = f.y;
    }
    const int col = v * 8;
    const bool rot = col < n_rope;
    const int i0 = (col % head_dim) / 2;
    uint32_t ow[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float e = bf16_lo(dw[t]), o = bf16_hi(dw[t]);
      acc = fmaf(e, qv[2 * t], fmaf(o, qv[2 * t + 1], acc));
      float ee = e, oo = o;
      if (rot) {
        const float2 c = __ldg(csr + i0 + t);
        ee = e * c.x + o * c.y;   // R^T: rotate by the negative angle
        oo = -e * c.y + o * c.x;
      }
      ow[t] = pack_bf16(rr * ee, rr * oo);
    }
    orow[v] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  }
  // block reduction of acc
  __shared__ float red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) s[m] = t * inv_d;
  }
}

// LayerNorm statistics from per-tile sums of h^2 and of h:
//   mu = sum h / d ; r = 1 / sqrt(max(sum h^2 / d - mu^2, 0) + eps)
__global__ void ln_stats_kernel(const float* __restrict__ psq, const float* __restrict__ psum,
                                int nparts, int M, float inv_d, float eps, float* __restrict__ r,
                                float* __restrict__ mu) {
  grid_dep_wait();  // the producer of our inputs has finished (no-op without PDL)
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  float a = 0.f, b = 0.f;
  for (int j = 0; j < nparts; ++j) {
    a += __ldg(psq + (size_t)j * M + m);
    b += __ldg(psum + (size_t)j * M + m);
  }
  const float mean = b * inv_d;
  const float var = fmaxf(fmaf(a, inv_d, -mean * mean), 0.f);
  mu[m] = mean;
  r[m] = 1.0f / sqrtf(var + eps);
}

// The two relocated LayerNorm-backward statistics:
//   s_a = sum dy w1 / d ; s_b = (sum dy y - sum dy b1) / d
__global__ void ln_bwd_stats_kernel(const float* __restrict__ sp, const float* __restrict__ spw,
                                    const float* __restrict__ spb, int nparts, int M, float inv_d,
                                    float* __restrict__ sa, float* __restrict__ sb) {
  grid_dep_wait();  // the producer of our inputs has finished (no-op without PDL)
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  float y = 0.f, w = 0.f, b = 0.f;
  for (int j = 0; j < nparts; ++j) {
    y += __ldg(sp + (size_t)j * M + m);
    w += __ldg(spw + (size_t)j * M + m);
    b += __ldg(spb + (size_t)j * M + m);
  }
  sa[m] = w * inv_d;
  sb[m] = (y - b) * inv_d;
}

// A kernel whose only job is to wait on an mbarrier that nothing arrives at,
// with a short bound: it must give up, record CODA_ERR_TIMEOUT and return.
// Used by the tests of the bounded-wait machinery.
__global__ void bounded_wait_probe_kernel(int* err, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    DevError e{err, &abort_flag, timeout_ns};
    (void)mbar_wait(smem_u32(&bar), 0, e, 99);
  }
}

// ------------------------------------------------------------------ launchers
// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream drains and waits for it in
// grid_dep_wait(). These kernels never release their own dependents early
// (their grids can span several waves), so nothing can crowd them out.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_row_rms(const float* part, int nparts, int M, float inv_d, float eps, float* r,
                           cudaStream_t st) {
  return launch_pdl(row_rms_kernel, dim3((M + 255) / 256), dim3(256), st, part, nparts, M, inv_d, eps, r);
}
cudaError_t launch_row_sum_scale(const float* part, int nparts, int M, float scale, float* out,
                                 cudaStream_t st) {
  return launch_pdl(row_sum_scale_kernel, dim3((M + 255) / 256), dim3(256), st, part, nparts, M, scale,
                    out);
}
cudaError_t launch_col_reduce(const float* part, int nparts, int N, float* out, cudaStream_t st) {
  return launch_pdl(col_reduce_kernel, dim3((N + 31) / 32), dim3(32, 8), st, part, nparts, N, out);
}
cudaError_t launch_ce_combine(const float2* part, int nparts, const float* tlogit, const int* targets,
                              int M, int V, float* lse, float* loss, int* err, cudaStream_t st) {
  return launch_pdl(ce_combine_kernel, dim3((M + 31) / 32), dim3(32, 8), st, part, nparts, tlogit,
                    targets, M, V, lse, loss, err);
}
cudaError_t launch_rope_table(float2* cs, int seq_len, int head_dim, double theta, cudaStream_t st) {
  const int n = seq_len * (head_dim / 2);
  return launch_pdl(rope_table_kernel, dim3((n + 255) / 256), dim3(256), st, cs, seq_len, head_dim,
                    theta);
}
cudaError_t launch_rope_bwd(const __nv_bfloat16* d, const __half* q, const float* r,
                            const float2* cs, int seq_len, int head_dim, int n_rope,
                            __nv_bfloat16* out, float* s, int M, int N, float inv_d, cudaStream_t st) {
  return launch_pdl(rope_bwd_kernel, dim3(M), dim3(128), st, d, q, r, cs, seq_len, head_dim, n_rope,
                    out, s, M, N, inv_d);
}
cudaError_t launch_ln_stats(const float* part_sq, const float* part_sum, int nparts, int M, float inv_d,
                            float eps, float* r, float* mu, cudaStream_t st) {
  return launch_pdl(ln_stats_kernel, dim3((M + 255) / 256), dim3(256), st, part_sq, part_sum, nparts,
                    M, inv_d, eps, r, mu);
}
cudaError_t launch_ln_bwd_stats(const float* spart, const float* spart_w, const float* spart_b,
                                int nparts, int M, float inv_d, float* sa, float* sb, cudaStream_t st) {
  return launch_pdl(ln_bwd_stats_kernel, dim3((M + 255) / 256), dim3(256), st, spart, spart_w,
                    spart_b, nparts, M, inv_d, sa, sb);
}
cudaError_t launch_bounded_wait_probe(int* err, unsigned long long timeout_ns, cudaStream_t st) {
  bounded_wait_probe_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace coda
