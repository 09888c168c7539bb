// C-ABI layer of libcoda: argument checks, TMA descriptor encoding and
// launches. Nothing here allocates device memory: every tensor and every
// scratch buffer is owned by the caller.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "coda.h"
#include "internal.h"

using namespace coda;

namespace {

__device__ int g_coda_err;  // device error word, one per device

thread_local std::string t_last_error;
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_skip_kb{-1};  // coda_debug_skip_kblock

// Every host-side error message lands here; with the environment variable
// CODA_DEBUG set to anything but "0" (read once) it is also written to
// stderr as it happens.
void note_host_error(const char* msg) {
  t_last_error = msg;
  static const bool echo = [] {
    const char* v = std::getenv("CODA_DEBUG");
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
  }();
  if (echo) std::fprintf(stderr, "libcoda: %s\n", msg);
}

coda_status_t fail(coda_status_t s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
coda_status_t fail(coda_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  note_host_error(buf);
  return s;
}

coda_status_t from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return CODA_OK;
  return fail(CODA_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct DevInfo {
  int ok = -1;  // -1 unknown, 0 unsupported, 1 supported
  int num_sms = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

coda_status_t launch_ctx(cudaStream_t st, LaunchCtx& lc) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(CODA_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (di.ok < 0) {
    int major = 0, minor = 0, sms = 0;
    // a failed query is reported, not cached as an unsupported device
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return from_cuda(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      di.ok = 0;
      return fail(CODA_ERR_UNSUPPORTED, "libcoda is built for sm_103a; device %d is sm_%d%d", dev,
                  major, minor);
    }
    di.num_sms = sms;
    di.ok = 1;
  }
  if (di.ok == 0) return fail(CODA_ERR_UNSUPPORTED, "device %d is not sm_103", dev);
  if (!encode_fn()) return fail(CODA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled not available");
  // The error word's device address is looked up on every call, not kept:
  // after a cudaDeviceReset the module is loaded again and a kept address
  // would point at memory the new context does not own.
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_coda_err);
  if (e != cudaSuccess) return from_cuda(e, "cudaGetSymbolAddress(error word)");
  lc.stream = st;
  lc.err = static_cast<int*>(p);
  lc.timeout_ns = g_timeout_ns.load();
  lc.num_sms = di.num_sms;
  lc.skip_kb = g_skip_kb.load();
  return CODA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D tensor map over a row-major matrix [outer, inner] with row stride ld
// (elements) and box [box_outer, box_inner].
bool tmap2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
            uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer,
            CUtensorMapSwizzle sw) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * (uint64_t)esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = encode_fn()(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Operand maps for the mainloop: 64-element (128-byte) swizzled rows.
bool map_a(CUtensorMap* m, const void* A, int lda, int transA, int M, int K) {
  if (!transA) return tmap2d(m, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, M, lda, 64, kTileM,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  return tmap2d(m, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, lda, 64, 64,
                CU_TENSOR_MAP_SWIZZLE_128B);
}
// Both forms load 64 x 64 boxes; the kernel issues as many as its tile needs.
bool map_b(CUtensorMap* m, const void* B, int ldb, int transB, int N, int K) {
  if (!transB) return tmap2d(m, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, K, ldb, 64, 64,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  return tmap2d(m, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N, ldb, 64, 64,
                CU_TENSOR_MAP_SWIZZLE_128B);
}
// Epilogue boxes of 32 rows: 32 bf16 (64 B), 16 bf16 (32 B), 64 bf16 (128 B), 32 fp32 (128 B).
bool map_bf16_32(CUtensorMap* m, const void* p, int rows, int cols, int ld) {
  return tmap2d(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, ld, 32, 32,
                CU_TENSOR_MAP_SWIZZLE_64B);
}
bool map_bf16_16(CUtensorMap* m, const void* p, int rows, int cols, int ld) {
  return tmap2d(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, ld, 16, 32,
                CU_TENSOR_MAP_SWIZZLE_32B);
}
bool map_bf16_64(CUtensorMap* m, const void* p, int rows, int cols, int ld) {
  return tmap2d(m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, ld, 64, 32,
                CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_f16_32(CUtensorMap* m, const void* p, int rows, int cols, int ld) {
  return tmap2d(m, p, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, cols, rows, ld, 32, 32,
                CU_TENSOR_MAP_SWIZZLE_64B);
}
bool map_f16_64(CUtensorMap* m, const void* p, int rows, int cols, int ld) {
  return tmap2d(m, p, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, cols, rows, ld, 64, 32,
                CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_f32_32(CUtensorMap* m, const void* p, int rows, int cols, int ld) {
  return tmap2d(m, p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, cols, rows, ld, 32, 32,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

#define CHECK_PTR(p)                                                                          \
  do {                                                                                        \
    if ((p) == nullptr) return fail(CODA_ERR_INVALID_VALUE, "%s: %s is null", __func__, #p);  \
    if (!aligned16(p))                                                                        \
      return fail(CODA_ERR_INVALID_VALUE, "%s: %s is not 16-byte aligned", __func__, #p);     \
  } while (0)
#define CHECK_OPT_PTR(p)                                                                      \
  do {                                                                                        \
    if ((p) != nullptr && !aligned16(p))                                                      \
      return fail(CODA_ERR_INVALID_VALUE, "%s: %s is not 16-byte aligned", __func__, #p);     \
  } while (0)
#define CHECK(cond, ...)                                            \
  do {                                                              \
    if (!(cond)) return fail(CODA_ERR_INVALID_VALUE, __VA_ARGS__);  \
  } while (0)
#define CHECK_MAP(expr)                                                                      \
  do {                                                                                       \
    if (!(expr)) return fail(CODA_ERR_INVALID_VALUE, "%s: tensor map rejected (%s)", __func__, #expr); \
  } while (0)
#define TRY_CTX(st, lc)                          \
  LaunchCtx lc;                                  \
  do {                                           \
    coda_status_t s_ = launch_ctx((st), lc);     \
    if (s_ != CODA_OK) return s_;                \
  } while (0)

constexpr int kMaxDim = 1 << 30;

}  // namespace

namespace coda {
// lets other translation units of the library report a host-side error
void set_last_error(const char* msg) { note_host_error(msg); }
}  // namespace coda

extern "C" {

int coda_version(void) { return 100; }
int coda_col_tiles(int N) { return N <= 0 ? 0 : (N + kRowPartCols - 1) / kRowPartCols; }
int coda_row_tiles32(int M) { return M <= 0 ? 0 : (M + 31) / 32; }
void coda_set_timeout_ms(int ms) {
  if (ms < 1) ms = 1;
  g_timeout_ns.store((unsigned long long)ms * 1000000ull);
}

const char* coda_last_error_string(void) { return t_last_error.c_str(); }

void coda_debug_skip_kblock(int kb) { g_skip_kb.store(kb >= 0 ? kb : -1); }

coda_status_t coda_get_device_error(coda_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return from_cuda(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_coda_err, sizeof(int));
  if (e != cudaSuccess) return from_cuda(e, "read device error word");
  if (v == 0) return CODA_OK;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_coda_err, &zero, sizeof(int));
  if (e != cudaSuccess) return from_cuda(e, "clear the device error word");
  const int code = v & 0xff, where = v >> 8;
  if (code == kErrTimeout)
    return fail(CODA_ERR_TIMEOUT, "a bounded wait in a kernel ran out (site %d)", where);
  if (code == kErrRange)
    return fail(CODA_ERR_RANGE, "a value saved in fp16 was outside the fp16 range (site %d)",
                where);
  return fail(CODA_ERR_INVALID_VALUE, "device-side invalid value (site %d)", where);
}

coda_status_t coda_gemm(const void* A, int lda, int transA, const void* B, int ldb, int transB,
                        const void* resid, float* rowsq_part, void* C, int ldc, int c_fp32, int M,
                        int N, int K, coda_stream_t stream) {
  CHECK_PTR(A);
  CHECK_PTR(B);
  CHECK_PTR(C);
  CHECK_OPT_PTR(resid);
  CHECK_OPT_PTR(rowsq_part);
  CHECK(M > 0 && N > 0 && K > 0 && M < kMaxDim && N < kMaxDim && K < kMaxDim,
        "coda_gemm: bad sizes M=%d N=%d K=%d", M, N, K);
  CHECK(lda >= (transA ? M : K) && ldb >= (transB ? K : N) && ldc >= N,
        "coda_gemm: leading dimension too small");
  CHECK(lda % 8 == 0 && ldb % 8 == 0 && ldc % (c_fp32 ? 4 : 8) == 0,
        "coda_gemm: row strides must be multiples of 16 bytes");
  CHECK(!rowsq_part || (!transA && !transB && !c_fp32),
        "coda_gemm: rowsq_part needs transA=0, transB=0, bf16 output");
  CHECK(!resid || (!transA && (c_fp32 || !transB)),
        "coda_gemm: resid needs transA=0 (and transB=0 for a bf16 output)");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  PlainArgs a{};
  CHECK_MAP(map_a(&a.tmA, A, lda, transA, M, K));
  CHECK_MAP(map_b(&a.tmB, B, ldb, transB, N, K));
  if (c_fp32) CHECK_MAP(map_f32_32(&a.tmC, C, M, N, ldc));
  else CHECK_MAP(map_bf16_32(&a.tmC, C, M, N, ldc));
  a.resid_ptr = resid;
  a.ld_res = (size_t)ldc * (c_fp32 ? 4 : 2);
  a.a_mn = transA != 0;
  a.b_mn = transB == 0;
  a.out_f32 = c_fp32 != 0;
  a.resid = resid != nullptr;
  a.rowsq = rowsq_part != nullptr;
  a.rowsq_part = rowsq_part;
  a.M = M;
  a.N = N;
  a.K = K;
  return from_cuda(launch_plain(a, lc), "coda_gemm launch");
}

coda_status_t coda_gemm_resid_norm_stats(const void* x, const void* W0, const void* z,
                                         const void* gamma, void* h, void* hg, float* part, int M,
                                         int N, int K, coda_stream_t stream) {
  CHECK_PTR(x);
  CHECK_PTR(W0);
  CHECK_PTR(z);
  CHECK_PTR(gamma);
  CHECK_PTR(h);
  CHECK_PTR(hg);
  CHECK_PTR(part);
  CHECK(M > 0 && N > 0 && K > 0 && M < kMaxDim && N < kMaxDim && K < kMaxDim,
        "coda_gemm_resid_norm_stats: bad sizes");
  CHECK(N % 8 == 0 && K % 8 == 0, "coda_gemm_resid_norm_stats: N and K must be multiples of 8");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  ResidNormStatsArgs a{};
  CHECK_MAP(map_a(&a.tmA, x, K, 0, M, K));
  CHECK_MAP(map_b(&a.tmB, W0, N, 0, N, K));
  a.z = static_cast<const bf16*>(z);
  CHECK_MAP(map_bf16_32(&a.tm_h, h, M, N, N));
  CHECK_MAP(map_bf16_32(&a.tm_hg, hg, M, N, N));
  a.gamma = static_cast<const bf16*>(gamma);
  a.part = part;
  a.M = M;
  a.N = N;
  a.K = K;
  return from_cuda(launch_resid_norm_stats(a, lc), "coda_gemm_resid_norm_stats launch");
}

coda_status_t coda_row_rms(const float* part, int nparts, int M, int d, float eps, float* r,
                           coda_stream_t stream) {
  CHECK_PTR(part);
  CHECK_PTR(r);
  CHECK(nparts > 0 && M > 0 && d > 0, "coda_row_rms: bad sizes");
  CHECK(eps >= 0.f, "coda_row_rms: eps must be >= 0");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  return from_cuda(launch_row_rms(part, nparts, M, 1.0f / (float)d, eps, r, lc.stream),
                   "coda_row_rms launch");
}

coda_status_t coda_gemm_rowscale_swiglu(const void* hg, const void* W1, const float* r, void* a,
                                        void* y_save, int M, int two_f, int K,
                                        coda_stream_t stream) {
  CHECK_PTR(hg);
  CHECK_PTR(W1);
  CHECK_PTR(r);
  CHECK_PTR(a);
  CHECK_OPT_PTR(y_save);
  CHECK(M > 0 && two_f > 0 && K > 0 && M < kMaxDim && two_f < kMaxDim && K < kMaxDim,
        "coda_gemm_rowscale_swiglu: bad sizes");
  CHECK(two_f % 16 == 0 && K % 8 == 0,
        "coda_gemm_rowscale_swiglu: two_f must be a multiple of 16, K of 8");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  RowScaleSwiGLUArgs p{};
  CHECK_MAP(map_a(&p.tmA, hg, K, 0, M, K));
  CHECK_MAP(map_b(&p.tmB, W1, two_f, 0, two_f, K));
  CHECK_MAP(map_bf16_16(&p.tm_a, a, M, two_f / 2, two_f / 2));
  if (y_save) CHECK_MAP(map_f16_32(&p.tm_y, y_save, M, two_f, two_f));
  else p.tm_y = p.tm_a;  // unused
  p.r = r;
  p.save_y = y_save != nullptr;
  p.M = M;
  p.N = two_f;
  p.K = K;
  return from_cuda(launch_rowscale_swiglu(p, lc), "coda_gemm_rowscale_swiglu launch");
}

coda_status_t coda_gemm_rope(const void* A, const void* W, const float* r, const float* cos_sin,
                             int seq_len, int head_dim, int n_rope_cols, void* out, void* out_f16,
                             int M, int N, int K, coda_stream_t stream) {
  CHECK_PTR(A);
  CHECK_PTR(W);
  CHECK_OPT_PTR(r);
  CHECK_PTR(cos_sin);
  CHECK_PTR(out);
  CHECK_OPT_PTR(out_f16);
  CHECK(M > 0 && N > 0 && K > 0 && M < kMaxDim && N < kMaxDim && K < kMaxDim,
        "coda_gemm_rope: bad sizes");
  CHECK(N % 8 == 0 && K % 8 == 0, "coda_gemm_rope: N and K must be multiples of 8");
  CHECK(seq_len > 0 && head_dim > 0 && head_dim % 32 == 0, "coda_gemm_rope: head_dim must be a positive multiple of 32");
  CHECK(n_rope_cols >= 0 && n_rope_cols <= N && n_rope_cols % head_dim == 0,
        "coda_gemm_rope: n_rope_cols must be a multiple of head_dim and <= N");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  RopeArgs p{};
  CHECK_MAP(map_a(&p.tmA, A, K, 0, M, K));
  CHECK_MAP(map_b(&p.tmB, W, N, 0, N, K));
  CHECK_MAP(map_bf16_32(&p.tm_out, out, M, N, N));
  if (out_f16) CHECK_MAP(map_f16_32(&p.tm_save, out_f16, M, N, N));
  else p.tm_save = p.tm_out;  // unused
  p.save = out_f16 != nullptr;
  p.r = r;
  p.cs = reinterpret_cast<const float2*>(cos_sin);
  p.seq_len = seq_len;
  p.head_dim = head_dim;
  p.n_rope = n_rope_cols;
  p.M = M;
  p.N = N;
  p.K = K;
  return from_cuda(launch_rope(p, lc), "coda_gemm_rope launch");
}

coda_status_t coda_rope_table(float* cos_sin, int seq_len, int head_dim, double theta,
                              coda_stream_t stream) {
  CHECK_PTR(cos_sin);
  CHECK(seq_len > 0 && head_dim > 0 && head_dim % 2 == 0 && theta > 0.0,
        "coda_rope_table: bad arguments");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  return from_cuda(launch_rope_table(reinterpret_cast<float2*>(cos_sin), seq_len, head_dim, theta,
                                     lc.stream),
                   "coda_rope_table launch");
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int ce_tiles(int V) { return (V + kCeTileN - 1) / kCeTileN; }

size_t coda_lmhead_ce_workspace_size(int M, int V) {
  if (M <= 0 || V <= 0) return 0;
  return align256((size_t)ce_tiles(V) * M * sizeof(float2)) + align256((size_t)M * sizeof(float));
}

coda_status_t coda_lmhead_ce(const void* hidden, const void* W, const int32_t* targets, float* lse,
                             float* loss, void* ws, size_t ws_bytes, int M, int V, int d,
                             coda_stream_t stream) {
  CHECK_PTR(hidden);
  CHECK_PTR(W);
  CHECK_PTR(targets);
  CHECK_PTR(lse);
  CHECK_PTR(loss);
  CHECK_PTR(ws);
  CHECK(M > 0 && V > 0 && d > 0 && M < kMaxDim && V < kMaxDim && d < kMaxDim,
        "coda_lmhead_ce: bad sizes");
  CHECK(V % 8 == 0 && d % 8 == 0, "coda_lmhead_ce: V and d must be multiples of 8");
  CHECK(ws_bytes >= coda_lmhead_ce_workspace_size(M, V),
        "coda_lmhead_ce: workspace too small (%zu < %zu)", ws_bytes,
        coda_lmhead_ce_workspace_size(M, V));
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  CEArgs p{};
  CHECK_MAP(map_a(&p.tmA, hidden, d, 0, M, d));
  CHECK_MAP(map_b(&p.tmB, W, V, 0, V, d));
  const int nparts = ce_tiles(V);
  p.targets = targets;
  p.part = static_cast<float2*>(ws);
  p.tlogit = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                      align256((size_t)nparts * M * sizeof(float2)));
  p.M = M;
  p.N = V;
  p.K = d;
  coda_status_t s = from_cuda(launch_ce(p, lc), "coda_lmhead_ce GEMM launch");
  if (s != CODA_OK) return s;
  return from_cuda(launch_ce_combine(p.part, nparts, p.tlogit, targets, M, V, lse, loss, lc.err,
                                     lc.stream),
                   "coda_lmhead_ce combine launch");
}

// Vocabulary columns per chunk of the CE backward. Wider chunks mean fewer
// read-modify-write passes over the fp32 dhidden and fewer, longer-K GEMMs:
// at M = 8192, d = 2048, V = 128256 the backward took 8.58 / 7.92 / 7.80 /
// 7.70 ms with chunks of 4096 / 8192 / 16384 / 32768. The recommended
// workspace holds 16384 columns; a larger one is used up to 32768.
constexpr int kCeBwdChunk = 16384;
constexpr int kCeBwdMaxChunk = 32768;
static int ce_bwd_chunk(int M, int V, size_t ws_bytes) {
  const int vr = (V + 255) / 256 * 256;
  size_t c = ws_bytes / ((size_t)M * 2) / 256 * 256;
  if (c > kCeBwdMaxChunk) c = kCeBwdMaxChunk;
  if (c > (size_t)vr) c = vr;
  return (int)c;
}

size_t coda_lmhead_ce_bwd_workspace_size(int M, int V) {
  if (M <= 0 || V <= 0) return 0;
  const int vr = (V + 255) / 256 * 256;
  return (size_t)M * (vr < kCeBwdChunk ? vr : kCeBwdChunk) * 2;
}

coda_status_t coda_lmhead_ce_bwd(const void* hidden, const void* W, const int32_t* targets,
                                 const float* lse, const float* dloss, float* dhidden, float* dW,
                                 void* ws, size_t ws_bytes, int M, int V, int d,
                                 coda_stream_t stream) {
  CHECK_PTR(hidden);
  CHECK_PTR(W);
  CHECK_PTR(targets);
  CHECK_PTR(lse);
  CHECK_PTR(dloss);
  CHECK_PTR(dhidden);
  CHECK_PTR(dW);
  CHECK_PTR(ws);
  CHECK(M > 0 && V > 0 && d > 0 && M < kMaxDim && V < kMaxDim && d < kMaxDim,
        "coda_lmhead_ce_bwd: bad sizes");
  CHECK(V % 8 == 0 && d % 8 == 0, "coda_lmhead_ce_bwd: V and d must be multiples of 8");
  const int chunk = ce_bwd_chunk(M, V, ws_bytes);
  CHECK(chunk >= 256, "coda_lmhead_ce_bwd: workspace too small (%zu bytes; at least %zu)",
        ws_bytes, (size_t)M * 256 * 2);
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  const bf16* Wb = static_cast<const bf16*>(W);
  for (int v0 = 0; v0 < V; v0 += chunk) {
    const int vc = V - v0 < chunk ? V - v0 : chunk;
    // (1) logits of this chunk, recomputed; the epilogue forms G in bf16
    CEGradArgs g{};
    CHECK_MAP(map_a(&g.tmA, hidden, d, 0, M, d));
    CHECK_MAP(tmap2d(&g.tmB, Wb + v0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, vc, d, V, 64, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B));
    CHECK_MAP(map_bf16_32(&g.tm_g, ws, M, vc, chunk));
    g.targets = targets;
    g.lse = lse;
    g.dloss = dloss;
    g.v0 = v0;
    g.M = M;
    g.N = vc;
    g.K = d;
    coda_status_t s = from_cuda(launch_ce_grad(g, lc), "coda_lmhead_ce_bwd logits launch");
    if (s != CODA_OK) return s;
    // (2) dhidden (+)= G W_chunk^T, fp32, accumulated over the chunks
    PlainArgs h{};
    CHECK_MAP(map_a(&h.tmA, ws, chunk, 0, M, vc));
    CHECK_MAP(tmap2d(&h.tmB, Wb + v0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, vc, d, V, 64, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B));
    CHECK_MAP(map_f32_32(&h.tmC, dhidden, M, d, d));
    h.resid_ptr = v0 > 0 ? dhidden : nullptr;
    h.ld_res = (size_t)d * 4;
    h.a_mn = false;
    h.b_mn = false;
    h.out_f32 = true;
    h.resid = v0 > 0;
    h.M = M;
    h.N = d;
    h.K = vc;
    s = from_cuda(launch_plain(h, lc), "coda_lmhead_ce_bwd dhidden launch");
    if (s != CODA_OK) return s;
    // (3) dW[:, v0 : v0 + vc] = hidden^T G
    PlainArgs w{};
    CHECK_MAP(map_a(&w.tmA, hidden, d, 1, d, M));
    CHECK_MAP(map_b(&w.tmB, ws, chunk, 0, vc, M));
    CHECK_MAP(map_f32_32(&w.tmC, dW + v0, d, vc, V));
    w.a_mn = true;
    w.b_mn = true;
    w.out_f32 = true;
    w.M = d;
    w.N = vc;
    w.K = M;
    s = from_cuda(launch_plain(w, lc), "coda_lmhead_ce_bwd dW launch");
    if (s != CODA_OK) return s;
  }
  return CODA_OK;
}

coda_status_t coda_gemm_rowscale_swiglu_bwd(const void* dout, const void* W2, const void* y,
                                            const float* r, void* dyhat, float* spart, int M,
                                            int f, int d, coda_stream_t stream) {
  CHECK_PTR(dout);
  CHECK_PTR(W2);
  CHECK_PTR(y);
  CHECK_PTR(r);
  CHECK_PTR(dyhat);
  CHECK_PTR(spart);
  CHECK(M > 0 && f > 0 && d > 0 && M < kMaxDim && f < kMaxDim / 2 && d < kMaxDim,
        "coda_gemm_rowscale_swiglu_bwd: bad sizes");
  CHECK(f % 8 == 0 && d % 8 == 0, "coda_gemm_rowscale_swiglu_bwd: f and d must be multiples of 8");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  SwiGLUBwdArgs p{};
  CHECK_MAP(map_a(&p.tmA, dout, d, 0, M, d));
  CHECK_MAP(map_b(&p.tmB, W2, d, 1, f, d));  // B[k, n] = W2[n, k]
  CHECK_MAP(map_f16_64(&p.tm_y, y, M, 2 * f, 2 * f));
  CHECK_MAP(map_bf16_64(&p.tm_dy, dyhat, M, 2 * f, 2 * f));
  p.r = r;
  p.spart = spart;
  p.M = M;
  p.N = f;
  p.K = d;
  return from_cuda(launch_swiglu_bwd(p, lc), "coda_gemm_rowscale_swiglu_bwd launch");
}

coda_status_t coda_row_rms_bwd(const float* spart, int nparts, int M, int d, float* s,
                               coda_stream_t stream) {
  CHECK_PTR(spart);
  CHECK_PTR(s);
  CHECK(nparts > 0 && M > 0 && d > 0, "coda_row_rms_bwd: bad sizes");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  return from_cuda(launch_row_sum_scale(spart, nparts, M, 1.0f / (float)d, s, lc.stream),
                   "coda_row_rms_bwd launch");
}

coda_status_t coda_gemm_resid_norm_stats_bwd(const void* dyhat, const void* W1, const void* h,
                                             const void* gamma, const float* r, const float* s,
                                             const void* dresid, void* dh, float* dgamma_part,
                                             int M, int d, int two_f, coda_stream_t stream) {
  CHECK_PTR(dyhat);
  CHECK_PTR(W1);
  CHECK_PTR(h);
  CHECK_PTR(gamma);
  CHECK_PTR(r);
  CHECK_PTR(s);
  CHECK_OPT_PTR(dresid);
  CHECK_PTR(dh);
  CHECK_PTR(dgamma_part);
  CHECK(M > 0 && d > 0 && two_f > 0 && M < kMaxDim && d < kMaxDim && two_f < kMaxDim,
        "coda_gemm_resid_norm_stats_bwd: bad sizes");
  CHECK(d % 8 == 0 && two_f % 8 == 0,
        "coda_gemm_resid_norm_stats_bwd: d and two_f must be multiples of 8");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  NormBwdArgs p{};
  CHECK_MAP(map_a(&p.tmA, dyhat, two_f, 0, M, two_f));
  CHECK_MAP(map_b(&p.tmB, W1, two_f, 1, d, two_f));  // B[k, n] = W1[n, k]
  CHECK_MAP(map_bf16_32(&p.tm_dh, dh, M, d, d));
  p.h = static_cast<const bf16*>(h);
  p.dres = static_cast<const bf16*>(dresid);
  p.gamma = static_cast<const bf16*>(gamma);
  p.r = r;
  p.s = s;
  p.dgpart = dgamma_part;
  p.M = M;
  p.N = d;
  p.K = two_f;
  return from_cuda(launch_norm_bwd(p, lc), "coda_gemm_resid_norm_stats_bwd launch");
}

coda_status_t coda_col_reduce(const float* part, int nparts, int N, float* out,
                              coda_stream_t stream) {
  CHECK_PTR(part);
  CHECK_PTR(out);
  CHECK(nparts > 0 && N > 0, "coda_col_reduce: bad sizes");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  return from_cuda(launch_col_reduce(part, nparts, N, out, lc.stream), "coda_col_reduce launch");
}

coda_status_t coda_gemm_rope_bwd(const void* dqkv_rot, const void* qkv_rot, const float* r,
                                 const float* cos_sin, int seq_len, int head_dim, int n_rope_cols,
                                 void* dqkv_hat, float* s, int M, int N, int d,
                                 coda_stream_t stream) {
  CHECK_PTR(dqkv_rot);
  CHECK_PTR(qkv_rot);
  CHECK_OPT_PTR(r);
  CHECK_PTR(cos_sin);
  CHECK_PTR(dqkv_hat);
  CHECK_PTR(s);
  CHECK(M > 0 && N > 0 && d > 0 && N % 8 == 0, "coda_gemm_rope_bwd: bad sizes");
  CHECK(seq_len > 0 && head_dim > 0 && head_dim % 8 == 0, "coda_gemm_rope_bwd: bad head_dim");
  CHECK(n_rope_cols >= 0 && n_rope_cols <= N && n_rope_cols % head_dim == 0,
        "coda_gemm_rope_bwd: n_rope_cols must be a multiple of head_dim and <= N");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  return from_cuda(launch_rope_bwd(static_cast<const bf16*>(dqkv_rot),
                                   static_cast<const __half*>(qkv_rot), r,
                                   reinterpret_cast<const float2*>(cos_sin), seq_len, head_dim,
                                   n_rope_cols, static_cast<bf16*>(dqkv_hat), s, M, N,
                                   1.0f / (float)d, lc.stream),
                   "coda_gemm_rope_bwd launch");
}

// ------------------------------------------------------------------ LayerNorm variant

coda_status_t coda_gemm_resid_ln_stats(const void* x, const void* W0, const void* z,
                                       const void* gamma, void* h, void* hg, float* part_sq,
                                       float* part_sum, int M, int N, int K, coda_stream_t stream) {
  CHECK_PTR(x);
  CHECK_PTR(W0);
  CHECK_PTR(z);
  CHECK_PTR(gamma);
  CHECK_PTR(h);
  CHECK_PTR(hg);
  CHECK_PTR(part_sq);
  CHECK_PTR(part_sum);
  CHECK(M > 0 && N > 0 && K > 0 && M < kMaxDim && N < kMaxDim && K < kMaxDim,
        "coda_gemm_resid_ln_stats: bad sizes");
  CHECK(N % 8 == 0 && K % 8 == 0, "coda_gemm_resid_ln_stats: N and K must be multiples of 8");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  ResidNormStatsArgs a{};
  CHECK_MAP(map_a(&a.tmA, x, K, 0, M, K));
  CHECK_MAP(map_b(&a.tmB, W0, N, 0, N, K));
  a.z = static_cast<const bf16*>(z);
  CHECK_MAP(map_bf16_32(&a.tm_h, h, M, N, N));
  CHECK_MAP(map_bf16_32(&a.tm_hg, hg, M, N, N));
  a.gamma = static_cast<const bf16*>(gamma);
  a.part = part_sq;
  a.part2 = part_sum;
  a.ln = 1;
  a.M = M;
  a.N = N;
  a.K = K;
  return from_cuda(launch_resid_norm_stats(a, lc), "coda_gemm_resid_ln_stats launch");
}

coda_status_t coda_row_ln(const float* part_sq, const float* part_sum, int nparts, int M, int d,
                          float eps, float* r, float* mu, coda_stream_t stream) {
  CHECK_PTR(part_sq);
  CHECK_PTR(part_sum);
  CHECK_PTR(r);
  CHECK_PTR(mu);
  CHECK(nparts > 0 && M > 0 && d > 0, "coda_row_ln: bad sizes");
  CHECK(eps >= 0.f, "coda_row_ln: eps must be >= 0");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  return from_cuda(launch_ln_stats(part_sq, part_sum, nparts, M, 1.0f / (float)d, eps, r, mu,
                                   lc.stream),
                   "coda_row_ln launch");
}

coda_status_t coda_gemm_ln_rowscale_swiglu(const void* hg, const void* W1, const float* r,
                                           const float* mu, const float* w1, const float* b1,
                                           void* a, void* y_save, int M, int two_f, int K,
                                           coda_stream_t stream) {
  CHECK_PTR(hg);
  CHECK_PTR(W1);
  CHECK_PTR(r);
  CHECK_PTR(mu);
  CHECK_PTR(w1);
  CHECK_PTR(b1);
  CHECK_PTR(a);
  CHECK_OPT_PTR(y_save);
  CHECK(M > 0 && two_f > 0 && K > 0 && M < kMaxDim && two_f < kMaxDim && K < kMaxDim,
        "coda_gemm_ln_rowscale_swiglu: bad sizes");
  CHECK(two_f % 16 == 0 && K % 8 == 0,
        "coda_gemm_ln_rowscale_swiglu: two_f must be a multiple of 16, K of 8");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  RowScaleSwiGLUArgs p{};
  CHECK_MAP(map_a(&p.tmA, hg, K, 0, M, K));
  CHECK_MAP(map_b(&p.tmB, W1, two_f, 0, two_f, K));
  CHECK_MAP(map_bf16_16(&p.tm_a, a, M, two_f / 2, two_f / 2));
  if (y_save) CHECK_MAP(map_f16_32(&p.tm_y, y_save, M, two_f, two_f));
  else p.tm_y = p.tm_a;  // unused
  p.r = r;
  p.mu = mu;
  p.w1 = w1;
  p.b1 = b1;
  p.ln = 1;
  p.save_y = y_save != nullptr;
  p.M = M;
  p.N = two_f;
  p.K = K;
  return from_cuda(launch_rowscale_swiglu(p, lc), "coda_gemm_ln_rowscale_swiglu launch");
}

coda_status_t coda_gemm_ln_rowscale_swiglu_bwd(const void* dout, const void* W2, const void* y,
                                               const float* r, const float* w1, const float* b1,
                                               void* dyhat, float* spart, float* spart_w,
                                               float* spart_b, int M, int f, int d,
                                               coda_stream_t stream) {
  CHECK_PTR(dout);
  CHECK_PTR(W2);
  CHECK_PTR(y);
  CHECK_PTR(r);
  CHECK_PTR(w1);
  CHECK_PTR(b1);
  CHECK_PTR(dyhat);
  CHECK_PTR(spart);
  CHECK_PTR(spart_w);
  CHECK_PTR(spart_b);
  CHECK(M > 0 && f > 0 && d > 0 && M < kMaxDim && f < kMaxDim / 2 && d < kMaxDim,
        "coda_gemm_ln_rowscale_swiglu_bwd: bad sizes");
  CHECK(f % 8 == 0 && d % 8 == 0,
        "coda_gemm_ln_rowscale_swiglu_bwd: f and d must be multiples of 8");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  SwiGLUBwdArgs p{};
  CHECK_MAP(map_a(&p.tmA, dout, d, 0, M, d));
  CHECK_MAP(map_b(&p.tmB, W2, d, 1, f, d));
  CHECK_MAP(map_f16_64(&p.tm_y, y, M, 2 * f, 2 * f));
  CHECK_MAP(map_bf16_64(&p.tm_dy, dyhat, M, 2 * f, 2 * f));
  p.r = r;
  p.spart = spart;
  p.ln = 1;
  p.w1 = w1;
  p.b1 = b1;
  p.spart_w = spart_w;
  p.spart_b = spart_b;
  p.M = M;
  p.N = f;
  p.K = d;
  return from_cuda(launch_swiglu_bwd(p, lc), "coda_gemm_ln_rowscale_swiglu_bwd launch");
}

coda_status_t coda_row_ln_bwd(const float* spart, const float* spart_w, const float* spart_b,
                              int nparts, int M, int d, float* s_a, float* s_b,
                              coda_stream_t stream) {
  CHECK_PTR(spart);
  CHECK_PTR(spart_w);
  CHECK_PTR(spart_b);
  CHECK_PTR(s_a);
  CHECK_PTR(s_b);
  CHECK(nparts > 0 && M > 0 && d > 0, "coda_row_ln_bwd: bad sizes");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  return from_cuda(launch_ln_bwd_stats(spart, spart_w, spart_b, nparts, M, 1.0f / (float)d, s_a,
                                       s_b, lc.stream),
                   "coda_row_ln_bwd launch");
}

coda_status_t coda_gemm_resid_ln_stats_bwd(const void* dyhat, const void* W1, const void* h,
                                           const void* gamma, const void* beta, const float* r,
                                           const float* mu, const float* s_a, const float* s_b,
                                           const void* dresid, void* dh, void* hhat,
                                           float* dgamma_part, float* dbeta_part, int M, int d,
                                           int two_f, coda_stream_t stream) {
  CHECK_PTR(dyhat);
  CHECK_PTR(W1);
  CHECK_PTR(h);
  CHECK_PTR(gamma);
  CHECK_PTR(beta);
  CHECK_PTR(r);
  CHECK_PTR(mu);
  CHECK_PTR(s_a);
  CHECK_PTR(s_b);
  CHECK_OPT_PTR(dresid);
  CHECK_PTR(dh);
  CHECK_OPT_PTR(hhat);
  CHECK_PTR(dgamma_part);
  CHECK_PTR(dbeta_part);
  CHECK(M > 0 && d > 0 && two_f > 0 && M < kMaxDim && d < kMaxDim && two_f < kMaxDim,
        "coda_gemm_resid_ln_stats_bwd: bad sizes");
  CHECK(d % 8 == 0 && two_f % 8 == 0,
        "coda_gemm_resid_ln_stats_bwd: d and two_f must be multiples of 8");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  NormBwdArgs p{};
  CHECK_MAP(map_a(&p.tmA, dyhat, two_f, 0, M, two_f));
  CHECK_MAP(map_b(&p.tmB, W1, two_f, 1, d, two_f));
  CHECK_MAP(map_bf16_32(&p.tm_dh, dh, M, d, d));
  p.h = static_cast<const bf16*>(h);
  p.dres = static_cast<const bf16*>(dresid);
  if (hhat) CHECK_MAP(map_bf16_32(&p.tm_hhat, hhat, M, d, d));
  else p.tm_hhat = p.tm_dh;  // unused
  p.gamma = static_cast<const bf16*>(gamma);
  p.beta = static_cast<const bf16*>(beta);
  p.r = r;
  p.s = s_b;
  p.sa = s_a;
  p.mu = mu;
  p.dgpart = dgamma_part;
  p.dbpart = dbeta_part;
  p.save_hhat = hhat != nullptr;
  p.ln = 1;
  p.M = M;
  p.N = d;
  p.K = two_f;
  return from_cuda(launch_norm_bwd(p, lc), "coda_gemm_resid_ln_stats_bwd launch");
}

coda_status_t coda_selftest_bounded_wait(int timeout_ms, coda_stream_t stream) {
  CHECK(timeout_ms > 0 && timeout_ms <= 10000, "coda_selftest_bounded_wait: timeout 1..10000 ms");
  TRY_CTX(reinterpret_cast<cudaStream_t>(stream), lc);
  cudaError_t e = launch_bounded_wait_probe(lc.err, (unsigned long long)timeout_ms * 1000000ull,
                                            lc.stream);
  if (e != cudaSuccess) return from_cuda(e, "bounded-wait probe launch");
  return coda_get_device_error(stream);
}

}  // extern "C"
