// LM head + cross-entropy for callers that may not allocate device memory.
//
// coda_lmhead_ce needs a scratch buffer for its per-tile (max, sum-exp)
// partials and target logits, which the caller allocates. Some callers
// cannot: a custom-operator hook of a host framework that is handed only its
// input and output buffers while that framework's allocator owns the rest of
// device memory, a process that reserved all device memory up front, or a
// latency-critical loop in which cudaMalloc / cudaFree (which may synchronise
// the device) are not allowed. This entry point gives them the same result
// with the scratch taken from a fixed array that the library itself holds in
// device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library keeps kNoAllocScratchBytes of it until the process exits. Host
// code may not pass the array's name to a kernel (on the host it is only a
// stand-in symbol); its device address on the current device is looked up
// with cudaGetSymbolAddress on every call. Nothing is kept between calls, so
// a cudaDeviceReset (after which the module is loaded again, possibly at
// another address) leaves no stale pointer behind. The first call on a
// device may load the library's module there; make it before any stream
// capture.
#include <cstdio>

#include "coda.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_lmhead_scratch[kNoAllocScratchBytes];

// Device address of g_lmhead_scratch on the current device. The lookup is a
// host-side query of the loaded module: no allocation, no stream operation.
coda_status_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_lmhead_scratch);
  if (e != cudaSuccess || p == nullptr) {
    char buf[256];
    snprintf(buf, sizeof(buf), "coda_lmhead_ce_noalloc: cudaGetSymbolAddress failed: %s",
             cudaGetErrorString(e));
    coda::set_last_error(buf);
    return CODA_ERR_LAUNCH;
  }
  *out = p;
  return CODA_OK;
}

}  // namespace

extern "C" size_t coda_lmhead_ce_noalloc_capacity(void) { return kNoAllocScratchBytes; }

extern "C" coda_status_t coda_lmhead_ce_noalloc(const void* hidden, const void* W,
                                                const int32_t* targets, float* lse, float* loss,
                                                int M, int V, int d, coda_stream_t stream) {
  // sizes first: an argument error is reported as one on any machine, before
  // the scratch lookup touches the device
  if (M <= 0 || V <= 0 || d <= 0) {
    coda::set_last_error("coda_lmhead_ce_noalloc: M, V and d must be positive");
    return CODA_ERR_INVALID_VALUE;
  }
  const size_t need = coda_lmhead_ce_workspace_size(M, V);
  if (need > kNoAllocScratchBytes) {
    char buf[320];
    snprintf(buf, sizeof(buf),
             "coda_lmhead_ce_noalloc: M=%d rows over V=%d classes need %zu bytes of scratch, "
             "more than the %zu bytes this variant holds; call it on fewer rows at a time or "
             "use coda_lmhead_ce with a caller-allocated workspace",
             M, V, need, kNoAllocScratchBytes);
    coda::set_last_error(buf);
    return CODA_ERR_INVALID_VALUE;
  }
  void* ws = nullptr;
  const coda_status_t s = scratch_address(&ws);
  if (s != CODA_OK) return s;
  // Every partial and every target logit the combine reads is written by this
  // call's GEMM first, so nothing left in the array by an earlier call is read
  // and nothing needs clearing.
  return coda_lmhead_ce(hidden, W, targets, lse, loss, ws, kNoAllocScratchBytes, M, V, d, stream);
}
