// attn_bwd_noalloc: the backward pass with its scratch memory built into the
// library, for callers that cannot allocate device memory themselves.
//
// Who needs this: code that runs where a cudaMalloc is not allowed or not
// wanted -- a host function or stream callback (which may not call into the
// CUDA API that allocates), a serving runtime that reserves its whole memory
// budget up front and forbids allocations on the request path, or a plugin
// whose host application owns every device buffer.  Such callers can pass
// their inputs and outputs but have no way to provide attn_bwd's workspace.
//
// How: the workspace lives in one file-scope __device__ array of
// ATTN_NOALLOC_SCRATCH_BYTES.  The CUDA runtime creates it on every GPU that
// loads this library and keeps it until the process exits.  Host code cannot
// use the array's name as a device address, so the first call on each device
// looks the address up with cudaGetSymbolAddress (with that device current)
// and caches it; make that first call before any stream capture.  Every call
// on a device shares the one array: calls whose kernels overlap on the GPU
// (different streams, no ordering between them) race on it.  The preprocess
// kernel clears the accumulator and tickets at the start of every call, so the
// previous call's contents do not leak into the result.
#include <cuda_runtime.h>
#include <stddef.h>

#include <mutex>

#include "attn.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_OK;
}

}  // namespace

namespace attn {
int bwd_on_scratch(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d_qk, int d_v, int causal, float scale,
                   int deterministic, void* scratch, size_t scratch_bytes, cudaStream_t stream);
}  // namespace attn

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d_qk,
                                int d_v, int causal, float scale, int deterministic, cudaStream_t stream) {
  const size_t need = attn_bwd_workspace_bytes(B, H, N, d_qk, d_v, deterministic);
  // need == 0: sizes the backward rejects, which it reports with the exact
  // error; a workspace larger than the array is an error unless all that does
  // not fit is the optional region for the persistent kernel's cut units
  void* scratch = nullptr;
  if (need != 0) {
    if (int st = noalloc_scratch(&scratch)) return st;
  }
  return attn::bwd_on_scratch(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d_qk, d_v, causal, scale, deterministic,
                              scratch, need != 0 ? (size_t)ATTN_NOALLOC_SCRATCH_BYTES : 0, stream);
}
