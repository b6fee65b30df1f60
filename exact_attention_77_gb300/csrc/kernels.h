// Launch interface between the C-ABI host code and the kernel translation
// units.  Host-only declarations; no device code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

struct DeviceStatus;

struct FwdParams {
  CUtensorMap tm_q;  // [BH, N, d_qk] bf16, box 64 x 128 x 1, 128-byte swizzle
  CUtensorMap tm_k;  // [BH, N, d_qk]
  CUtensorMap tm_v;  // [BH, N, d_v]
  void* o;           // bf16 [BH, N, d_v]
  float* lse;        // fp32 [BH, N]
  DeviceStatus* status;
  unsigned long long* rescale_counter;  // may be null
  unsigned long long timeout_ns;
  int N;
  int BH;
  int n_qtiles;  // ceil(N / 128)
  int n_blocks;  // work units: BH * ceil(n_qtiles / tiles per CTA)
  int max_ctas;  // persistent grid size (0: as many CTAs as fit)
  int persist;   // 1: persistent CTAs looping over units; 0: one CTA per unit
  float scale_log2;  // scale * log2(e)
  float tau;         // rescale threshold, log2 units
};

struct BwdParams {
  CUtensorMap tm_q;   // [BH, N, d_qk]
  CUtensorMap tm_k;   // [BH, N, d_qk]
  CUtensorMap tm_v;   // [BH, N, d_v]
  CUtensorMap tm_do;  // [BH, N, d_v]
  CUtensorMap tm_q_half;   // Q with 64-row boxes (CTA-pair backward)
  CUtensorMap tm_do_half;  // dO with 64-row boxes (CTA-pair backward)
  const void* o;      // bf16 [BH, N, d_v]
  const void* dO;     // bf16 [BH, N, d_v]
  const float* lse;   // fp32 [BH, N]
  void* dq;           // bf16 [BH, N, d_qk]
  void* dk;           // bf16 [BH, N, d_qk]
  void* dv;           // bf16 [BH, N, d_v]
  float* row_lse2;    // workspace fp32 [BH, Npad]: -LSE * log2(e), -inf on padding rows
  float* row_d;       // workspace fp32 [BH, Npad]: -rowsum(dO * O), 0 on padding rows
  float* dq_acc;      // workspace fp32 [BH, n_tiles, d_qk/4, 128, 4]; [BH, n_tiles, 2, d_qk/4, 64, 4] when pair_mode
  int* tickets;       // workspace int32 [BH, n_tiles] (deterministic mode)
  DeviceStatus* status;
  unsigned long long timeout_ns;
  int N;
  int Npad;      // n_tiles * 128
  int BH;
  int n_tiles;   // ceil(N / 128)
  float scale;
  float scale_log2;
  int pair_mode;  // 1: CTA-pair main kernel (d = 128) and its accumulator layout
};

// Optional events recorded on the launch stream around each backward kernel:
// ev[0] before the preprocess, ev[1] between preprocess and main, ev[2]
// between main and dQ conversion, ev[3] after it.  Null entries are skipped.
struct LaunchEvents {
  cudaEvent_t ev[4];
};

// Forward (one kernel): per head-dim translation unit.
cudaError_t launch_fwd_d64(const FwdParams& p, bool causal, int nqt, int poly, cudaStream_t s);
cudaError_t launch_fwd_d128(const FwdParams& p, bool causal, int nqt, int poly, cudaStream_t s);
cudaError_t launch_fwd_d192(const FwdParams& p, bool causal, int nqt, int poly, cudaStream_t s);

// Backward: preprocess, main, dQ conversion.
cudaError_t launch_bwd_d64(const BwdParams& p, bool causal, bool deterministic, cudaStream_t s, const LaunchEvents* ev);
cudaError_t launch_bwd_d128(const BwdParams& p, bool causal, bool deterministic, cudaStream_t s, const LaunchEvents* ev);

// Probes of the exponential paths.
cudaError_t launch_exp2_probe(const float* x, float* out, int n, int method, cudaStream_t s);
cudaError_t launch_exp2_throughput(float* sink, int blocks, int iters, int method, cudaStream_t s);
cudaError_t launch_wait_selftest(DeviceStatus* status, unsigned long long timeout_ns, cudaStream_t s);

}  // namespace attn
