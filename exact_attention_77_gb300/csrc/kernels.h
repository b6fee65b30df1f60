// Launch interface between the C-ABI host code and the kernel translation
// units.  Host-only declarations; no device code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

struct DeviceStatus;

// Mask of the masked forward / backward (attn_fwd_masked, attn_bwd_masked):
// query i sees key j when i - left <= j <= i + right (left / right < 0:
// unbounded), j < N, and block[i / 128 * n_tiles + j / 128] != 0 (block may
// be null: all ones).
struct MaskSpec {
  int left, right;
  const uint8_t* block;  // device [n_tiles, n_tiles] or null
  int n_tiles;
  int N;
};

struct FwdParams {
  CUtensorMap tm_q;  // [BH, N, d_qk] bf16, box 64 x 128 x 1, 128-byte swizzle
  CUtensorMap tm_k;  // [BH, N, d_qk]
  CUtensorMap tm_v;  // [BH, N, d_v]
  CUtensorMap tm_o;  // [BH, N, d_v] bf16 output, box 64 x 128 x 1 (the epilogue's TMA stores)
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
  // split-KV (attn_fwd_splitkv): keys from a sequence of Nk rows in n_splits
  // ranges of split_tiles 128-key tiles; partial outputs [n_splits, BH, N, d_v]
  // and LSEs [n_splits, BH, N], FP32
  int Nk;
  int n_kv_tiles;
  int n_splits;
  int split_tiles;
  float* o_part;
  float* lse_part;
  // FP8 forward (attn_fwd_fp8): e4m3 scales per (b, h, 128-row tile) of Q
  // and K, and per (b, h) of V
  const float* sq;
  const float* sk;
  const float* sv;
  float p_off;  // FP8: P is stored as e4m3(2^p_off P), p_off = 8 - tau
  MaskSpec mask;  // masked instances only
  // grouped-query attention: unit (b, h) reads K/V head b * h_kv + h / kv_group
  // (h < h_q query heads, h_kv = h_q / kv_group); kv_group = 1: one K/V head
  // per query head
  int h_q;
  int kv_group;
  float scale_log2;  // scale * log2(e)
  float tau;         // rescale threshold, log2 units
};

struct BwdParams {
  CUtensorMap tm_q;   // [BH, N, d_qk]
  CUtensorMap tm_k;   // [BH, N, d_qk]
  CUtensorMap tm_v;   // [BH, N, d_v]
  CUtensorMap tm_do;  // [BH, N, d_v]
  CUtensorMap tm_dk;  // [BH_kv, N, d_qk] bf16 output (the one-CTA kernels' TMA stores)
  CUtensorMap tm_dv;  // [BH_kv, N, d_v]
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
  MaskSpec mask;  // masked instances only
  // grouped-query instances: BH counts query heads; h_q query heads per batch
  // entry, kv_group of them per K/V head
  int h_q;
  int kv_group;
  int persist;  // 1: persistent CTAs (one per SM) over the (head, key tile) units
  // deterministic mode's unit order (det_unit in attn_bwd.cuh): key-tile-major
  // inside groups of det_group heads (1 .. K/V heads); det_desc = 1 takes the
  // key tiles from the last down (and each dQ tile adds them in that order)
  int det_group;
  int det_desc;
  // 1 (deterministic mode; chosen by the host): each dQ tile's first
  // contribution (ticket 0) is a plain bulk store, so the preprocess leaves
  // the FP32 accumulator unzeroed
  int acc_first_store;
  // atomic dQ, persistent kernel without the causal mask: when its last round
  // is partial, that round's tail_units units (from unit tail_first on) are
  // cut into tail_s pieces over the query tiles, one per CTA; the piece of CTA
  // b leaves FP32 dV / dK partials in slot b ([slot][2][128][d], dV then dK),
  // which the dQ conversion sums into dV and dK.  tail_cap slots fit (0: units
  // are never cut); tail_s <= 1: no cut (set by the persistent launch).
  float* tail_part;
  int tail_cap;
  int tail_s;
  int tail_first;
  int tail_units;
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
// Once per (kernel, device): raise the kernel's dynamic shared-memory limit
// to smem_bytes and check that it compiled to launch_regs registers per
// thread (the setmaxnreg split assumes it; cudaErrorInvalidConfiguration
// otherwise).  *sms (may be null) receives the device's multiprocessor count.
cudaError_t prepare_kernel(const void* kernel, int smem_bytes, int launch_regs, int* sms);

// nqt: query tiles per CTA (1 only for d_qk <= 128)
cudaError_t launch_fwd_split(const FwdParams& p, int d_qk, int nqt, cudaStream_t s);

// FP8 forward (d = 128, two query tiles per CTA) and the quantiser that
// prepares its inputs (attn_fp8.cu).
cudaError_t launch_fwd_fp8(const FwdParams& p, bool causal, cudaStream_t s);

// Masked forward / backward (p.mask), d = 64 or 128 (attn_masked.cu).
cudaError_t launch_fwd_masked(const FwdParams& p, int d, cudaStream_t s);
cudaError_t launch_bwd_masked(const BwdParams& p, int d, bool deterministic, cudaStream_t s, const LaunchEvents* ev);
// Grouped-query backward (p.kv_group > 1), d = 64 or 128 (attn_bwd_gqa.cu).
cudaError_t launch_bwd_gqa(const BwdParams& p, int d, bool causal, bool deterministic, cudaStream_t s,
                           const LaunchEvents* ev);
struct QuantParams {
  const void* q;
  const void* k;
  const void* v;
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* v8;
  float* sq;
  float* sk;
  float* sv;
  unsigned* vmax;     // [BH] scratch: bit patterns of max |V| per head
  uint32_t signs[4];  // bit i set: coordinate i of Q and K is negated before the Hadamard transform
  int BH, N, n_tiles;
};
cudaError_t launch_fp8_quantize(const QuantParams& p, cudaStream_t s);

// Merge of split partials: [n_parts, BH, N, d_v] FP32 outputs and [n_parts,
// BH, N] LSEs into bf16 O [BH, N, d_v] and FP32 LSE [BH, N].
// pdl: launch as a programmatic dependent of the previous kernel on s (the
// merge waits for that kernel's completion inside, griddepcontrol.wait).
cudaError_t launch_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int BH,
                         int N, int d_v, cudaStream_t s, bool pdl);

// Backward: preprocess, main, dQ conversion.
cudaError_t launch_bwd_d64(const BwdParams& p, bool causal, bool deterministic, cudaStream_t s, const LaunchEvents* ev);
cudaError_t launch_bwd_d128(const BwdParams& p, bool causal, bool deterministic, cudaStream_t s, const LaunchEvents* ev);
// d_qk = 192, d_v = 128 (attn_bwd_d192.cu); gqa: p.kv_group query heads share a K/V head.
cudaError_t launch_bwd_d192(const BwdParams& p, bool causal, bool deterministic, bool gqa, cudaStream_t s,
                            const LaunchEvents* ev);

// Probes of the exponential paths.
cudaError_t launch_exp2_probe(const float* x, float* out, int n, int method, cudaStream_t s);
cudaError_t launch_exp2_throughput(float* sink, int blocks, int iters, int method, cudaStream_t s);
cudaError_t launch_wait_selftest(DeviceStatus* status, unsigned long long timeout_ns, cudaStream_t s);

}  // namespace attn
