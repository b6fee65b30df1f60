// C ABI of the library: argument checks, TMA descriptors, workspace layout,
// kernel selection and launch, and the device status word.  No device
// allocation happens here; the caller owns every buffer.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "attn.h"
#include "det_order.h"
#include "kernels.h"
#include "sm103.cuh"

__device__ attn::DeviceStatus g_attn_status;

namespace {

constexpr int kMaxDevices = 64;

struct Settings {
  unsigned long long timeout_ns = 5ull * 1000 * 1000 * 1000;
  int fwd_tiles = 2;  // query tiles per forward CTA (d = 64 / 128)
  int fwd_poly = 0;   // 1: a share of the exponentials on the FMA-pipe polynomial
  int fwd_max_ctas = 0;  // persistent forward grid size (0: one CTA per free SM slot)
  int fwd_persist = -1;  // -1: by sequence length; 0 / 1 forces
  int bwd_pair = 0;      // 1: d = 128 backward on CTA pairs
  int bwd_persist = -1;  // -1: by sequence length; 0 / 1 forces persistent backward CTAs
  int det_group = 0;     // deterministic backward: heads per group of the unit order (0: all heads)
  int det_desc = 0;      // deterministic backward: 1 = key tiles from the last down
  int merge_pdl = 1;     // 1: split-KV merge as a programmatic dependent launch
  float fp8_tau = 4.f;   // FP8 forward: rescale threshold (P stored as e4m3(2^(8 - tau) P))
  float tau = 8.0f;
  unsigned long long* rescale_counter = nullptr;
};

std::mutex g_mu;
Settings g_settings;
bool g_env_read = false;
attn::DeviceStatus* g_status_ptr[kMaxDevices] = {nullptr};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Events recorded while profiling: kind 0 = forward, 1..3 = backward pieces,
// 4 / 5 = split-KV forward / merge.
struct ProfileRecord {
  int kind;
  cudaEvent_t a, b;
};
bool g_profiling = false;
std::vector<ProfileRecord> g_records;

bool profiling() {
  std::lock_guard<std::mutex> lock(g_mu);
  return g_profiling;
}

void add_record(int kind, cudaEvent_t a, cudaEvent_t b) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_records.push_back({kind, a, b});
}

Settings settings() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_env_read) {
    g_env_read = true;
    if (const char* e = getenv("ATTN_TIMEOUT_MS")) {
      const long ms = atol(e);
      if (ms > 0) g_settings.timeout_ns = (unsigned long long)ms * 1000000ull;
    }
    if (const char* e = getenv("ATTN_FWD_TILES")) {
      const int v = atoi(e);
      if (v == 1 || v == 2) g_settings.fwd_tiles = v;
    }
    if (const char* e = getenv("ATTN_EXP_POLY")) g_settings.fwd_poly = atoi(e) != 0;
    if (const char* e = getenv("ATTN_FWD_MAX_CTAS")) g_settings.fwd_max_ctas = atoi(e);
    if (const char* e = getenv("ATTN_FWD_PERSIST")) g_settings.fwd_persist = atoi(e);
    if (const char* e = getenv("ATTN_BWD_PAIR")) g_settings.bwd_pair = atoi(e) != 0;
    if (const char* e = getenv("ATTN_BWD_PERSIST")) g_settings.bwd_persist = atoi(e);
    if (const char* e = getenv("ATTN_MERGE_PDL")) g_settings.merge_pdl = atoi(e) != 0;
    if (const char* e = getenv("ATTN_DET_GROUP")) {
      const int v = atoi(e);
      if (v >= 0) g_settings.det_group = v;
    }
    if (const char* e = getenv("ATTN_DET_DESC")) g_settings.det_desc = atoi(e) != 0;
    if (const char* e = getenv("ATTN_FP8_TAU")) {
      const int v = atoi(e);
      if (v >= 0 && v <= 8) g_settings.fp8_tau = (float)v;
    }
  }
  return g_settings;
}

// Device status word of the current device (resolved once per device).
int status_ptr(attn::DeviceStatus** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_status) != cudaSuccess) return ATTN_ERR_CUDA;
    g_status_ptr[dev] = static_cast<attn::DeviceStatus*>(p);
  }
  *out = g_status_ptr[dev];
  return ATTN_OK;
}

int encoder(EncodeTiledFn* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = g_encode;
  return ATTN_OK;
}

// 3-D view [BH, N, d] of a contiguous tensor of bf16 (elem_bytes 2) or of
// 8-bit codes (elem_bytes 1); box 128 bytes of d x box_rows rows x 1 with the
// 128-byte swizzle; rows past N read as zero.
// Encoded descriptors are kept in a small cache keyed by every input of the
// encoding (a descriptor holds only the address and the shape, so a reused
// address with the same shape gets an identical descriptor).
struct MapKey {
  const void* ptr;
  int BH, N, d, box_rows, elem_bytes;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && BH == o.BH && N == o.N && d == o.d && box_rows == o.box_rows && elem_bytes == o.elem_bytes;
  }
};
constexpr int kMapCache = 64;
struct MapCache {
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int used = 0, next = 0;
};
MapCache g_maps;

int make_map_uncached(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows, int elem_bytes);

int make_map(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows = 128, int elem_bytes = 2) {
  const MapKey k{ptr, BH, N, d, box_rows, elem_bytes};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_maps.used; ++i)
      if (g_maps.key[i] == k) {
        *map = g_maps.map[i];
        return ATTN_OK;
      }
  }
  if (int st = make_map_uncached(map, ptr, BH, N, d, box_rows, elem_bytes)) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  const int slot = g_maps.used < kMapCache ? g_maps.used++ : (g_maps.next++ % kMapCache);
  g_maps.key[slot] = k;
  g_maps.map[slot] = *map;
  return ATTN_OK;
}

int make_map_uncached(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows, int elem_bytes) {
  EncodeTiledFn enc;
  if (int st = encoder(&enc)) return st;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * elem_bytes, (cuuint64_t)N * d * elem_bytes};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = enc(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int H, int N, float scale, int causal) {
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * H >= (1ll << 31) || N >= (1 << 24)) return ATTN_ERR_INVALID_ARG;
  // the running max is taken as max(S) * scale, and hidden scores are -inf
  // before the scale is applied: the scale must be positive
  if (!isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

bool fwd_dims_ok(int d_qk, int d_v) {
  return (d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128) || (d_qk == 192 && d_v == 128);
}

bool bwd_dims_ok(int d_qk, int d_v) {
  return (d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128) || (d_qk == 192 && d_v == 128);
}
// masked forward and backward: one head dim for Q, K and V
bool masked_dims_ok(int d_qk, int d_v) { return (d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128); }

struct WorkspaceLayout {
  size_t lse2, d, acc, tickets, base;  // base: end of what every backward needs
  size_t tail_part, total;  // the persistent kernel's cut units (atomic, d <= 128)
  int tail_cap;             // pieces the tail region holds
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Pieces the persistent backward may cut its last round's units into: at most
// one per CTA, and it runs one CTA per SM (152 on GB300), only when there are
// more units than CTAs.
constexpr int kMaxTailPieces = 160;

WorkspaceLayout workspace_layout(int B, int H, int N, int d_qk, int deterministic) {
  WorkspaceLayout w;
  const size_t bh = (size_t)B * H;
  const size_t tiles = ((size_t)N + 127) / 128;
  const size_t npad = tiles * 128;
  w.lse2 = 0;
  w.d = round_up(w.lse2 + bh * npad * 4, 256);
  w.acc = round_up(w.d + bh * npad * 4, 256);
  w.tickets = round_up(w.acc + bh * npad * (size_t)d_qk * 4, 256);
  w.base = round_up(w.tickets + (deterministic ? bh * tiles * 4 : 0), 256);
  // FP32 dV and dK partials of 128 rows x d per piece
  const size_t units = bh * tiles;
  w.tail_cap = (!deterministic && d_qk <= 128 && units > 1)
                   ? (int)(units - 1 < (size_t)kMaxTailPieces ? units - 1 : (size_t)kMaxTailPieces)
                   : 0;
  w.tail_part = w.base;
  w.total = round_up(w.tail_part + (size_t)w.tail_cap * 2 * 128 * d_qk * 4, 256);
  return w;
}

// Split of N_k keys into whole 128-key tiles: n_splits requested parts of
// split_tiles tiles each (the last one ragged); no part is empty.
struct SplitGeom {
  int n_kv_tiles, split_tiles, n_splits;
};

SplitGeom split_geom(int N_k, int n_splits) {
  SplitGeom g;
  g.n_kv_tiles = (N_k + 127) / 128;
  const int req = n_splits < g.n_kv_tiles ? n_splits : g.n_kv_tiles;
  g.split_tiles = (g.n_kv_tiles + req - 1) / req;
  g.n_splits = (g.n_kv_tiles + g.split_tiles - 1) / g.split_tiles;
  return g;
}

struct SplitWorkspace {
  size_t lse, total;
};

SplitWorkspace split_workspace(int BH, int N_q, int d_v, int n_splits) {
  SplitWorkspace w;
  const size_t rows = (size_t)n_splits * BH * N_q;
  w.lse = round_up(rows * d_v * 4, 256);
  w.total = round_up(w.lse + rows * 4, 256);
  return w;
}

int check_split(int B, int H, int N_q, int N_k, int n_splits) {
  if (B < 1 || H < 1 || N_q < 1 || N_k < 1 || n_splits < 1) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * H >= (1ll << 31) || N_q >= (1 << 24) || N_k >= (1 << 24)) return ATTN_ERR_INVALID_ARG;
  const SplitGeom g = split_geom(N_k, n_splits);
  if ((long long)B * H * ((N_q + 127) / 128) * g.n_splits >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Query tiles per split-KV CTA: one 128-row tile when the queries fit in one
// (decode), which lets two CTAs share a multiprocessor; else two tiles share
// each K/V tile load.  d_qk = 192 has only the two-tile layout.
int split_nqt(int N_q, int d_qk) { return (N_q <= 128 && d_qk <= 128) ? 1 : 2; }
int split_ctas_per_sm(int nqt) { return nqt == 1 ? 2 : 1; }

}  // namespace

namespace attn {

cudaError_t prepare_kernel(const void* kernel, int smem_bytes, int launch_regs, int* sms) {
  struct Prepared {
    const void* kernel;
    int dev, sms;
  };
  static std::mutex mu;
  static std::vector<Prepared> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Prepared& d : done)
      if (d.kernel == kernel && d.dev == dev) {
        if (sms) *sms = d.sms;
        return cudaSuccess;
      }
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != launch_regs) return cudaErrorInvalidConfiguration;
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  done.push_back({kernel, dev, n});
  if (sms) *sms = n;
  return cudaSuccess;
}

}  // namespace attn

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_BOUNDS: return "ATTN_ERR_BOUNDS";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

int attn_set_rescale_counter(unsigned long long* counter) {
  settings();
  std::lock_guard<std::mutex> lock(g_mu);
  g_settings.rescale_counter = counter;
  return ATTN_OK;
}

int attn_set_bwd_pair(int enable) {
  if (enable != 0 && enable != 1) return ATTN_ERR_INVALID_ARG;
  settings();
  std::lock_guard<std::mutex> lock(g_mu);
  g_settings.bwd_pair = enable;
  return ATTN_OK;
}

int attn_set_fwd_persist(int mode) {
  if (mode < -1 || mode > 1) return ATTN_ERR_INVALID_ARG;
  settings();
  std::lock_guard<std::mutex> lock(g_mu);
  g_settings.fwd_persist = mode;
  return ATTN_OK;
}

int attn_set_bwd_persist(int mode) {
  if (mode < -1 || mode > 1) return ATTN_ERR_INVALID_ARG;
  settings();
  std::lock_guard<std::mutex> lock(g_mu);
  g_settings.bwd_persist = mode;
  return ATTN_OK;
}

int attn_set_det_schedule(int head_group, int descending) {
  if (head_group < 0 || (descending != 0 && descending != 1)) return ATTN_ERR_INVALID_ARG;
  settings();
  std::lock_guard<std::mutex> lock(g_mu);
  g_settings.det_group = head_group;
  g_settings.det_desc = descending;
  return ATTN_OK;
}

int attn_bwd_det_plan(int n_heads, int n_tiles, int n_ctas, int head_group, int descending, int causal, int rotated,
                      int* unit_head, int* unit_key_tile, int* unit_first_tile, int* rank) {
  if (n_heads < 1 || n_tiles < 1 || n_ctas < 1 || head_group < 1 || (descending != 0 && descending != 1) ||
      (causal != 0 && causal != 1) || (rotated != 0 && rotated != 1) || (rotated && causal) ||
      (long long)n_heads * n_tiles * n_tiles > (1ll << 28) || unit_head == nullptr || unit_key_tile == nullptr ||
      unit_first_tile == nullptr || rank == nullptr)
    return ATTN_ERR_INVALID_ARG;
  const int n = n_tiles;
  const int group = head_group < n_heads ? head_group : n_heads;
  for (int u = 0; u < n_heads * n; ++u) {
    const attn::DetUnit d = attn::det_unit_of(u, n_heads, n, group, descending);
    unit_head[u] = d.bh;
    unit_key_tile[u] = d.j;
    int* row = rank + (size_t)u * n;
    if (rotated) {
      const attn::DetRot r = attn::det_rot(u, n_ctas, n_heads, n, group, descending);
      unit_first_tile[u] = attn::det_rot_first(r.jj, n, r.sigma);
      for (int i = 0; i < n; ++i) row[i] = attn::det_rot_rank(i, r, n);
    } else {
      unit_first_tile[u] = n - 1;
      for (int i = 0; i < n; ++i) row[i] = (causal && i < d.j) ? -1 : attn::det_rank(i, d.j, n, causal != 0, descending);
    }
  }
  return ATTN_OK;
}

int attn_set_exp_poly(int enable) {
  if (enable != 0 && enable != 1) return ATTN_ERR_INVALID_ARG;
  settings();
  std::lock_guard<std::mutex> lock(g_mu);
  g_settings.fwd_poly = enable;
  return ATTN_OK;
}

int attn_set_rescale_threshold(float tau) {
  if (!isfinite(tau) || tau < 0.f || tau > 16.f) return ATTN_ERR_INVALID_ARG;
  settings();
  std::lock_guard<std::mutex> lock(g_mu);
  g_settings.tau = tau;
  return ATTN_OK;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d_qk,
             int d_v, int causal, float scale, cudaStream_t stream) {
  return attn_fwd_gqa(q, k, v, o, lse, B, H, H, N, d_qk, d_v, causal, scale, stream);
}

int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                 int d_qk, int d_v, int causal, float scale, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (int st = check_common(B, H, N, scale, causal)) return st;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (!fwd_dims_ok(d_qk, d_v)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  const Settings cfg = settings();
  attn::FwdParams p;
  memset(&p, 0, sizeof(p));
  const int BH = B * H;
  if (int st = make_map(&p.tm_q, q, BH, N, d_qk)) return st;
  if (int st = make_map(&p.tm_k, k, B * H_kv, N, d_qk)) return st;
  if (int st = make_map(&p.tm_v, v, B * H_kv, N, d_v)) return st;
  if (int st = make_map(&p.tm_o, o, BH, N, d_v)) return st;
  if (int st = status_ptr(&p.status)) return st;
  p.o = o;
  p.lse = lse;
  p.rescale_counter = cfg.rescale_counter;
  p.timeout_ns = cfg.timeout_ns;
  p.N = N;
  p.BH = BH;
  p.h_q = H;
  p.kv_group = H / H_kv;
  p.n_qtiles = (N + 127) / 128;
  const int nqt = d_qk == 192 ? 2 : cfg.fwd_tiles;
  p.n_blocks = BH * ((p.n_qtiles + nqt - 1) / nqt);
  p.max_ctas = cfg.fwd_max_ctas;
  // short units run persistent: N <= 2048 (at most 16 K/V tiles each), and
  // causal N <= 4096 (measured on GB300: non-causal N = 4096 is 3 % faster
  // with one CTA per unit, causal 1.5 % slower)
  p.persist = cfg.fwd_persist >= 0 ? cfg.fwd_persist : ((N <= 2048 || (causal && N <= 4096)) ? 1 : 0);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.tau = cfg.tau;
  cudaEvent_t ea = nullptr, eb = nullptr;
  if (profiling()) {
    if (cudaEventCreate(&ea) != cudaSuccess || cudaEventCreate(&eb) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaEventRecord(ea, stream);
  }
  cudaError_t e;
  if (d_qk == 64) e = attn::launch_fwd_d64(p, causal != 0, nqt, cfg.fwd_poly, stream);
  else if (d_qk == 128) e = attn::launch_fwd_d128(p, causal != 0, nqt, cfg.fwd_poly, stream);
  else e = attn::launch_fwd_d192(p, causal != 0, nqt, cfg.fwd_poly, stream);
  if (ea != nullptr) {
    cudaEventRecord(eb, stream);
    add_record(0, ea, eb);
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_splitkv_heuristic(int B, int H, int N_q, int N_k, int d_qk, int n_sms) {
  if (check_split(B, H, N_q, N_k, 1) != ATTN_OK || n_sms < 1 || !fwd_dims_ok(d_qk, d_qk == 192 ? 128 : d_qk))
    return 0;
  // units without a split: (b, h, block of nqt 128-row query tiles), and the
  // CTAs that run at once
  const int nqt = split_nqt(N_q, d_qk);
  const long long units = (long long)B * H * (((N_q + 127) / 128 + nqt - 1) / nqt);
  const long long slots = (long long)n_sms * split_ctas_per_sm(nqt);
  if (2 * units > slots) return 1;
  const int n_kv_tiles = (N_k + 127) / 128;
  // the largest power of two that keeps every part in one wave (a second,
  // partial wave costs as much as the first), each part at least two key
  // tiles long
  long long n = 1;
  while (2 * n * units <= slots) n *= 2;
  const int max_parts = n_kv_tiles / 2 > 1 ? n_kv_tiles / 2 : 1;
  if (n > max_parts) n = max_parts;
  return split_geom(N_k, (int)n).n_splits;
}

size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int N_q, int N_k, int d_v, int n_splits) {
  if (check_split(B, H, N_q, N_k, n_splits) != ATTN_OK || (d_v != 64 && d_v != 128)) return 0;
  return split_workspace(B * H, N_q, d_v, split_geom(N_k, n_splits).n_splits).total;
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N_q,
                     int N_k, int d_qk, int d_v, float scale, int n_splits, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (int st = check_split(B, H, N_q, N_k, n_splits)) return st;
  if (!isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!fwd_dims_ok(d_qk, d_v)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  const int BH = B * H;
  const SplitGeom g = split_geom(N_k, n_splits);
  const SplitWorkspace w = split_workspace(BH, N_q, d_v, g.n_splits);
  if (workspace == nullptr || workspace_bytes < w.total) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  const Settings cfg = settings();
  attn::FwdParams p;
  memset(&p, 0, sizeof(p));
  if (int st = make_map(&p.tm_q, q, BH, N_q, d_qk)) return st;
  if (int st = make_map(&p.tm_k, k, BH, N_k, d_qk)) return st;
  if (int st = make_map(&p.tm_v, v, BH, N_k, d_v)) return st;
  if (int st = status_ptr(&p.status)) return st;
  char* ws = static_cast<char*>(workspace);
  p.o_part = reinterpret_cast<float*>(ws);
  p.lse_part = reinterpret_cast<float*>(ws + w.lse);
  p.rescale_counter = cfg.rescale_counter;
  p.timeout_ns = cfg.timeout_ns;
  p.N = N_q;
  p.Nk = N_k;
  p.BH = BH;
  p.n_qtiles = (N_q + 127) / 128;
  p.n_kv_tiles = g.n_kv_tiles;
  p.n_splits = g.n_splits;
  p.split_tiles = g.split_tiles;
  const int nqt = split_nqt(N_q, d_qk);
  p.n_blocks = BH * ((p.n_qtiles + nqt - 1) / nqt) * g.n_splits;
  p.persist = 1;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.tau = cfg.tau;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  if (profiling()) {
    for (auto& x : ev)
      if (cudaEventCreate(&x) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaEventRecord(ev[0], stream);
  }
  cudaError_t e = attn::launch_fwd_split(p, d_qk, nqt, stream);
  if (ev[0] != nullptr) cudaEventRecord(ev[1], stream);
  // the merge is a programmatic dependent launch unless events sit between
  if (e == cudaSuccess)
    e = attn::launch_merge(p.o_part, p.lse_part, g.n_splits, o, lse, BH, N_q, d_v, stream,
                          cfg.merge_pdl && ev[0] == nullptr);
  if (ev[0] != nullptr) {
    cudaEventRecord(ev[2], stream);
    add_record(4, ev[0], ev[1]);
    add_record(5, ev[1], ev[2]);
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_fp8_quantize_workspace_bytes(int B, int H) {
  if (B < 1 || H < 1 || (long long)B * H >= (1ll << 31)) return 0;
  return round_up((size_t)B * H * 4, 256);
}

int attn_fp8_quantize(const void* q, const void* k, const void* v, const signed char* signs, void* q8, void* k8,
                      void* v8, float* sq, float* sk, float* sv, int B, int H, int N, int d, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !signs || !q8 || !k8 || !v8 || !sq || !sk || !sv) return ATTN_ERR_INVALID_ARG;
  if (int st = check_common(B, H, N, 1.0f, 0)) return st;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  const int n_tiles = (N + 127) / 128;
  if ((long long)B * H * n_tiles >= (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  attn::QuantParams p;
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < d; ++i) {
    if (signs[i] != 1 && signs[i] != -1) return ATTN_ERR_INVALID_ARG;
    if (signs[i] < 0) p.signs[i / 32] |= 1u << (i % 32);
  }
  const void* ptrs[] = {q, k, v, q8, k8, v8, sq, sk, sv};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return ATTN_ERR_MISALIGNED;
  if (workspace == nullptr || workspace_bytes < attn_fp8_quantize_workspace_bytes(B, H)) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  p.q = q;
  p.k = k;
  p.v = v;
  p.q8 = static_cast<uint8_t*>(q8);
  p.k8 = static_cast<uint8_t*>(k8);
  p.v8 = static_cast<uint8_t*>(v8);
  p.sq = sq;
  p.sk = sk;
  p.sv = sv;
  p.vmax = static_cast<unsigned*>(workspace);
  p.BH = B * H;
  p.N = N;
  p.n_tiles = n_tiles;
  return attn::launch_fp8_quantize(p, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* sq, const float* sk, const float* sv,
                 void* o, float* lse, int B, int H, int N, int d, int causal, float scale, cudaStream_t stream) {
  if (!q8 || !k8 || !v8 || !sq || !sk || !sv || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (int st = check_common(B, H, N, scale, causal)) return st;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  const void* ptrs[] = {q8, k8, v8, sq, sk, sv, o, lse};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return ATTN_ERR_MISALIGNED;
  const Settings cfg = settings();
  attn::FwdParams p;
  memset(&p, 0, sizeof(p));
  const int BH = B * H;
  if (int st = make_map(&p.tm_q, q8, BH, N, d, 128, 1)) return st;
  if (int st = make_map(&p.tm_k, k8, BH, N, d, 128, 1)) return st;
  if (int st = make_map(&p.tm_v, v8, BH, N, d, 128, 1)) return st;
  if (int st = make_map(&p.tm_o, o, BH, N, d)) return st;
  if (int st = status_ptr(&p.status)) return st;
  p.o = o;
  p.lse = lse;
  p.sq = sq;
  p.sk = sk;
  p.sv = sv;
  p.rescale_counter = cfg.rescale_counter;
  p.timeout_ns = cfg.timeout_ns;
  p.N = N;
  p.BH = BH;
  p.n_qtiles = (N + 127) / 128;
  p.n_blocks = BH * ((p.n_qtiles + 1) / 2);
  p.max_ctas = cfg.fwd_max_ctas;
  p.persist = cfg.fwd_persist >= 0 ? cfg.fwd_persist : (N <= 4096 ? 1 : 0);
  // the codes hold (x sqrt(d) R) / s: the scores carry a factor d
  p.scale_log2 = scale * 1.4426950408889634f / (float)d;
  // P (<= 2^tau against the stale max) is stored as e4m3(2^(8 - tau) P)
  p.tau = cfg.fp8_tau;
  p.p_off = 8.f - cfg.fp8_tau;
  cudaEvent_t ea = nullptr, eb = nullptr;
  if (profiling()) {
    if (cudaEventCreate(&ea) != cudaSuccess || cudaEventCreate(&eb) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaEventRecord(ea, stream);
  }
  const cudaError_t e = attn::launch_fwd_fp8(p, causal != 0, stream);
  if (ea != nullptr) {
    cudaEventRecord(eb, stream);
    add_record(0, ea, eb);
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd_splitkv_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
                         int N_q, int N_k, int d_qk, int d_v, float scale, int n_splits, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  if (H < 1 || H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  const long long rows = (long long)(H / H_kv) * N_q;
  if (N_q < 1 || rows >= (1 << 24)) return ATTN_ERR_INVALID_ARG;
  // the H / H_kv query heads of one K/V head are contiguous in [B, H, N_q, d]:
  // as split-KV over B * H_kv heads of (H / H_kv) * N_q query rows
  return attn_fwd_splitkv(q, k, v, o, lse, B, H_kv, (int)rows, N_k, d_qk, d_v, scale, n_splits, workspace,
                          workspace_bytes, stream);
}

int attn_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int BH, int N,
               int d_v, cudaStream_t stream) {
  if (!o_parts || !lse_parts || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (n_parts < 1 || BH < 1 || N < 1 || (long long)BH * N >= (1ll << 33)) return ATTN_ERR_INVALID_ARG;
  if (d_v != 64 && d_v != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  return attn::launch_merge(o_parts, lse_parts, n_parts, o, lse, BH, N, d_v, stream, false) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d_qk, int d_v, int deterministic) {
  if (check_common(B, H, N, 1.0f, 0) != ATTN_OK || !bwd_dims_ok(d_qk, d_v)) return 0;
  if (deterministic != 0 && deterministic != 1) return 0;
  return workspace_layout(B, H, N, d_qk, deterministic).total;
}

}  // extern "C"

namespace {

// attn_bwd and attn_bwd_masked (mask != null: the masked one-CTA instances).
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
             void* dk, void* dv, int B, int H, int H_kv, int N, int d_qk, int d_v, int causal, float scale,
             int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream,
             const attn::MaskSpec* mask, bool tail_optional = false) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (H_kv < 1 || H_kv > H || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (int st = check_common(B, H, N, scale, causal)) return st;
  if (deterministic != 0 && deterministic != 1) return ATTN_ERR_INVALID_ARG;
  if (!bwd_dims_ok(d_qk, d_v) || (mask != nullptr && !masked_dims_ok(d_qk, d_v))) return ATTN_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return ATTN_ERR_MISALIGNED;
  const WorkspaceLayout w = workspace_layout(B, H, N, d_qk, deterministic);
  if (workspace == nullptr || workspace_bytes < (tail_optional ? w.base : w.total)) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  const Settings cfg = settings();
  attn::BwdParams p;
  memset(&p, 0, sizeof(p));
  const int BH = B * H;
  const bool gqa = H_kv < H;
  if (int st = make_map(&p.tm_q, q, BH, N, d_qk)) return st;
  if (int st = make_map(&p.tm_k, k, B * H_kv, N, d_qk)) return st;
  if (int st = make_map(&p.tm_v, v, B * H_kv, N, d_v)) return st;
  if (int st = make_map(&p.tm_do, dO, BH, N, d_v)) return st;
  if (int st = make_map(&p.tm_dk, dk, B * H_kv, N, d_qk)) return st;
  if (int st = make_map(&p.tm_dv, dv, B * H_kv, N, d_v)) return st;
  p.h_q = H;
  p.kv_group = H / H_kv;
  // d = 128 runs the CTA-pair main kernel when enabled (attn_set_bwd_pair)
  p.pair_mode = (d_qk == 128 && cfg.bwd_pair && mask == nullptr && !gqa) ? 1 : 0;
  if (mask != nullptr) p.mask = *mask;
  // persistent CTAs (measured on GB300, H = 16, with their TMA epilogue):
  // with atomic dQ at every N (d = 128 without the causal mask +3.7 % at
  // N = 16384 and +3.5 % at 8192; with it +6 % at 16384 and +10-16 % at
  // 8192 .. 2048; d = 64 with it +9-16 %); with tickets for N <= 2048, where
  // its rotated walk beats the one-unit kernel's best order by 9-21 % (the
  // one-unit kernel is 8-9 % faster above).  d_qk = 64 and 128 have a
  // persistent kernel, without grouped-query heads or masks.
  p.persist = cfg.bwd_persist >= 0 ? cfg.bwd_persist : ((N <= 2048 || !deterministic) ? 1 : 0);
  {
    const int n_heads = B * H_kv;  // the units' heads (K/V heads)
    const bool persistent_kernel = p.persist && !p.pair_mode && d_qk <= 128 && mask == nullptr && !gqa;
    // measured on GB300 (H = 16, d = 128): the persistent kernel without the
    // causal mask (its rotated walk) is fastest with one-head groups for
    // N <= 2048 and one group of all heads above; the one-unit kernel
    // without a mask with 8-head groups for N > 2048 (1-4 % over one
    // all-head group); under the causal mask, and for short sequences on the
    // one-unit kernel, one group over all heads, longest key tiles first
    const int g = cfg.det_group > 0              ? cfg.det_group
                  : (persistent_kernel && !causal) ? (N <= 2048 ? 1 : n_heads)
                  : (causal || N <= 2048)           ? n_heads
                                                    : 8;
    p.det_group = g < n_heads ? g : n_heads;
    p.det_desc = mask != nullptr ? 0 : cfg.det_desc;
    // the first contribution (ticket 0) to each dQ tile as a plain store, the
    // accumulator left unzeroed: measured on GB300 with the causal mask at
    // d = 64 / 128, main kernel +1-4 % and call +2-7 % (N = 1024 .. 16384);
    // the kernels take it in their causal instances only (in the others the
    // branch alone cost the one-unit kernel 10 % at N = 16384), and the
    // d_qk = 192 kernel not at all (mixed).  (Every dQ tile has a first
    // contribution unless a mask map leaves it without any; grouped-query
    // heads and CTA pairs add as before.)
    p.acc_first_store = (deterministic && causal && d_qk <= 128 && mask == nullptr && !gqa && !p.pair_mode) ? 1 : 0;
  }
  if (p.pair_mode) {
    if (int st = make_map(&p.tm_q_half, q, BH, N, d_qk, 64)) return st;
    if (int st = make_map(&p.tm_do_half, dO, BH, N, d_v, 64)) return st;
  }
  if (int st = status_ptr(&p.status)) return st;
  char* ws = static_cast<char*>(workspace);
  p.o = o;
  p.dO = dO;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.row_lse2 = reinterpret_cast<float*>(ws + w.lse2);
  p.row_d = reinterpret_cast<float*>(ws + w.d);
  p.dq_acc = reinterpret_cast<float*>(ws + w.acc);
  p.tickets = deterministic ? reinterpret_cast<int*>(ws + w.tickets) : nullptr;
  if (w.tail_cap > 0 && workspace_bytes >= w.total) {
    p.tail_part = reinterpret_cast<float*>(ws + w.tail_part);
    p.tail_cap = w.tail_cap;
  }
  p.timeout_ns = cfg.timeout_ns;
  p.N = N;
  p.n_tiles = (N + 127) / 128;
  p.Npad = p.n_tiles * 128;
  p.BH = BH;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  attn::LaunchEvents evs{};
  const bool prof = profiling();
  if (prof)
    for (auto& ev : evs.ev)
      if (cudaEventCreate(&ev) != cudaSuccess) return ATTN_ERR_CUDA;
  cudaError_t e;
  if (mask != nullptr)
    e = attn::launch_bwd_masked(p, d_qk, deterministic != 0, stream, prof ? &evs : nullptr);
  else if (d_qk == 192)
    e = attn::launch_bwd_d192(p, causal != 0, deterministic != 0, gqa, stream, prof ? &evs : nullptr);
  else if (gqa)
    e = attn::launch_bwd_gqa(p, d_qk, causal != 0, deterministic != 0, stream, prof ? &evs : nullptr);
  else
    e = d_qk == 64 ? attn::launch_bwd_d64(p, causal != 0, deterministic != 0, stream, prof ? &evs : nullptr)
                   : attn::launch_bwd_d128(p, causal != 0, deterministic != 0, stream, prof ? &evs : nullptr);
  if (prof)
    for (int k = 0; k < 3; ++k) add_record(1 + k, evs.ev[k], evs.ev[k + 1]);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Mask of attn_fwd_masked / attn_bwd_masked from its arguments.
int make_mask(attn::MaskSpec* m, int N, int window_left, int window_right, const unsigned char* block_mask) {
  if (window_left < -1 || window_right < -1) return ATTN_ERR_INVALID_ARG;
  m->left = window_left;
  m->right = window_right;
  m->block = block_mask;
  m->n_tiles = (N + 127) / 128;
  m->N = N;
  return ATTN_OK;
}

}  // namespace

namespace attn {

// attn_bwd_noalloc's backward: attn_bwd on the library's fixed scratch array,
// which may be too small for the region of the persistent kernel's cut units
// only (its last round then runs whole units).
int bwd_on_scratch(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d_qk, int d_v, int causal, float scale,
                   int deterministic, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d_qk, d_v, causal, scale, deterministic, scratch,
                  scratch_bytes, stream, nullptr, true);
}

}  // namespace attn

extern "C" {

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int N, int d_qk, int d_v, int causal, float scale,
             int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d_qk, d_v, causal, scale, deterministic, workspace,
                  workspace_bytes, stream, nullptr);
}

int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d_qk, int d_v, int causal,
                 float scale, int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, H_kv, N, d_qk, d_v, causal, scale, deterministic, workspace,
                  workspace_bytes, stream, nullptr);
}

int attn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    void* dq, void* dk, void* dv, int B, int H, int N, int d_qk, int d_v, int window_left,
                    int window_right, const unsigned char* block_mask, float scale, int deterministic,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  attn::MaskSpec m;
  if (int st = check_common(B, H, N, scale, 0)) return st;
  if (int st = make_mask(&m, N, window_left, window_right, block_mask)) return st;
  if (block_mask != nullptr && !aligned16(block_mask)) return ATTN_ERR_MISALIGNED;
  return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d_qk, d_v, 0, scale, deterministic, workspace,
                  workspace_bytes, stream, &m);
}

int attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d_qk,
                    int d_v, int window_left, int window_right, const unsigned char* block_mask, float scale,
                    cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (int st = check_common(B, H, N, scale, 0)) return st;
  attn::FwdParams p;
  memset(&p, 0, sizeof(p));
  if (int st = make_mask(&p.mask, N, window_left, window_right, block_mask)) return st;
  if (!masked_dims_ok(d_qk, d_v)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  if (block_mask != nullptr && !aligned16(block_mask)) return ATTN_ERR_MISALIGNED;
  const Settings cfg = settings();
  const int BH = B * H;
  if (int st = make_map(&p.tm_q, q, BH, N, d_qk)) return st;
  if (int st = make_map(&p.tm_k, k, BH, N, d_qk)) return st;
  if (int st = make_map(&p.tm_v, v, BH, N, d_v)) return st;
  if (int st = make_map(&p.tm_o, o, BH, N, d_v)) return st;
  if (int st = status_ptr(&p.status)) return st;
  p.o = o;
  p.lse = lse;
  p.rescale_counter = cfg.rescale_counter;
  p.timeout_ns = cfg.timeout_ns;
  p.N = N;
  p.BH = BH;
  p.n_qtiles = (N + 127) / 128;
  p.n_blocks = BH * p.n_qtiles;  // one query tile per CTA
  p.max_ctas = cfg.fwd_max_ctas;
  // persistent CTAs when units are short: short sequences, or a window that
  // bounds every query tile to at most 32 key tiles
  const bool short_window = window_left >= 0 && window_right >= 0 &&
                            (long long)window_left + window_right <= 30ll * 128;
  p.persist = cfg.fwd_persist >= 0 ? cfg.fwd_persist : ((N <= 4096 || short_window) ? 1 : 0);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.tau = cfg.tau;
  cudaEvent_t ea = nullptr, eb = nullptr;
  if (profiling()) {
    if (cudaEventCreate(&ea) != cudaSuccess || cudaEventCreate(&eb) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaEventRecord(ea, stream);
  }
  const cudaError_t e = attn::launch_fwd_masked(p, d_qk, stream);
  if (ea != nullptr) {
    cudaEventRecord(eb, stream);
    add_record(0, ea, eb);
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_get_device_status(cudaStream_t stream, int* where) {
  if (where) *where = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  attn::DeviceStatus* dev_status;
  if (int st = status_ptr(&dev_status)) return st;
  attn::DeviceStatus host{0, 0};
  if (cudaMemcpy(&host, dev_status, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (host.code != 0) {
    const attn::DeviceStatus zero{0, 0};
    if (cudaMemcpy(dev_status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (where) *where = host.where;
  return host.code;
}

int attn_exp2_probe(const float* x, float* out, int n, int method, cudaStream_t stream) {
  if (!x || !out || n < 0) return ATTN_ERR_INVALID_ARG;
  if (method != 0 && method != 3 && method != 4 && method != 5) return ATTN_ERR_INVALID_ARG;
  if (n == 0) return ATTN_OK;
  return attn::launch_exp2_probe(x, out, n, method, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_exp2_throughput(float* sink, int blocks, int iters, int method, cudaStream_t stream) {
  if (!sink || blocks < 1 || iters < 1) return ATTN_ERR_INVALID_ARG;
  if (method != 0 && method != 3 && method != 4 && method != 5) return ATTN_ERR_INVALID_ARG;
  return attn::launch_exp2_throughput(sink, blocks, iters, method, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_profile_start(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_profiling = true;
  return ATTN_OK;
}

int attn_profile_stop(attn_kernel_times_t* out) {
  if (out == nullptr) return ATTN_ERR_INVALID_ARG;
  std::vector<ProfileRecord> recs;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_profiling) return ATTN_ERR_INVALID_ARG;
    g_profiling = false;
    recs.swap(g_records);
  }
  memset(out, 0, sizeof(*out));
  int st = ATTN_OK;
  // the backward's four events are shared by its three records: destroy each once
  std::vector<cudaEvent_t> to_free;
  for (const ProfileRecord& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      st = ATTN_ERR_CUDA;
    switch (r.kind) {
      case 0: out->launches_fwd++; out->ms_fwd += ms; break;
      case 1: out->launches_bwd_pre++; out->ms_bwd_pre += ms; break;
      case 2: out->launches_bwd_main++; out->ms_bwd_main += ms; break;
      case 3: out->launches_bwd_convert++; out->ms_bwd_convert += ms; break;
      case 4: out->launches_fwd_split++; out->ms_fwd_split += ms; break;
      default: out->launches_merge++; out->ms_merge += ms; break;
    }
    to_free.push_back(r.a);
    if (r.kind == 0 || r.kind == 3 || r.kind == 5) to_free.push_back(r.b);
  }
  for (cudaEvent_t e : to_free) cudaEventDestroy(e);
  return st;
}

int attn_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream) {
  if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return ATTN_ERR_INVALID_ARG;
  attn::DeviceStatus* st;
  if (int e = status_ptr(&st)) return e;
  return attn::launch_wait_selftest(st, (unsigned long long)timeout_us * 1000ull, stream) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

}  // extern "C"
