// Backward attention kernels for sm_103a (templates; instantiated per head dim
// in attn_bwd_d*.cu).
//
// What they compute: dQ, dK, dV of L = sum(O * dO) for O = softmax(S) V,
// S = scale Q K^T (+ causal mask).  With P recomputed from the saved LSE,
// D_i = dO_i . O_i and dS = P o (dP - D), dP = dO V^T:
//     dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
// "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
// Hardware Scaling", Figure 2 and Table 3, describe this graph of five
// products and two elementwise steps; the abstract and Figures 7-8 the atomic
// and the deterministic accumulation of dQ.
//
// Kernels:
//   bwd_pre_kernel   -D_i = -rowsum(dO o O) and -LSE_i * log2(e) into the
//                    workspace (negated so the main kernel adds them; padding
//                    rows: 0 and -inf, so P = 0 there);
//                    zeroes the FP32 dQ accumulator and the tickets.
//   bwd_kernel       one CTA per (b, h, 128-key tile j), K_j and V_j resident;
//                    for each query tile i it runs, with keys on the tensor-
//                    memory lanes:
//                      S^T  = K_j Q_i^T          (SS)
//                      dP^T = V_j dO_i^T         (SS)
//                      P^T  = 2^(S^T*scale*log2e - LSE2_i), dS^T = P^T o (dP^T - D_i)
//                      dV  += P^T dO_i           (TS, P^T bf16 in tensor memory)
//                      dK  += dS^T Q_i           (TS, dS^T bf16 in tensor memory)
//                      dQ_i = dS K_j             (SS, dS bf16 in shared memory)
//                    and adds dQ_i into the FP32 accumulator with bulk
//                    reduce-add copies from a shared-memory staging tile
//                    (atomic mode), or with the same copies in ascending-j
//                    order behind a per-(b, h, i) ticket (deterministic mode).
//   dq_convert_kernel  dQ = scale * accumulator, as bf16 [B,H,N,d]; and the
//                    dV / dK rows of units the persistent kernel cut into
//                    pieces: the pieces' FP32 partials summed in piece order.
//
// Warp roles in bwd_kernel (512 threads): warp 0 producer (TMA), warp 1 MMA
// issuer and tensor-memory owner, warps 4-7 and 8-11 two compute warpgroups
// that split each tile's query columns for the elementwise step (one key row
// per thread), warps 12-15 the dQ warpgroup (one query row per thread) that
// reads dQ out of tensor memory and stages it for the copy engine's
// reduce-add, off the critical path.
#pragma once

#include <type_traits>

#include "attn_mask.cuh"
#include "det_order.h"
#include "kernels.h"
#include "sm103.cuh"

namespace attn {

constexpr int kBTile = 128;
constexpr int kBSub = 128 * 128;  // 128 rows x 128 bytes

template <int D>
struct BwdLayout {
  static constexpr int kTileBytes = kBTile * D * 2;  // one bf16 [128, D] tile
  // Q_i (with its -LSE2 / -D vectors) is double-buffered: the S^T product of
  // the next tile must not wait for its load.  dO_i is double-buffered at
  // d = 64; at d = 128 it has one stage (released right after the dV product)
  // so that 32 KiB stays free for the dQ staging tile.
  static constexpr int kQStages = 2;
  static constexpr int kDOStages = D == 64 ? 2 : 1;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;
  static constexpr int kDOOff = kQOff + kQStages * kTileBytes;
  static constexpr int kDSOff = kDOOff + kDOStages * kTileBytes;  // dS (bf16 128x128), MN-major for the dQ product
  static constexpr int kDSBytes = kBTile * kBTile * 2;
  // dQ_i FP32 staging in the accumulator's [D/4][128][4] order: 32 KiB, a
  // ring of two 16 KiB slots through which a tile goes in kRounds rounds
  // (round r in slot r % 2), so that one round is staged while the copy
  // engine reads the other
  static constexpr int kStgOff = kDSOff + kDSBytes;
  static constexpr int kStgBytes = 32 * 1024;
  static constexpr int kSlotBytes = kStgBytes / 2;
  static constexpr int kRounds = kBTile * D * 4 / kSlotBytes;
  static_assert(kRounds % 2 == 0, "every tile starts at slot 0");
  static constexpr int kVecOff = kStgOff + kStgBytes;  // per Q stage: -LSE2[128], -D[128] fp32
  static constexpr int kVecBytes = 2 * kBTile * 4;
  static constexpr int kBarOff = kVecOff + kQStages * kVecBytes;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;  // + stage
  static constexpr int kBarQEmpty = kBarQFull + kQStages;
  static constexpr int kBarDOFull = kBarQEmpty + kQStages;
  static constexpr int kBarDOEmpty = kBarDOFull + kDOStages;
  static constexpr int kBarSFull = kBarDOEmpty + kDOStages;  // S^T in tensor memory (commit)
  static constexpr int kBarDPFull = kBarSFull + 1;            // dP^T in tensor memory (commit)
  // + half m: P^T of queries 64h+32m .. 64h+32m+31 of both warpgroups h
  // written (256 arrivals); the dV product starts on the first half
  static constexpr int kBarPReady = kBarDPFull + 1;
  static constexpr int kBarDSFull = kBarPReady + 2;  // + half m: dS^T and dS, the same way
  static constexpr int kBarDQFull = kBarDSFull + 2;
  static constexpr int kBarDQFree = kBarDQFull + 1;
  static constexpr int kBarAccDone = kBarDQFree + 1;
  // Deterministic mode: + 2 w + s: staging slot s holds a round of reducer
  // warp w's tile (tiles alternate between two reducers; 4 dQ-warp
  // arrivals); + s: slot s has been read by the copy engine (1 arrival).
  static constexpr int kBarStgFull = kBarAccDone + 1;
  static constexpr int kBarStgFree = kBarStgFull + 4;
  static constexpr int kNumBars = kBarStgFree + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  // tensor memory columns
  // S^T fp32 [128 keys x 128 queries]; warpgroup h packs P^T (bf16) for its
  // queries 64h .. 64h+63 into columns 64h .. 64h+31, inside the columns it read
  static constexpr int kColS = 0;
  static constexpr int kColDP = 128;   // dP^T fp32; dS^T bf16 packed the same way
  static constexpr int kColDV = 256;   // dV accumulator [128 x D]
  static constexpr int kColDK = 256 + D;
  // dQ: its own columns at d = 64; at d = 128 it shares the dP^T columns, so
  // the next tile's S^T can start right after the dQ product and only dP^T
  // waits for the dQ read-out
  static constexpr int kColDQ = D == 64 ? 384 : 128;
  // 16 warps in four warpgroups: control (producer, MMA issuer), two compute
  // warpgroups, one dQ warpgroup.  setmaxnreg split of the 128 registers a
  // thread gets at launch: 112 * 128 + 128 * 256 + 144 * 128 <= 128 * 512.
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128;
  static constexpr int kCtlRegs = 112;
  static constexpr int kComputeRegs = 128;
  static constexpr int kDqRegs = 144;
  static_assert(kCtlRegs * 128 + kComputeRegs * 256 + kDqRegs * 128 <= kLaunchRegs * kThreads, "register split");
};

enum : int {
  kBWhereProd = 110, kBWhereMma = 120, kBWhereEw = 130, kBWhereDq = 140, kBWhereTicket = 141, kBWhereFin = 150
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Deterministic mode's unit order and ticket ranks: det_order.h.
__device__ __forceinline__ void det_unit(int u, int n_heads, int n, int group, int desc, int& j, int& bh) {
  const DetUnit d = det_unit_of(u, n_heads, n, group, desc);
  j = d.j;
  bh = d.bh;
}

// -------------------------------------------------------------- preprocess
// One group of D/8 lanes per row, 16-byte loads.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(BwdParams p) {
  constexpr int kLanes = D / 8;
  constexpr int kRowsPerBlock = 256 / kLanes;
  const int sub = threadIdx.x % kLanes;
  const long row = (long)blockIdx.x * kRowsPerBlock + threadIdx.x / kLanes;  // over BH * Npad
  const long total_rows = (long)p.BH * p.Npad;
  const bool in_range = row < total_rows;
  const int bh = in_range ? (int)(row / p.Npad) : 0;
  const int i = in_range ? (int)(row - (long)bh * p.Npad) : p.N;
  float acc = 0.f;
  if (i < p.N) {
    const size_t off = ((size_t)bh * p.N + i) * D + sub * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.dO) + off);
    const uint4 b = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.o) + off);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 fa = __bfloat1622float2(a2[k]);
      const float2 fb = __bfloat1622float2(b2[k]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, kLanes);
  if (in_range && sub == 0) {
    p.row_d[row] = -acc;
    p.row_lse2[row] = i < p.N ? -p.lse[(size_t)bh * p.N + i] * 1.4426950408889634f : -INFINITY;
  }
  // zero the dQ accumulator (unless each tile's first contribution is a
  // store) and the tickets (grid-stride, 16-byte stores)
  const size_t n4 = p.acc_first_store ? 0 : (size_t)p.BH * p.Npad * D / 4;
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n4; k += (size_t)gridDim.x * blockDim.x)
    acc4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.tickets != nullptr)
    for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < (size_t)p.BH * p.n_tiles;
         k += (size_t)gridDim.x * blockDim.x)
      p.tickets[k] = 0;  // one ticket per (bh, query tile)
}

// ---------------------------------------------------------------- dQ out
// Accumulator layout per (bh, tile): [D/4 groups][128 rows][4] (pair mode:
// [2 row halves][D/4][64][4]).  A thread takes one row and four consecutive
// groups; a warp takes 32 consecutive rows of the same groups, so each of
// its loads reads 512 contiguous bytes and each thread writes 32 contiguous
// bytes of its dQ row (one whole sector).
// Blocks past the dQ ones (dq_convert_blocks) finish the units the
// persistent kernel cut: one thread per (unit, tensor, key row, 8 columns),
// a warp on two rows of one tensor, reading the pieces' FP32 partials (slots
// of consecutive CTAs) and writing 16 bytes of bf16.  Those units are
// head-major like the persistent kernel's (unit u: head u / n_tiles, key tile
// u mod n_tiles).
template <int D>
__host__ __device__ __forceinline__ long dq_convert_blocks(const BwdParams& p) {
  return ((long)p.BH * p.n_tiles * 128 * (D / 16) + 255) / 256;
}

template <int D>
inline long tail_sum_blocks(const BwdParams& p) {
  return p.tail_s > 1 ? ((long)p.tail_units * 2 * 128 * (D / 8) + 255) / 256 : 0;
}

template <int D>
__device__ __forceinline__ void tail_sum(const BwdParams& p, long y) {
  constexpr int kChunks = D / 8;
  if (y >= (long)p.tail_units * 2 * 128 * kChunks) return;
  const int c8 = (int)(y % kChunks);
  const int row = (int)((y / kChunks) % 128);
  const int pass = (int)((y / (kChunks * 128)) % 2);  // 0: dV, 1: dK
  const int q = (int)(y / (kChunks * 128 * 2));       // cut unit
  const int u = p.tail_first + q;
  const int bh = u / p.n_tiles, j = u - bh * p.n_tiles;
  const int k_glob = j * 128 + row;
  if (k_glob >= p.N) return;
  constexpr size_t kSlot = 2 * (size_t)128 * D;
  const float* src = p.tail_part + (size_t)q * p.tail_s * kSlot + (size_t)(pass * 128 + row) * D + c8 * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int k = 0; k < p.tail_s; ++k) {
    const float4 a = *reinterpret_cast<const float4*>(src + (size_t)k * kSlot);
    const float4 b = *reinterpret_cast<const float4*>(src + (size_t)k * kSlot + 4);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  const float mul = pass == 0 ? 1.f : p.scale;
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(pass == 0 ? p.dv : p.dk) +
                                        ((size_t)bh * p.N + k_glob) * D + c8 * 8);
  *dst = make_uint4(pack_bf16(acc[0] * mul, acc[1] * mul), pack_bf16(acc[2] * mul, acc[3] * mul),
                    pack_bf16(acc[4] * mul, acc[5] * mul), pack_bf16(acc[6] * mul, acc[7] * mul));
}

template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(BwdParams p) {
  constexpr int kGroups = D / 4;    // 32 or 16
  constexpr int kQuads = kGroups / 4;  // threads per row
  const long nb = dq_convert_blocks<D>(p);
  if ((long)blockIdx.x >= nb) {
    tail_sum<D>(p, ((long)blockIdx.x - nb) * blockDim.x + threadIdx.x);
    return;
  }
  const long x = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long per_tile = 128L * kQuads;
  const long tile_g = x / per_tile;  // over BH * n_tiles
  if (tile_g >= (long)p.BH * p.n_tiles) return;
  const int tt = (int)(x - tile_g * per_tile);
  const int w = tt >> 5;
  const int r = (w & 3) * 32 + (threadIdx.x & 31);
  const int q = w >> 2;
  const int bh = (int)(tile_g / p.n_tiles);
  const int tile = (int)(tile_g - (long)bh * p.n_tiles);
  const int i = tile * 128 + r;
  float4 a[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int g = 4 * q + k;
    const size_t idx = p.pair_mode ? (((size_t)tile_g * 2 + (r >> 6)) * kGroups + g) * 64 + (r & 63)
                                   : ((size_t)tile_g * kGroups + g) * 128 + r;
    a[k] = *reinterpret_cast<const float4*>(p.dq_acc + idx * 4);
  }
  if (i >= p.N) return;
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    o[2 * k] = pack_bf16(a[k].x * p.scale, a[k].y * p.scale);
    o[2 * k + 1] = pack_bf16(a[k].z * p.scale, a[k].w * p.scale);
  }
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dq) + ((size_t)bh * p.N + i) * D + 16 * q);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// ---------------------------------------------------------------- main
// MASK: pairs follow p.mask (window and block map; not with CAUSAL): each
// key tile visits only the query tiles holding a visible pair, P is zeroed
// per pair in tiles that are not fully visible, and in deterministic mode a
// query tile takes its visible key tiles in ascending order.
// GQA: bh indexes K/V heads (p.kv_group query heads share one); each key tile
// walks the query tiles of all its query heads, so dK and dV sum over them
// in tensor memory, while dQ and the tickets stay per query head.
template <int D, bool CAUSAL, bool DETERMINISTIC, bool MASK = false, bool GQA = false>
__global__ void __launch_bounds__(512, 1) bwd_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdLayout<D>;
  static_assert(!(MASK && CAUSAL), "the masked instance expresses causality as a window");
  static_assert(!(MASK && GQA), "the masked instance has one K/V head per query head");
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(p.status, ATTN_ERR_BOUNDS, 2);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  // work unit: key tile j of head bh.  Causal key tiles with small j are the
  // longest (they see the most query tiles) and go first in either order.
  const int n = p.n_tiles;
  const int n_heads = GQA ? p.BH / p.kv_group : p.BH;  // K/V heads
  int j, bh;
  if (DETERMINISTIC) {  // a CTA waits only on CTAs launched before it
    det_unit(blockIdx.x, n_heads, n, MASK ? n_heads : p.det_group, MASK ? 0 : p.det_desc, j, bh);
  } else {  // head-major: resident CTAs share one or two heads' dQ accumulators in L2
    bh = blockIdx.x / n;
    j = blockIdx.x - bh * n;
  }
  const int i_lo = CAUSAL ? j : 0;  // query tiles i_lo .. n-1, visited from n-1 down
  int n_it = n - i_lo;
  // GQA: walk position qi = g * n + i over query head g of the group and
  // query tile i (from n-1 down to i_lo, head after head); the first query
  // head of K/V head bh is qh0
  int qh0 = bh;
  if (GQA) {
    const int h_kv = p.h_q / p.kv_group;
    qh0 = (bh / h_kv) * p.h_q + (bh % h_kv) * p.kv_group;
    n_it *= p.kv_group;
  }
  auto tile_i = [&](int qi) { return GQA ? qi % n : qi; };
  auto head_q = [&](int qi) { return GQA ? qh0 + qi / n : bh; };
  if (MASK) {  // only the query tiles holding a visible pair with key tile j
    n_it = 0;
    for (int i = 0; i < n; ++i) n_it += mask_tile_visible(p.mask, i, j) ? 1 : 0;
  }
  // every role walks the same query tiles, from the last down
  const int i_first = MASK ? mask_prev_query_tile(p.mask, j, n) : n - 1;
  auto i_next = [&](int i) {
    if (GQA) return (i % n) > i_lo ? i - 1 : (i / n + 1) * n + (n - 1);
    return MASK ? mask_prev_query_tile(p.mask, j, i) : i - 1;
  };

  if (threadIdx.x == 0) {
    for (int b = 0; b < L::kNumBars; ++b) {
      uint32_t cnt = 1;
      if ((b >= L::kBarPReady && b < L::kBarPReady + 2) || (b >= L::kBarDSFull && b < L::kBarDSFull + 2))
        cnt = 256;  // both compute warpgroups
      if (b == L::kBarDQFree) cnt = 128;  // the dQ warpgroup
      if (b >= L::kBarStgFull && b < L::kBarStgFull + 4) cnt = 4;  // the dQ warpgroup's warps
      mbar_init(bar(b), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(L::kCtlRegs));
   if (warp == 0) {
    // ============================ producer ============================
    if (lane == 0) {
      prefetch_tensormap(&p.tm_q);
      prefetch_tensormap(&p.tm_k);
      prefetch_tensormap(&p.tm_v);
      prefetch_tensormap(&p.tm_do);
      mbar_arrive_expect_tx(bar(L::kBarKV), 2 * L::kTileBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sbase + L::kKOff + c * kBSub, &p.tm_k, c * 64, j * kBTile, bh, bar(L::kBarKV));
        tma_load_3d(sbase + L::kVOff + c * kBSub, &p.tm_v, c * 64, j * kBTile, bh, bar(L::kBarKV));
      }
      int issued_q = 0, issued_do = 0;  // loads issued per ring
      for (int it = 0, qi = i_first; it < n_it; ++it, qi = i_next(qi)) {
        const int i = tile_i(qi);
        const int qh = head_q(qi);
        const int s = it % L::kQStages;
        const uint32_t ph = ((it / L::kQStages) & 1) ^ 1;
        const int sd = it % L::kDOStages;
        const uint32_t phd = ((it / L::kDOStages) & 1) ^ 1;
        if (!mbar_wait(bar(L::kBarQEmpty + s), ph, ctl, kBWhereProd)) break;
        mbar_arrive_expect_tx(bar(L::kBarQFull + s), L::kTileBytes + L::kVecBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sbase + L::kQOff + s * L::kTileBytes + c * kBSub, &p.tm_q, c * 64, i * kBTile, qh,
                      bar(L::kBarQFull + s));
        const size_t vrow = (size_t)qh * p.Npad + (size_t)i * kBTile;
        bulk_load(sbase + L::kVecOff + s * L::kVecBytes, p.row_lse2 + vrow, kBTile * 4, bar(L::kBarQFull + s));
        bulk_load(sbase + L::kVecOff + s * L::kVecBytes + kBTile * 4, p.row_d + vrow, kBTile * 4,
                  bar(L::kBarQFull + s));
        ATTN_TRACE_AT(blockIdx.x, it, 13);
        issued_q = it + 1;
        if (!mbar_wait(bar(L::kBarDOEmpty + sd), phd, ctl, kBWhereProd + 1)) break;
        mbar_arrive_expect_tx(bar(L::kBarDOFull + sd), L::kTileBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sbase + L::kDOOff + sd * L::kTileBytes + c * kBSub, &p.tm_do, c * 64, i * kBTile, qh,
                      bar(L::kBarDOFull + sd));
        ATTN_TRACE_AT(blockIdx.x, it, 14);
        issued_do = it + 1;
      }
      // loads still in flight land before the CTA exits: each ring's last
      // (stage count) loads, each on the newest phase of its stage
      mbar_wait_drain(bar(L::kBarKV), 0, p.timeout_ns);
      for (int it = issued_q > L::kQStages ? issued_q - L::kQStages : 0; it < issued_q; ++it)
        mbar_wait_drain(bar(L::kBarQFull + it % L::kQStages), (it / L::kQStages) & 1, p.timeout_ns);
      for (int it = issued_do > L::kDOStages ? issued_do - L::kDOStages : 0; it < issued_do; ++it)
        mbar_wait_drain(bar(L::kBarDOFull + it % L::kDOStages), (it / L::kDOStages) & 1, p.timeout_ns);
    }
    __syncwarp();  // lanes 1-31 wait for lane 0 before the final barrier
  } else if (warp == 1) {
    // ============================ MMA issuer ===========================
    if (lane == 0) {
      constexpr uint32_t kIdSq = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, false, true);    // dV, dK (A in tensor memory)
      constexpr uint32_t kIdDq = idesc_bf16_f32(128, D, true, true);      // dQ (A = dS, MN-major)
      // C = A B^T with A [128 x D] K-major at a_base and B [128 x D] K-major at b_base
      auto mma_kmajor = [&](uint32_t d_col, uint32_t a_base, uint32_t b_base) {
        const uint64_t da = sdesc_sw128(a_base, 16, 1024);
        const uint64_t db = sdesc_sw128(b_base, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * kBSub + (kk % 4) * 32;
          mma_ss(tmem + d_col, sdesc_advance(da, off), sdesc_advance(db, off), kIdSq, kk > 0);
        }
      };
      // C (+)= A[tmem, 128 x 128 bf16] B, B = [128 (K) x D] MN-major at b_base.
      // A's queries 64h..64h+63 sit packed in columns 64h..64h+31.  Half m
      // takes the K steps of queries 64h+32m .. 64h+32m+31 (h = 0, 1).
      auto mma_tmem_a_half = [&](uint32_t d_col, uint32_t a_col, uint32_t b_base, bool acc, int m) {
        const uint64_t db = sdesc_sw128(b_base, kBSub, 1024);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int kk = 4 * hh + 2 * m + u;
            mma_ts(tmem + d_col, tmem + a_col + (kk / 4) * 64 + (kk % 4) * 8, sdesc_advance(db, kk * 2048), kIdAcc,
                   (acc || m > 0 || hh > 0 || u > 0) ? 1u : 0u);
          }
      };
      bool ok = mbar_wait(bar(L::kBarKV), 0, ctl, kBWhereMma);
      tc_fence_after();
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it % L::kQStages;
        const uint32_t ph = (it / L::kQStages) & 1;
        const int sd = it % L::kDOStages;
        const uint32_t phd = (it / L::kDOStages) & 1;
        const uint32_t qs = sbase + L::kQOff + s * L::kTileBytes;
        const uint32_t dos = sbase + L::kDOOff + sd * L::kTileBytes;
        if (!(ok = mbar_wait(bar(L::kBarQFull + s), ph, ctl, kBWhereMma + 1))) break;
        ATTN_TRACE_AT(blockIdx.x, it, 0);
        tc_fence_after();
        mma_kmajor(L::kColS, sbase + L::kKOff, qs);  // the compute warpgroups start P on it
        tc_commit(bar(L::kBarSFull));
        ATTN_TRACE_AT(blockIdx.x, it, 10);
        if (!(ok = mbar_wait(bar(L::kBarDOFull + sd), phd, ctl, kBWhereMma + 3))) break;
        ATTN_TRACE_AT(blockIdx.x, it, 2);
        if (L::kColDQ == L::kColDP && it > 0)  // dP^T columns still hold dQ of the previous tile
          if (!(ok = mbar_wait(bar(L::kBarDQFree), (it - 1) & 1, ctl, kBWhereMma + 2))) break;
        ATTN_TRACE_AT(blockIdx.x, it, 1);
        tc_fence_after();
        mma_kmajor(L::kColDP, sbase + L::kVOff, dos);  // runs while P is computed
        tc_commit(bar(L::kBarDPFull));
        // dV on each half of P^T as it lands (runs while dS is computed)
#pragma unroll
        for (int m = 0; m < 2 && ok; ++m) {
          if (!(ok = mbar_wait(bar(L::kBarPReady + m), it & 1, ctl, kBWhereMma + 4))) break;
          if (m == 0) ATTN_TRACE_AT(blockIdx.x, it, 3);
          tc_fence_after();
          mma_tmem_a_half(L::kColDV, L::kColS, dos, it > 0, m);
        }
        if (!ok) break;
        tc_commit(bar(L::kBarDOEmpty + sd));  // dO_i's last reader: reload it early
#pragma unroll
        for (int m = 0; m < 2 && ok; ++m) {
          if (!(ok = mbar_wait(bar(L::kBarDSFull + m), it & 1, ctl, kBWhereMma + 6))) break;
          if (m == 0) ATTN_TRACE_AT(blockIdx.x, it, 12);
          tc_fence_after();
          mma_tmem_a_half(L::kColDK, L::kColDP, qs, it > 0, m);
        }
        if (!ok) break;
        tc_commit(bar(L::kBarQEmpty + s));
        if (L::kColDQ != L::kColDP && it > 0)
          if (!(ok = mbar_wait(bar(L::kBarDQFree), (it - 1) & 1, ctl, kBWhereMma + 5))) break;
        tc_fence_after();
        {
          const uint64_t da = sdesc_sw128(sbase + L::kDSOff, kBSub, 1024);
          const uint64_t db = sdesc_sw128(sbase + L::kKOff, kBSub, 1024);
#pragma unroll
          for (int kk = 0; kk < kBTile / 16; ++kk)
            mma_ss(tmem + L::kColDQ, sdesc_advance(da, kk * 2048), sdesc_advance(db, kk * 2048), kIdDq, kk > 0);
        }
        tc_commit(bar(L::kBarDQFull));
        ATTN_TRACE_AT(blockIdx.x, it, 4);
      }
      tc_commit(bar(L::kBarAccDone));
      mbar_wait_drain(bar(L::kBarAccDone), 0, p.timeout_ns);
    }
    __syncwarp();
   } else if (DETERMINISTIC) {
    // ==================== dQ reducers (deterministic mode) ====================
    // Warps 2 and 3 take the query tiles in turn.  For each of its tiles a
    // reducer waits for the staging rounds the dQ warpgroup writes, waits for
    // the tile's ticket, hands each round to the copy engine as a bulk FP32
    // reduce-add (the next round is issued before the previous one's slot is
    // freed, so the copy engine always has one queued) and frees each ring
    // slot once it has been read; then it waits until its additions are
    // complete and passes the ticket on.  That
    // wait overlaps the other reducer's next tile, so neither the dQ
    // warpgroup nor the products behind it wait for the completion of the
    // additions.
    if (lane == 0) {
      const int w = warp - 2;
      int kt = 0;  // tiles this reducer has taken
      bool ok = true;
      for (int it = 0, qi = i_first; ok && it < n_it; ++it, qi = i_next(qi)) {
        if ((it & 1) != w) continue;
        const int i = tile_i(qi);
        const int qh = head_q(qi);
        float* gdst = p.dq_acc + ((size_t)qh * p.n_tiles + i) * (size_t)(D * kBTile);
        int* ticket = p.tickets + (size_t)qh * p.n_tiles + i;
        // tile i takes its (visible) key tiles in the schedule's order
        int rank = det_rank(i, j, n, CAUSAL, p.det_desc);
        if (MASK) {
          rank = 0;
          for (int jj = 0; jj < j; ++jj) rank += mask_tile_visible(p.mask, i, jj) ? 1 : 0;
        }
        constexpr int kRoundFloats = L::kSlotBytes / 4;
        for (int r = 0; ok && r < L::kRounds; ++r) {
          const int sl = r & 1;
          const uint32_t par = (uint32_t)(kt * (L::kRounds / 2) + (r >> 1)) & 1;
          if (!(ok = mbar_wait(bar(L::kBarStgFull + 2 * w + sl), par, ctl, kBWhereDq + 2))) break;
          if (r == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(ticket) != rank) {
              if (*ctl.abort || globaltimer_ns() - t0 > ctl.timeout_ns) {
                if (!*ctl.abort) report_error(ctl.status, ATTN_ERR_TIMEOUT, kBWhereTicket);
                *ctl.abort = 1;
                break;
              }
            }
            fence_proxy_async_global();
            if (*ctl.abort) ok = false;
          }
          if (!ok) break;
          if (CAUSAL && p.acc_first_store && rank == 0)  // the tile's first contribution (causal instances only)
            bulk_store(gdst + (size_t)r * kRoundFloats, sbase + L::kStgOff + sl * L::kSlotBytes, L::kSlotBytes);
          else
            bulk_reduce_add_f32(gdst + (size_t)r * kRoundFloats, sbase + L::kStgOff + sl * L::kSlotBytes,
                                L::kSlotBytes);
          bulk_commit();
          if (r > 0) {  // the previous round's slot has been read: it may be overwritten
            bulk_wait_read<1>();
            mbar_arrive(bar(L::kBarStgFree + (sl ^ 1)));
          }
        }
        if (!ok) break;
        bulk_wait_read<0>();
        mbar_arrive(bar(L::kBarStgFree + ((L::kRounds - 1) & 1)));
        ++kt;
        bulk_wait_all<0>();  // the additions are performed before the next key tile's
        fence_proxy_async_global();
        red_release_gpu_add(ticket, 1);
      }
      bulk_wait_all<0>();  // nothing in flight when the CTA exits
    }
    __syncwarp();
   }
#ifdef ATTN_TRACE
   else if (warp == 2) {
    // debug only: completion times of the products, seen by polling
    if (lane == 0 && blockIdx.x < kTraceCtas) {
      bool live = true;
      auto seen = [&](uint32_t b, uint32_t par) {
        for (int i = 0; live && i < (1 << 22); ++i)
          if (mbar_test(b, par)) return;
        live = false;
      };
      for (int it = 0; live && it < n_it && it < kTraceIters; ++it) {
        seen(bar(L::kBarSFull), it & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 16);
        seen(bar(L::kBarDPFull), it & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 17);
        seen(bar(L::kBarDOEmpty + it % L::kDOStages), (it / L::kDOStages) & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 18);
        seen(bar(L::kBarQEmpty + it % L::kQStages), (it / L::kQStages) & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 19);
        seen(bar(L::kBarDQFull), it & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 20);
      }
    }
    __syncwarp();
   }
#endif
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kComputeRegs));
    // ================= two compute warpgroups (h = 0, 1) =================
    // Warpgroup h takes queries 64h .. 64h+63 of the elementwise steps (keys on
    // tensor-memory lanes) and writes columns [h*D/2, (h+1)*D/2) of the dV /
    // dK epilogue.  The next tile's dS is only written after its dP^T product
    // completed, and that product was issued after this tile's dQ product
    // (which reads dS), so the buffer is free.
    const int h = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int lrow = quad * 32 + lane;      // tensor-memory lane: key row
    const int tid = threadIdx.x - 128 - 128 * h;  // 0..127 within the warpgroup
    const int k_glob = j * kBTile + lrow;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::kColS;
    const uint32_t tDP = tmem + lane_base + L::kColDP;
    const float c_log2 = p.scale_log2;
    const bool key_dead = k_glob >= p.N;
    bool ok = true;
    for (int it = 0, qi = i_first; it < n_it; ++it, qi = i_next(qi)) {
      const int i = tile_i(qi);
      const int s = it % L::kQStages;
      // LSE2 / D vectors arrive with Q_i on the stage's barrier
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarQFull + s), (it / L::kQStages) & 1, ctl, kBWhereEw + 3));
      if (!ok) break;
      const float* vec = reinterpret_cast<const float*>(smem + L::kVecOff + s * L::kVecBytes);
      const bool diag = CAUSAL && i == j;
      // the mask only bites on the diagonal tile and on a ragged last key tile
      // (masked instance: on every tile the window does not cover whole)
      const bool mask_tile = MASK ? !mask_tile_full(p.mask, i, j) : (diag || (j * kBTile + kBTile > p.N));
      // Phase 1 (needs S^T): P = 2^(S^T * scale * log2e - LSE2) for this
      // warpgroup's 64 queries, kept in FP32 registers and packed as bf16
      // P^T into columns 64h .. 64h+31 (inside the columns just read).
      // Phase 2 (needs dP^T): dS = P o (dP - D), packed as dS^T the same way
      // and written to shared memory as dS for the dQ product.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull), it & 1, ctl, kBWhereEw));
      if (!ok) break;
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 5 + h);
      tc_fence_after();
      float pv[64];
      auto p_chunk = [&](int m, auto masked) {
        const int c0 = 64 * h + 32 * m;
        float sv[32];
        tmem_ld32(tS + c0, sv);
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float4 nl = *reinterpret_cast<const float4*>(vec + c0 + q);  // -LSE2 (negated upstream)
          const float2 x01 = __ffma2_rn(make_float2(sv[q], sv[q + 1]), make_float2(c_log2, c_log2), make_float2(nl.x, nl.y));
          const float2 x23 = __ffma2_rn(make_float2(sv[q + 2], sv[q + 3]), make_float2(c_log2, c_log2), make_float2(nl.z, nl.w));
          float p0 = ex2_mufu(x01.x), p1 = ex2_mufu(x01.y), p2 = ex2_mufu(x23.x), p3 = ex2_mufu(x23.y);
          if constexpr (decltype(masked)::value) {
            const int q0 = i * kBTile + c0 + q;  // global query index of p0
            if constexpr (MASK) {  // key k_glob is visible from query r when r - left <= k_glob <= r + right
              auto hid = [&](int r) {
                return key_dead || (p.mask.left >= 0 && k_glob < r - p.mask.left) ||
                       (p.mask.right >= 0 && k_glob > r + p.mask.right);
              };
              if (hid(q0)) p0 = 0.f;
              if (hid(q0 + 1)) p1 = 0.f;
              if (hid(q0 + 2)) p2 = 0.f;
              if (hid(q0 + 3)) p3 = 0.f;
            } else {
              if (key_dead || (diag && q0 < k_glob)) p0 = 0.f;
              if (key_dead || (diag && q0 + 1 < k_glob)) p1 = 0.f;
              if (key_dead || (diag && q0 + 2 < k_glob)) p2 = 0.f;
              if (key_dead || (diag && q0 + 3 < k_glob)) p3 = 0.f;
            }
          }
          pv[32 * m + q] = p0;
          pv[32 * m + q + 1] = p1;
          pv[32 * m + q + 2] = p2;
          pv[32 * m + q + 3] = p3;
          pk[q >> 1] = pack_bf16(p0, p1);
          pk[(q >> 1) + 1] = pack_bf16(p2, p3);
        }
        tmem_st16(tS + 64 * h + 16 * m, pk);
      };
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (mask_tile) p_chunk(m, std::true_type{});
        else p_chunk(m, std::false_type{});
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kBarPReady + m));
      }

      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDPFull), it & 1, ctl, kBWhereEw + 1));
      if (!ok) break;
      tc_fence_after();
      // dS (queries x keys) into shared memory, MN-major with the 128-byte
      // swizzle: query chunk h at 16 KB, key row lrow at
      // (lrow/8)*1024 + (lrow%8)*128, 16-byte unit (q%64)/8 xor (lrow%8).
      uint8_t* ds_row = smem + L::kDSOff + h * kBSub + (lrow >> 3) * 1024 + (lrow & 7) * 128;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int c0 = 64 * h + 32 * m;
        float dp[32];
        tmem_ld32(tDP + c0, dp);
        uint32_t dk[16];
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float4 nd = *reinterpret_cast<const float4*>(vec + kBTile + c0 + q);  // -D (negated upstream)
          const float2 ds01 = __fmul2_rn(make_float2(pv[32 * m + q], pv[32 * m + q + 1]),
                                         __fadd2_rn(make_float2(dp[q], dp[q + 1]), make_float2(nd.x, nd.y)));
          const float2 ds23 = __fmul2_rn(make_float2(pv[32 * m + q + 2], pv[32 * m + q + 3]),
                                         __fadd2_rn(make_float2(dp[q + 2], dp[q + 3]), make_float2(nd.z, nd.w)));
          dk[q >> 1] = pack_bf16(ds01.x, ds01.y);
          dk[(q >> 1) + 1] = pack_bf16(ds23.x, ds23.y);
        }
        tmem_st16(tDP + 64 * h + 16 * m, dk);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (4 * m + u) ^ (lrow & 7);
          *reinterpret_cast<uint4*>(ds_row + unit * 16) = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::kBarDSFull + m));
      }
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 7 + h);
    }
    // epilogue: dV and dK rows of this key tile.  Warpgroup h takes columns
    // [h*D/2, (h+1)*D/2): each thread writes its key row into 64-column boxes
    // in shared memory (the Q stages, free now: the last products have
    // completed), in the 128-byte swizzled layout (16-byte unit c of row r at
    // unit c ^ (r % 8)), then one thread has the copy engine store the boxes
    // as whole rows (rows past N left out).
    // (The deterministic instances keep direct row stores from registers:
    // there the TMA epilogue measured 3-4 % slower at N = 16384.)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarAccDone), 0, ctl, kBWhereFin));
    if constexpr (DETERMINISTIC) {
      if (ok) {
        tc_fence_after();
        const size_t row = (size_t)bh * p.N + (key_dead ? 0 : k_glob);
        uint4* dvrow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dv) + row * D);
        uint4* dkrow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dk) + row * D);
#pragma unroll
        for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
          float a[32], b[32];
          if (n_it > 0) {
            tmem_ld32(tmem + lane_base + L::kColDV + c0, a);
            tmem_ld32(tmem + lane_base + L::kColDK + c0, b);
          } else {  // (masked instance) no query sees this key tile: dK = dV = 0
#pragma unroll
            for (int q = 0; q < 32; ++q) a[q] = b[q] = 0.f;
          }
          uint32_t pa[16], pb[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            pa[q] = pack_bf16(a[2 * q], a[2 * q + 1]);
            pb[q] = pack_bf16(b[2 * q] * p.scale, b[2 * q + 1] * p.scale);
          }
          if (!key_dead) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              dvrow[c0 / 8 + v] = make_uint4(pa[4 * v], pa[4 * v + 1], pa[4 * v + 2], pa[4 * v + 3]);
              dkrow[c0 / 8 + v] = make_uint4(pb[4 * v], pb[4 * v + 1], pb[4 * v + 2], pb[4 * v + 3]);
            }
          }
        }
      }
    } else {
    ok = named_bar_and(2, 256, ok);  // both compute warpgroups (the stores below need every row)
    if (ok) {
      tc_fence_after();
      constexpr int kBoxes = D / 64;          // per tensor
      constexpr uint32_t kBoxBytes = kBTile * 128;
      const uint32_t stg_dv = sbase + L::kQOff;
      const uint32_t stg_dk = stg_dv + kBoxes * kBoxBytes;
      static_assert(2 * kBoxes * kBoxBytes <= L::kQStages * L::kTileBytes, "dV / dK boxes fit the Q stages");
#pragma unroll
      for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
        float a[32], b[32];
        if (n_it > 0) {
          tmem_ld32(tmem + lane_base + L::kColDV + c0, a);
          tmem_ld32(tmem + lane_base + L::kColDK + c0, b);
        } else {  // (masked instance) no query sees this key tile: dK = dV = 0
#pragma unroll
          for (int q = 0; q < 32; ++q) a[q] = b[q] = 0.f;
        }
        uint32_t pa[16], pb[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          pa[q] = pack_bf16(a[2 * q], a[2 * q + 1]);
          pb[q] = pack_bf16(b[2 * q] * p.scale, b[2 * q + 1] * p.scale);
        }
        const uint32_t box_off = (uint32_t)(c0 / 64) * kBoxBytes + (uint32_t)lrow * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t unit = (uint32_t)(((c0 % 64) / 8 + v) ^ (lrow & 7)) * 16;
          st_shared_v4(stg_dv + box_off + unit, pa[4 * v], pa[4 * v + 1], pa[4 * v + 2], pa[4 * v + 3]);
          st_shared_v4(stg_dk + box_off + unit, pb[4 * v], pb[4 * v + 1], pb[4 * v + 2], pb[4 * v + 3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(2, 256);
      if (h == 0 && tid == 0) {
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx) {
          tma_store_3d(&p.tm_dv, stg_dv + bx * kBoxBytes, bx * 64, j * kBTile, bh);
          tma_store_3d(&p.tm_dk, stg_dk + bx * kBoxBytes, bx * 64, j * kBTile, bh);
        }
        bulk_commit();
        bulk_wait_read<0>();  // shared memory is read before the CTA exits
      }
    }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kDqRegs));
    // ========================== dQ warpgroup ===========================
    // Reads dQ_i (queries on tensor-memory lanes) as soon as its product is
    // done, frees those columns, and has the copy engine add the tile into
    // the FP32 accumulator while the other warpgroups move on to the next
    // query tile.
    const int quad = warp & 3;
    const int qrow = quad * 32 + lane;
    const int tid = threadIdx.x - 384;
    const uint32_t tDQ = tmem + ((uint32_t)(quad * 32) << 16) + L::kColDQ;
    bool ok = true;
    for (int it = 0, qi = i_first; it < n_it; ++it, qi = i_next(qi)) {
      const int i = tile_i(qi);
      const int qh = head_q(qi);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDQFull), it & 1, ctl, kBWhereDq));
      // the four warps leave together (the atomic mode's named barriers below)
      if (!DETERMINISTIC) ok = named_bar_and(1, 128, ok);
      if (!ok) break;
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 9);
      tc_fence_after();
      float dq[D];
      if constexpr (D == 128) {  // two 64-column loads, one wait each
        tmem_ld64(tDQ, *reinterpret_cast<float(*)[64]>(dq));
        tmem_ld64(tDQ + 64, *reinterpret_cast<float(*)[64]>(dq + 64));
      } else {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) tmem_ld32p(tDQ + c0, dq + c0);
      }
      tc_fence_before();
      mbar_arrive(bar(L::kBarDQFree));  // tensor-memory dQ columns may be overwritten
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 15);
      // Stage the tile in shared memory in the accumulator's [D/4 column
      // groups][128 rows][4] order (each thread's 16-byte stores land side by
      // side with its neighbours') round by round through the two-slot ring,
      // and the copy engine adds each round into the FP32 accumulator as a
      // bulk reduce-add.
      float* stg = reinterpret_cast<float*>(smem + L::kStgOff);
      constexpr int kRoundGroups = D / 4 / L::kRounds;
      if constexpr (DETERMINISTIC) {
        // the reducer warps (above) issue the additions in ticket order; here
        // each round is staged into its ring slot once the slot's previous
        // round has been read
#pragma unroll
        for (int r = 0; r < L::kRounds && ok; ++r) {
          const int sl = r & 1;
          const int use = (it * L::kRounds + r) >> 1;  // earlier rounds through this slot
          if (use > 0)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(L::kBarStgFree + sl), (uint32_t)(use - 1) & 1, ctl, kBWhereDq + 1));
          if (!ok) break;
          float* slot = stg + sl * (L::kSlotBytes / 4);
#pragma unroll
          for (int g = 0; g < kRoundGroups; ++g) {
            const int gg = r * kRoundGroups + g;
            *reinterpret_cast<float4*>(slot + (g * kBTile + qrow) * 4) =
                make_float4(dq[4 * gg], dq[4 * gg + 1], dq[4 * gg + 2], dq[4 * gg + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::kBarStgFull + 2 * (it & 1) + sl));
        }
        if (!ok) break;
        if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 11);
        continue;
      }
      // atomic mode: this warpgroup issues the reduce-adds itself; a round is
      // staged into its ring slot once the slot's previous round has been
      // read (all but the newest bulk group complete), while the copy engine
      // still reads the other slot
      float* gdst = p.dq_acc + ((size_t)qh * p.n_tiles + i) * (size_t)(D * kBTile);
#pragma unroll
      for (int r = 0; r < L::kRounds; ++r) {
        const int sl = r & 1;
        if (it > 0 || r > 1) {
          if (tid == 0) bulk_wait_read<1>();
          __syncwarp();
          named_bar_sync(1, 128);
        }
        float* slot = stg + sl * (L::kSlotBytes / 4);
#pragma unroll
        for (int g = 0; g < kRoundGroups; ++g) {
          const int gg = r * kRoundGroups + g;
          *reinterpret_cast<float4*>(slot + (g * kBTile + qrow) * 4) =
              make_float4(dq[4 * gg], dq[4 * gg + 1], dq[4 * gg + 2], dq[4 * gg + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (tid == 0 && !*ctl.abort) {
          bulk_reduce_add_f32(gdst + (size_t)r * (L::kSlotBytes / 4), smem_u32(slot), L::kSlotBytes);
          bulk_commit();
        }
        __syncwarp();  // lane 0 rejoins its warp before the next (aligned) named barrier
      }
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 11);
    }
    if (tid == 0) bulk_wait_all<0>();  // staging reads done before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Main kernel of the CTA-pair backward (defined in attn_bwd2.cuh, d = 128).
template <bool CAUSAL, bool DET>
cudaError_t launch_bwd2_main(const BwdParams& p, cudaStream_t stream);

// Persistent main kernel for short sequences (attn_bwd_persist.cuh).
template <int D, bool CAUSAL, bool DET>
cudaError_t launch_bwd_persist_main(BwdParams& p, cudaStream_t stream);

template <int D, bool CAUSAL, bool DET, bool MASK = false, bool GQA = false>
cudaError_t launch_bwd_instance(const BwdParams& p, cudaStream_t stream, const LaunchEvents* evs) {
  using L = BwdLayout<D>;
  auto mark = [&](int i) {
    if (evs != nullptr && evs->ev[i] != nullptr) cudaEventRecord(evs->ev[i], stream);
  };
  mark(0);
  // preprocess: D, LSE2, zeroed accumulator / tickets
  {
    const long rows = (long)p.BH * p.Npad;
    const int rows_per_block = 256 / (D / 8);
    const long blocks = (rows + rows_per_block - 1) / rows_per_block;
    bwd_pre_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  mark(1);
  bool paired = false;
  if constexpr (D == 128) {
    if (p.pair_mode && !MASK && !GQA) {
      cudaError_t e = launch_bwd2_main<CAUSAL, DET>(p, stream);
      if (e != cudaSuccess) return e;
      paired = true;
    }
  }
  BwdParams pc = p;  // the persistent launch adds its cut-tail plan, which the conversion finishes
  pc.tail_s = 1;
  if constexpr (!MASK && !GQA) {
    if (!paired && p.persist) {
      cudaError_t e = launch_bwd_persist_main<D, CAUSAL, DET>(pc, stream);
      if (e != cudaSuccess) return e;
      paired = true;  // (the main kernel has run: skip the one-unit launch)
    }
  }
  if (!paired) {
    auto kernel = bwd_kernel<D, CAUSAL, DET, MASK, GQA>;
    // setmaxnreg.inc waits for registers the dec released: the split must
    // match what the launch hands out
    cudaError_t e = prepare_kernel((const void*)kernel, L::kSmemBytes, L::kLaunchRegs, nullptr);
    if (e != cudaSuccess) return e;
    const int n_heads = GQA ? p.BH / p.kv_group : p.BH;  // one CTA per (K/V head, key tile)
    kernel<<<n_heads * p.n_tiles, L::kThreads, L::kSmemBytes, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  mark(2);
  {
    const long blocks = dq_convert_blocks<D>(pc) + tail_sum_blocks<D>(pc);
    dq_convert_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(pc);
    cudaError_t e = cudaGetLastError();
    mark(3);
    return e;
  }
}

}  // namespace attn
