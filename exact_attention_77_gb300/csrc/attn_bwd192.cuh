// Backward attention for d_qk = 192, d_v = 128 (sm_103a).
//
// The same graph of five products and two elementwise steps as bwd_kernel
// ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", Figure 2 and Table 3), for the head shape
// d_qk = 192, d_v = 128 that the same page's Figure 5 measures its forward on:
//     S^T  = K_j Q_i^T   (K = 192)        dP^T = V_j dO_i^T   (K = 128)
//     dV  += P^T dO_i    (N = 128)        dK  += dS^T Q_i     (N = 192)
//     dQ_i = dS K_j      (N = 192)
//
// What differs from bwd_kernel is the tensor-memory plan.  Its layout would
// need dV (128) + dK (192) + S^T (128) + dP^T (128) = 576 columns, over the
// 512 an SM has.  Here S^T and dP^T take turns in one 128-column region X:
// the compute warpgroups read S^T into registers (they keep P there for dS
// anyway) and pack bf16 P^T into a separate 64-column region PK.  The query
// columns go in two halves of 64: once both warpgroups have read half m of
// S^T, dP^T of those queries (an N = 64 product) is written over it while
// they work on the other half.  dS^T is packed into PK after the dV product
// has read P^T.  dQ_i (192 columns) spans X and PK; its read-out frees X
// first, so the next tile's S^T starts before the last columns are read.
// Totals: dV 128 + dK 192 + X 128 + PK 64 = 512.
//
// Shared memory: K_j 48 KiB, V_j 32 KiB, one Q_i stage 48 KiB, one dO_i stage
// 32 KiB, dS 32 KiB, the dQ staging tile 32 KiB: 225 KiB.
//
// Warp roles as in bwd_kernel: warp 0 producer, warp 1 MMA issuer, warps
// 4-11 two compute warpgroups (half m of the queries: warpgroup h takes
// queries 64m+32h .. 64m+32h+31), warps 12-15 the dQ warpgroup.  Atomic or
// deterministic dQ accumulation, causal or not, grouped-query heads.
#pragma once

#include <type_traits>

#include "attn_bwd.cuh"

namespace attn {

struct Bwd192Layout {
  static constexpr int kDQK = 192;
  static constexpr int kDV = 128;
  static constexpr int kQKBytes = kBTile * kDQK * 2;  // K_j, Q_i: three 64-column chunks
  static constexpr int kVBytes = kBTile * kDV * 2;    // V_j, dO_i: two chunks
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kQKBytes;
  static constexpr int kQOff = kVOff + kVBytes;
  static constexpr int kDOOff = kQOff + kQKBytes;
  static constexpr int kDSOff = kDOOff + kVBytes;  // dS (bf16 128x128), MN-major for the dQ product
  static constexpr int kDSBytes = kBTile * kBTile * 2;
  // dQ_i staging: a ring of two 16 KiB slots; a tile goes through it in six
  // rounds of 32 columns, round r in slot r % 2, so that one round is staged
  // while the copy engine reads the other
  static constexpr int kStgOff = kDSOff + kDSBytes;
  static constexpr int kStgBytes = 32 * 1024;
  static constexpr int kSlotBytes = kStgBytes / 2;
  static constexpr int kRounds = kBTile * kDQK * 4 / kSlotBytes;  // 6
  static constexpr int kRoundGroups = kSlotBytes / (kBTile * 16);  // 8 four-column groups
  static constexpr int kVecOff = kStgOff + kStgBytes;  // -LSE2[128], -D[128] fp32 of Q_i
  static constexpr int kVecBytes = 2 * kBTile * 4;
  static constexpr int kBarOff = kVecOff + kVecBytes;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;
  static constexpr int kBarQEmpty = 2;
  static constexpr int kBarDOFull = 3;
  static constexpr int kBarDOEmpty = 4;
  static constexpr int kBarSFull = 5;
  static constexpr int kBarDPFull = 6;   // + half m: dP^T of queries 64m .. 64m+63 (commit)
  static constexpr int kBarPReady = 8;   // + half m: S^T half m read, P^T half m packed (256 arrivals)
  static constexpr int kBarDSFull = 10;  // + half m: dS^T and dS of half m (256 arrivals)
  static constexpr int kBarDQFull = 12;
  static constexpr int kBarDQFreeX = 13;   // 128 arrivals: dQ columns over X read
  static constexpr int kBarDQFreePK = 14;  // 128 arrivals: dQ columns over PK read
  static constexpr int kBarAccDone = 15;
  // deterministic mode (as in bwd_kernel): + 2 w + s: staging slot s holds a
  // round of reducer warp w's tile (4 dQ-warp arrivals); + s: slot s has
  // been read by the copy engine (1 arrival)
  static constexpr int kBarStgFull = 16;
  static constexpr int kBarStgFree = 20;
  static constexpr int kNumBars = 22;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kKOff % 1024 == 0 && kVOff % 1024 == 0 && kQOff % 1024 == 0 && kDOOff % 1024 == 0 &&
                    kDSOff % 1024 == 0 && kStgOff % 1024 == 0,
                "128-byte-swizzled tiles start on 1024-byte boundaries");
  // tensor memory columns
  static constexpr int kColDV = 0;
  static constexpr int kColDK = kColDV + kDV;
  static constexpr int kColX = kColDK + kDQK;  // S^T, then dP^T (fp32, 128 columns)
  static constexpr int kColPK = kColX + 128;   // P^T, then dS^T (bf16 packed, 64 columns)
  static constexpr int kColDQ = kColX;         // dQ_i fp32 over X and PK (192 columns)
  static_assert(kColPK + 64 == 512 && kColDQ + kDQK == 512, "tensor-memory plan");
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128;
  static constexpr int kCtlRegs = 112;
  static constexpr int kComputeRegs = 128;
  static constexpr int kDqRegs = 144;
  static_assert(kCtlRegs * 128 + kComputeRegs * 256 + kDqRegs * 128 <= kLaunchRegs * kThreads, "register split");
};

enum : int { kB192WhereProd = 160, kB192WhereMma = 170, kB192WhereEw = 180, kB192WhereDq = 190 };

// Preprocess for this head shape: -D and -LSE2 as bwd_pre_kernel<128> (dO and
// O rows are d_v = 128 wide), zeroing the 192-wide dQ accumulator.
__global__ void __launch_bounds__(256) bwd192_pre_kernel(BwdParams p) {
  constexpr int kLanes = 16;  // 128 / 8
  constexpr int kRowsPerBlock = 256 / kLanes;
  const int sub = threadIdx.x % kLanes;
  const long row = (long)blockIdx.x * kRowsPerBlock + threadIdx.x / kLanes;
  const long total_rows = (long)p.BH * p.Npad;
  const bool in_range = row < total_rows;
  const int bh = in_range ? (int)(row / p.Npad) : 0;
  const int i = in_range ? (int)(row - (long)bh * p.Npad) : p.N;
  float acc = 0.f;
  if (i < p.N) {
    const size_t off = ((size_t)bh * p.N + i) * 128 + sub * 8;
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
  const size_t n4 = (size_t)p.BH * p.Npad * Bwd192Layout::kDQK / 4;
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n4; k += (size_t)gridDim.x * blockDim.x)
    acc4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.tickets != nullptr)
    for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < (size_t)p.BH * p.n_tiles;
         k += (size_t)gridDim.x * blockDim.x)
      p.tickets[k] = 0;
}

// dQ = scale * accumulator as bf16 [BH, N, 192]; accumulator per (bh, tile)
// in [48 column groups][128 rows][4] order.
__global__ void __launch_bounds__(256) dq192_convert_kernel(BwdParams p) {
  // as dq_convert_kernel: one row and four consecutive column groups per
  // thread, 32 consecutive rows of the same groups per warp
  constexpr int kGroups = Bwd192Layout::kDQK / 4;  // 48
  constexpr int kQuads = kGroups / 4;              // 12
  const long x = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long per_tile = 128L * kQuads;
  const long tile_g = x / per_tile;  // over BH * n_tiles
  if (tile_g >= (long)p.BH * p.n_tiles) return;
  const int tt = (int)(x - tile_g * per_tile);
  const int w = tt >> 5;
  const int r = (w & 3) * 32 + (threadIdx.x & 31);
  const int q = w >> 2;
  const int bh = (int)(tile_g / p.n_tiles);
  const int i = (int)(tile_g - (long)bh * p.n_tiles) * 128 + r;
  float4 a[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    a[k] = *reinterpret_cast<const float4*>(p.dq_acc + (((size_t)tile_g * kGroups + 4 * q + k) * 128 + r) * 4);
  if (i >= p.N) return;
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    o[2 * k] = pack_bf16(a[k].x * p.scale, a[k].y * p.scale);
    o[2 * k + 1] = pack_bf16(a[k].z * p.scale, a[k].w * p.scale);
  }
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dq) +
                                        ((size_t)bh * p.N + i) * Bwd192Layout::kDQK + 16 * q);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

template <bool CAUSAL, bool DETERMINISTIC, bool GQA>
__global__ void __launch_bounds__(512, 1) bwd192_kernel(const __grid_constant__ BwdParams p) {
  using L = Bwd192Layout;
  constexpr int DQK = L::kDQK;
  constexpr int DV = L::kDV;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report_error(p.status, ATTN_ERR_BOUNDS, 3);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  // work unit: key tile j of K/V head bh (unit order as in bwd_kernel)
  const int n = p.n_tiles;
  const int n_heads = GQA ? p.BH / p.kv_group : p.BH;
  int j, bh;
  if (DETERMINISTIC) {
    det_unit(blockIdx.x, n_heads, n, p.det_group, p.det_desc, j, bh);
  } else {
    bh = blockIdx.x / n;
    j = blockIdx.x - bh * n;
  }
  const int i_lo = CAUSAL ? j : 0;
  int n_it = n - i_lo;
  int qh0 = bh;
  if (GQA) {
    const int h_kv = p.h_q / p.kv_group;
    qh0 = (bh / h_kv) * p.h_q + (bh % h_kv) * p.kv_group;
    n_it *= p.kv_group;
  }
  // walk position qi = g * n + i: query head g of the group, query tile i
  // from n-1 down to i_lo
  auto tile_i = [&](int qi) { return GQA ? qi % n : qi; };
  auto head_q = [&](int qi) { return GQA ? qh0 + qi / n : bh; };
  auto i_next = [&](int qi) {
    if (GQA) return (qi % n) > i_lo ? qi - 1 : (qi / n + 1) * n + (n - 1);
    return qi - 1;
  };
  const int i_first = n - 1;

  if (threadIdx.x == 0) {
    for (int b = 0; b < L::kNumBars; ++b) {
      uint32_t cnt = 1;
      if (b == L::kBarPReady || b == L::kBarPReady + 1 || b == L::kBarDSFull || b == L::kBarDSFull + 1) cnt = 256;
      if (b == L::kBarDQFreeX || b == L::kBarDQFreePK) cnt = 128;
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
        mbar_arrive_expect_tx(bar(L::kBarKV), L::kQKBytes + L::kVBytes);
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_3d(sbase + L::kKOff + c * kBSub, &p.tm_k, c * 64, j * kBTile, bh, bar(L::kBarKV));
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(sbase + L::kVOff + c * kBSub, &p.tm_v, c * 64, j * kBTile, bh, bar(L::kBarKV));
        int issued_q = 0, issued_do = 0;
        for (int it = 0, qi = i_first; it < n_it; ++it, qi = i_next(qi)) {
          const int i = tile_i(qi);
          const int qh = head_q(qi);
          const uint32_t ph = (it & 1) ^ 1;
          if (!mbar_wait(bar(L::kBarQEmpty), ph, ctl, kB192WhereProd)) break;
          ATTN_TRACE_AT(blockIdx.x, it, 25);
          mbar_arrive_expect_tx(bar(L::kBarQFull), L::kQKBytes + L::kVecBytes);
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            tma_load_3d(sbase + L::kQOff + c * kBSub, &p.tm_q, c * 64, i * kBTile, qh, bar(L::kBarQFull));
          const size_t vrow = (size_t)qh * p.Npad + (size_t)i * kBTile;
          bulk_load(sbase + L::kVecOff, p.row_lse2 + vrow, kBTile * 4, bar(L::kBarQFull));
          bulk_load(sbase + L::kVecOff + kBTile * 4, p.row_d + vrow, kBTile * 4, bar(L::kBarQFull));
          issued_q = it + 1;
          if (!mbar_wait(bar(L::kBarDOEmpty), ph, ctl, kB192WhereProd + 1)) break;
          mbar_arrive_expect_tx(bar(L::kBarDOFull), L::kVBytes);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(sbase + L::kDOOff + c * kBSub, &p.tm_do, c * 64, i * kBTile, qh, bar(L::kBarDOFull));
          issued_do = it + 1;
          // With one Q stage the next Q_i load sits on the critical path (it
          // starts when this tile's dK product is done): its tiles are
          // fetched into L2 a whole tile ahead.  Measured on GB300: +3-4 %
          // in deterministic mode; with atomic dQ 3 % slower while the dQ
          // partials went through one 32 KiB staging tile, and 0-2 % faster
          // since they go through the two-slot ring.
          if (it + 1 < n_it) {
            const int qn = i_next(qi);
#pragma unroll
            for (int c = 0; c < DQK / 64; ++c) tma_prefetch_l2_3d(&p.tm_q, c * 64, tile_i(qn) * kBTile, head_q(qn));
#pragma unroll
            for (int c = 0; c < DV / 64; ++c) tma_prefetch_l2_3d(&p.tm_do, c * 64, tile_i(qn) * kBTile, head_q(qn));
          }
        }
        // loads in flight land before the CTA exits (one stage per ring)
        mbar_wait_drain(bar(L::kBarKV), 0, p.timeout_ns);
        if (issued_q > 0) mbar_wait_drain(bar(L::kBarQFull), (issued_q - 1) & 1, p.timeout_ns);
        if (issued_do > 0) mbar_wait_drain(bar(L::kBarDOFull), (issued_do - 1) & 1, p.timeout_ns);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ============================ MMA issuer ===========================
      if (lane == 0) {
        constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);   // S^T
        constexpr uint32_t kIdDP = idesc_bf16_f32(128, 64, false, false);   // dP^T, one query half
        constexpr uint32_t kIdDV = idesc_bf16_f32(128, DV, false, true);    // dV (A in tensor memory)
        constexpr uint32_t kIdDK = idesc_bf16_f32(128, DQK, false, true);   // dK (A in tensor memory)
        constexpr uint32_t kIdDQ = idesc_bf16_f32(128, DQK, true, true);    // dQ (A = dS, MN-major)
        // C = A B^T, A [128 x KD] and B [rows x KD] K-major in 64-column
        // chunks kBSub apart
        auto mma_kmajor = [&](uint32_t d_col, uint32_t a_base, uint32_t b_base, uint32_t id, auto kd) {
          const uint64_t da = sdesc_sw128(a_base, 16, 1024);
          const uint64_t db = sdesc_sw128(b_base, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < decltype(kd)::value / 16; ++kk) {
            const uint32_t off = (kk / 4) * kBSub + (kk % 4) * 32;
            mma_ss(tmem + d_col, sdesc_advance(da, off), sdesc_advance(db, off), id, kk > 0);
          }
        };
        // C (+)= A[tensor memory: 128 keys x 128 queries, bf16] B, B [128
        // queries (K) x N] MN-major in 64-column chunks kBSub apart.  A's
        // queries 16kk .. 16kk+15 sit in columns kColPK + 8kk .. +7; half m
        // takes K steps kk = 4m .. 4m+3.
        auto mma_pk_half = [&](uint32_t d_col, uint32_t b_base, uint32_t id, bool acc, int m) {
          const uint64_t db = sdesc_sw128(b_base, kBSub, 1024);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int kk = 4 * m + u;
            mma_ts(tmem + d_col, tmem + L::kColPK + kk * 8, sdesc_advance(db, kk * 2048), id,
                   (acc || m > 0 || u > 0) ? 1u : 0u);
          }
        };
        bool ok = mbar_wait(bar(L::kBarKV), 0, ctl, kB192WhereMma);
        tc_fence_after();
        for (int it = 0; ok && it < n_it; ++it) {
          const uint32_t ph = it & 1;
          const uint32_t qs = sbase + L::kQOff;
          const uint32_t dos = sbase + L::kDOOff;
          if (!(ok = mbar_wait(bar(L::kBarQFull), ph, ctl, kB192WhereMma + 1))) break;
          ATTN_TRACE_AT(blockIdx.x, it, 0);
          // X holds dQ of the previous tile until its read-out got past it
          if (it > 0 && !(ok = mbar_wait(bar(L::kBarDQFreeX), ph ^ 1, ctl, kB192WhereMma + 2))) break;
          ATTN_TRACE_AT(blockIdx.x, it, 1);
          tc_fence_after();
          mma_kmajor(L::kColX, sbase + L::kKOff, qs, kIdS, std::integral_constant<int, DQK>{});
          tc_commit(bar(L::kBarSFull));
          if (!(ok = mbar_wait(bar(L::kBarDOFull), ph, ctl, kB192WhereMma + 3))) break;
          ATTN_TRACE_AT(blockIdx.x, it, 3);
          // per query half m, once both warpgroups have read it from S^T and
          // packed P^T: dV on it, then its dP^T over the S^T columns just read
#pragma unroll
          for (int m = 0; m < 2 && ok; ++m) {
            if (!(ok = mbar_wait(bar(L::kBarPReady + m), ph, ctl, kB192WhereMma + 4))) break;
            ATTN_TRACE_AT(blockIdx.x, it, 4 + 2 * m);
            tc_fence_after();
            mma_pk_half(L::kColDV, dos, kIdDV, it > 0, m);
            mma_kmajor(L::kColX + 64 * m, sbase + L::kVOff, dos + m * 8192, kIdDP, std::integral_constant<int, DV>{});
            tc_commit(bar(L::kBarDPFull + m));
          }
          if (!ok) break;
          tc_commit(bar(L::kBarDOEmpty));  // dO_i's last reader
#pragma unroll
          for (int m = 0; m < 2 && ok; ++m) {
            if (!(ok = mbar_wait(bar(L::kBarDSFull + m), ph, ctl, kB192WhereMma + 6))) break;
            ATTN_TRACE_AT(blockIdx.x, it, 8 + m);
            tc_fence_after();
            mma_pk_half(L::kColDK, qs, kIdDK, it > 0, m);
          }
          if (!ok) break;
          tc_commit(bar(L::kBarQEmpty));
          {
            const uint64_t da = sdesc_sw128(sbase + L::kDSOff, kBSub, 1024);
            const uint64_t db = sdesc_sw128(sbase + L::kKOff, kBSub, 1024);
#pragma unroll
            for (int kk = 0; kk < kBTile / 16; ++kk)
              mma_ss(tmem + L::kColDQ, sdesc_advance(da, kk * 2048), sdesc_advance(db, kk * 2048), kIdDQ, kk > 0);
          }
          tc_commit(bar(L::kBarDQFull));
          ATTN_TRACE_AT(blockIdx.x, it, 10);
        }
        tc_commit(bar(L::kBarAccDone));
        mbar_wait_drain(bar(L::kBarAccDone), 0, p.timeout_ns);
      }
      __syncwarp();
    } else if (DETERMINISTIC) {
      // ================= dQ reducers (deterministic mode) ==================
      // Warps 2 and 3 take the query tiles in turn: for each of the tile's
      // six staged rounds the reducer waits for it, (first round) waits for
      // the tile's ticket, hands it to the copy engine as a bulk FP32
      // reduce-add and frees its ring slot once read (one round later, so
      // the copy engine always has the next one queued); after the last
      // round it waits for the additions to complete and passes the ticket
      // on, while the other reducer already serves the next tile.
      if (lane == 0) {
        const int w = warp - 2;
        int kt = 0;  // tiles this reducer has taken
        bool ok = true;
        for (int it = 0, qi = i_first; ok && it < n_it; ++it, qi = i_next(qi)) {
          if ((it & 1) != w) continue;
          const int i = tile_i(qi);
          const int qh = head_q(qi);
          float* gdst = p.dq_acc + ((size_t)qh * p.n_tiles + i) * (size_t)(DQK * kBTile);
          int* ticket = p.tickets + (size_t)qh * p.n_tiles + i;
          const int rank = det_rank(i, j, n, CAUSAL, p.det_desc);  // the fixed order
          for (int r = 0; ok && r < L::kRounds; ++r) {
            const int sl = r & 1;
            const uint32_t par = (uint32_t)(kt * (L::kRounds / 2) + (r >> 1)) & 1;
            if (!(ok = mbar_wait(bar(L::kBarStgFull + 2 * w + sl), par, ctl, kB192WhereDq + 2))) break;
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
            bulk_reduce_add_f32(gdst + (size_t)r * (L::kSlotBytes / 4), sbase + L::kStgOff + sl * L::kSlotBytes,
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
          ATTN_TRACE_AT(blockIdx.x, it, 27);
          seen(bar(L::kBarDPFull), it & 1);
          ATTN_TRACE_AT(blockIdx.x, it, 28);
          seen(bar(L::kBarDPFull + 1), it & 1);
          ATTN_TRACE_AT(blockIdx.x, it, 29);
          seen(bar(L::kBarQEmpty), it & 1);
          ATTN_TRACE_AT(blockIdx.x, it, 30);
          seen(bar(L::kBarDQFull), it & 1);
          ATTN_TRACE_AT(blockIdx.x, it, 31);
        }
      }
      __syncwarp();
    }
#endif
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kComputeRegs));
    // ================= two compute warpgroups (h = 0, 1) =================
    const int h = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int lrow = quad * 32 + lane;  // tensor-memory lane: key row
    const int tid = threadIdx.x - 128 - 128 * h;  // 0..127 within the warpgroup
    const int k_glob = j * kBTile + lrow;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tX = tmem + lane_base + L::kColX;
    const uint32_t tPK = tmem + lane_base + L::kColPK + 16 * h;
    const float c_log2 = p.scale_log2;
    const bool key_dead = k_glob >= p.N;
    const float* vec = reinterpret_cast<const float*>(smem + L::kVecOff);
    bool ok = true;
    for (int it = 0, qi = i_first; it < n_it; ++it, qi = i_next(qi)) {
      const int i = tile_i(qi);
      const uint32_t ph = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarQFull), ph, ctl, kB192WhereEw + 3));
      if (!ok) break;
      const bool diag = CAUSAL && i == j;
      const bool mask_tile = diag || (j * kBTile + kBTile > p.N);
      // Phase 1 (S^T in X): P = 2^(S^T * scale * log2e - LSE2) for this
      // warpgroup's queries c0 = 64m+32h .. c0+31 of each half m, kept in
      // registers and packed as bf16 P^T into PK columns c0/2 .. c0/2+15.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull), ph, ctl, kB192WhereEw));
      if (!ok) break;
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 11 + h);
      // PK held dQ of the previous tile until its read-out got past it
      if (it > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDQFreePK), ph ^ 1, ctl, kB192WhereEw + 2));
      if (!ok) break;
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 13 + h);
      tc_fence_after();
      float pv[64];
      auto p_chunk = [&](int m, auto masked) {
        const int c0 = 64 * m + 32 * h;
        float sv[32];
        tmem_ld32(tX + c0, sv);
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float4 nl = *reinterpret_cast<const float4*>(vec + c0 + q);  // -LSE2
          const float2 x01 = __ffma2_rn(make_float2(sv[q], sv[q + 1]), make_float2(c_log2, c_log2), make_float2(nl.x, nl.y));
          const float2 x23 = __ffma2_rn(make_float2(sv[q + 2], sv[q + 3]), make_float2(c_log2, c_log2), make_float2(nl.z, nl.w));
          float p0 = ex2_mufu(x01.x), p1 = ex2_mufu(x01.y), p2 = ex2_mufu(x23.x), p3 = ex2_mufu(x23.y);
          if constexpr (decltype(masked)::value) {
            const int q0 = i * kBTile + c0 + q;
            if (key_dead || (diag && q0 < k_glob)) p0 = 0.f;
            if (key_dead || (diag && q0 + 1 < k_glob)) p1 = 0.f;
            if (key_dead || (diag && q0 + 2 < k_glob)) p2 = 0.f;
            if (key_dead || (diag && q0 + 3 < k_glob)) p3 = 0.f;
          }
          pv[32 * m + q] = p0;
          pv[32 * m + q + 1] = p1;
          pv[32 * m + q + 2] = p2;
          pv[32 * m + q + 3] = p3;
          pk[q >> 1] = pack_bf16(p0, p1);
          pk[(q >> 1) + 1] = pack_bf16(p2, p3);
        }
        tmem_st16(tPK + 32 * m, pk);
      };
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (mask_tile) p_chunk(m, std::true_type{});
        else p_chunk(m, std::false_type{});
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kBarPReady + m));
      }
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 15 + h);

      // Phase 2 (dP^T half m in X, written once half m of S^T was read):
      // dS = P o (dP - D), packed as dS^T into PK (the dV product of half m
      // has read P^T there: it was issued before that dP^T) and written to
      // shared memory as dS: query half m at m * 16 KB, key row lrow at
      // (lrow/8)*1024 + (lrow%8)*128, 16-byte unit (q%64)/8 xor (lrow%8).
      uint8_t* ds_row = smem + L::kDSOff + (lrow >> 3) * 1024 + (lrow & 7) * 128;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDPFull + m), ph, ctl, kB192WhereEw + 1));
        if (!ok) break;
        if (tid == 0 && m == 0) ATTN_TRACE_AT(blockIdx.x, it, 17 + h);
        tc_fence_after();
        const int c0 = 64 * m + 32 * h;
        float dp[32];
        tmem_ld32(tX + c0, dp);
        uint32_t dk[16];
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float4 nd = *reinterpret_cast<const float4*>(vec + kBTile + c0 + q);  // -D
          const float2 ds01 = __fmul2_rn(make_float2(pv[32 * m + q], pv[32 * m + q + 1]),
                                         __fadd2_rn(make_float2(dp[q], dp[q + 1]), make_float2(nd.x, nd.y)));
          const float2 ds23 = __fmul2_rn(make_float2(pv[32 * m + q + 2], pv[32 * m + q + 3]),
                                         __fadd2_rn(make_float2(dp[q + 2], dp[q + 3]), make_float2(nd.z, nd.w)));
          dk[q >> 1] = pack_bf16(ds01.x, ds01.y);
          dk[(q >> 1) + 1] = pack_bf16(ds23.x, ds23.y);
        }
        tmem_st16(tPK + 32 * m, dk);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (4 * h + u) ^ (lrow & 7);
          *reinterpret_cast<uint4*>(ds_row + m * kBSub + unit * 16) =
              make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::kBarDSFull + m));
      }
      if (!ok) break;
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 19 + h);
    }
    // epilogue: warpgroup h takes dV columns [64h, 64h+64) and dK columns
    // [96h, 96h+96) of its key row, writes them into 64-column boxes in
    // shared memory (the Q and dO stages, free now) in the 128-byte swizzled
    // layout, and one thread has the copy engine store the boxes as whole
    // rows (rows past N left out)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarAccDone), 0, ctl, kB192WhereEw + 4));
    ok = named_bar_and(2, 256, ok);  // both compute warpgroups (the stores below need every row)
    if (ok) {
      tc_fence_after();
      constexpr uint32_t kBoxBytes = kBTile * 128;
      const uint32_t stg_dv = sbase + L::kQOff;                   // DV / 64 boxes
      const uint32_t stg_dk = stg_dv + (DV / 64) * kBoxBytes;    // DQK / 64 boxes
      static_assert(L::kDOOff == L::kQOff + L::kQKBytes && (DV + DQK) / 64 * kBoxBytes <= L::kQKBytes + L::kVBytes,
                    "dV / dK boxes fit the Q and dO stages");
      auto stage32 = [&](uint32_t col, uint32_t stg, int c0, float mul) {
        float a[32];
        if (n_it > 0) {
          tmem_ld32(tmem + lane_base + col, a);
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) a[q] = 0.f;
        }
        uint32_t pa[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) pa[q] = pack_bf16(a[2 * q] * mul, a[2 * q + 1] * mul);
        const uint32_t box_off = (uint32_t)(c0 / 64) * kBoxBytes + (uint32_t)lrow * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v)
          st_shared_v4(stg + box_off + (uint32_t)(((c0 % 64) / 8 + v) ^ (lrow & 7)) * 16, pa[4 * v], pa[4 * v + 1],
                       pa[4 * v + 2], pa[4 * v + 3]);
      };
#pragma unroll
      for (int c0 = 64 * h; c0 < 64 * h + 64; c0 += 32) stage32(L::kColDV + c0, stg_dv, c0, 1.f);
#pragma unroll
      for (int c0 = 96 * h; c0 < 96 * h + 96; c0 += 32) stage32(L::kColDK + c0, stg_dk, c0, p.scale);
      fence_proxy_async_smem();
      named_bar_sync(2, 256);
      if (h == 0 && tid == 0) {
#pragma unroll
        for (int bx = 0; bx < DV / 64; ++bx) tma_store_3d(&p.tm_dv, stg_dv + bx * kBoxBytes, bx * 64, j * kBTile, bh);
#pragma unroll
        for (int bx = 0; bx < DQK / 64; ++bx) tma_store_3d(&p.tm_dk, stg_dk + bx * kBoxBytes, bx * 64, j * kBTile, bh);
        bulk_commit();
        bulk_wait_read<0>();  // shared memory is read before the CTA exits
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kDqRegs));
    // ========================== dQ warpgroup ===========================
    // Round r stages dQ columns 32r .. 32r+31 in the accumulator's [48
    // groups][128 rows][4] order and has the copy engine add them.  Columns
    // 0 .. 127 (over X) are read first and released to the next tile's S^T;
    // columns 128 .. 191 (over PK) after the first two rounds.
    const int quad = warp & 3;
    const int qrow = quad * 32 + lane;
    const int tid = threadIdx.x - 384;
    const uint32_t tDQ = tmem + ((uint32_t)(quad * 32) << 16) + L::kColDQ;
    float* stg = reinterpret_cast<float*>(smem + L::kStgOff);
    bool ok = true;
    for (int it = 0, qi = i_first; it < n_it; ++it, qi = i_next(qi)) {
      const int i = tile_i(qi);
      const int qh = head_q(qi);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDQFull), it & 1, ctl, kB192WhereDq));
      // the four warps leave together (the atomic mode's named barriers below)
      if (!DETERMINISTIC) ok = named_bar_and(1, 128, ok);
      if (!ok) break;
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 21);
      tc_fence_after();
      float* gdst = p.dq_acc + ((size_t)qh * p.n_tiles + i) * (size_t)(DQK * kBTile);
      // stage round rr (32 columns, 8 four-column groups, from v) into ring
      // slot rr % 2 and have the copy engine add it
      auto round = [&](int rr, const float* v) {
        const int sl = rr & 1;
        float* slot = stg + sl * (L::kSlotBytes / 4);
        if constexpr (DETERMINISTIC) {
          // the reducer warps (above) issue the additions in ticket order;
          // the round is staged once the slot's previous round has been read
          const int use = (it * L::kRounds + rr) >> 1;  // earlier rounds through this slot
          if (ok && use > 0)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(L::kBarStgFree + sl), (uint32_t)(use - 1) & 1, ctl, kB192WhereDq + 1));
          if (!ok) return;
#pragma unroll
          for (int g = 0; g < L::kRoundGroups; ++g)
            *reinterpret_cast<float4*>(slot + (g * kBTile + qrow) * 4) =
                make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::kBarStgFull + 2 * (it & 1) + sl));
          return;
        }
        // atomic: the slot's previous round has been read once all but the
        // newest bulk group are complete
        if (it > 0 || rr > 1) {
          if (tid == 0) bulk_wait_read<1>();
          __syncwarp();
          named_bar_sync(1, 128);
        }
#pragma unroll
        for (int g = 0; g < L::kRoundGroups; ++g)
          *reinterpret_cast<float4*>(slot + (g * kBTile + qrow) * 4) =
              make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (tid == 0 && !*ctl.abort) {
          bulk_reduce_add_f32(gdst + (size_t)rr * (L::kSlotBytes / 4), smem_u32(slot), L::kSlotBytes);
          bulk_commit();
        }
        __syncwarp();
      };
      float a[64], b[64];
      tmem_ld64(tDQ, a);
      tmem_ld64(tDQ + 64, b);
      tc_fence_before();
      mbar_arrive(bar(L::kBarDQFreeX));
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 22);
      round(0, a);
      round(1, a + 32);
      tmem_ld64(tDQ + 128, a);
      tc_fence_before();
      mbar_arrive(bar(L::kBarDQFreePK));
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 23);
      round(2, b);
      round(3, b + 32);
      round(4, a);
      round(5, a + 32);
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 24);
      if (DETERMINISTIC && !ok) break;
      __syncwarp();
    }
    if (tid == 0) bulk_wait_all<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool CAUSAL, bool DET, bool GQA>
cudaError_t launch_bwd192_instance(const BwdParams& p, cudaStream_t stream, const LaunchEvents* evs) {
  using L = Bwd192Layout;
  auto mark = [&](int i) {
    if (evs != nullptr && evs->ev[i] != nullptr) cudaEventRecord(evs->ev[i], stream);
  };
  mark(0);
  {
    const long rows = (long)p.BH * p.Npad;
    const long blocks = (rows + 15) / 16;
    bwd192_pre_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  mark(1);
  {
    auto kernel = bwd192_kernel<CAUSAL, DET, GQA>;
    cudaError_t e = prepare_kernel((const void*)kernel, L::kSmemBytes, L::kLaunchRegs, nullptr);
    if (e != cudaSuccess) return e;
    const int n_heads = GQA ? p.BH / p.kv_group : p.BH;
    kernel<<<n_heads * p.n_tiles, L::kThreads, L::kSmemBytes, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  mark(2);
  {
    const long blocks = ((long)p.BH * p.n_tiles * 128 * 12 + 255) / 256;  // 12 threads per row
    dq192_convert_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    mark(3);
    return e;
  }
}

}  // namespace attn
