// Forward attention kernel for sm_103a (template; instantiated per head dim in
// attn_fwd_d*.cu).
//
// What it computes: O = softmax(scale Q K^T + causal mask) V and the per-row
// natural-log LSE, with the score matrix kept on chip ("Attention at Scale --
// From FlashAttention to FlashAttention-4", sections "The Problem" and "The
// Evolution"), the online softmax with conditional rescaling ("FlashAttention
// 3 and 4: When the Bottleneck Moves", section 3.2), and the exponentials split
// between the hardware unit and a polynomial (same section; "FlashAttention-4:
// Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling",
// abstract and Table 2).
//
// CTA structure (one CTA = NQT query tiles of 128 rows of one (b, h)):
//   warp 0      producer: TMA loads of the Q tiles, then K_j / V_j tiles into a
//               ring of shared-memory stages behind full/empty mbarriers;
//   warp 1      owns tensor memory; one thread issues every tcgen05.mma:
//               S_t = Q_t K_j^T (both operands K-major in shared memory) and
//               O_t += P_t V_j (P_t from tensor memory, V_j MN-major);
//   warps 2-3   idle (the first warpgroup hands its registers to the others);
//   warps 4..   one warpgroup per query tile: thread r owns row r of the tile,
//               loads its 128 scores from tensor memory, takes the row max,
//               rescales O_t and l only when the max rose by more than tau,
//               forms P = 2^(S*scale*log2e - m) in FP32 and writes it back as
//               bf16 over the first 64 columns of S_t, then normalises once at
//               the end.
// With two query tiles the issue order S_0(j+1) .. PV_1(j) .. S_1(j+1) lets one
// tile's softmax overlap the other tile's products ("FlashAttention-4 ...",
// Figure 1).  Tensor memory per query tile: S (128 columns) then O (d_v).
//
// Every wait is bounded (see sm103.cuh): on a timeout the kernel records
// ATTN_ERR_TIMEOUT, every role stops, in-flight copies and products are
// drained, tensor memory is released and the CTA exits.
#pragma once

#include "attn_mask.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace attn {

constexpr int kTile = 128;
constexpr int kSubTile = 128 * 128;  // bytes: 128 rows x 128 B (one 128-byte swizzle span: 64 bf16 or 128 e4m3)
// Of every 32 score columns, this many take the polynomial exponential and the
// rest the hardware unit (the "poly" kernel variants; 0 = hardware only).
constexpr int kPolyCols = 10;

// ES: bytes per operand element (2: bf16; 1: e4m3).
// KS, VS: 0 for one K/V ring of kStages equal stages that K_j and V_j take in
// turn; else KS stages sized for a K tile and VS for a V tile (K and V each
// in their own ring) and no O staging tile (the instance must stage O in its
// freed Q region).
template <int DQK, int DV, int NQT, int ES = 2, int KS = 0, int VS = 0>
struct FwdLayout {
  static constexpr int kQBytes = kTile * DQK * ES;
  static constexpr int kKBytes = kTile * DQK * ES;
  static constexpr int kVBytes = kTile * DV * ES;
  static constexpr int kChunkElems = 128 / ES;        // elements per 128-byte swizzle span
  static constexpr int kChunksQK = DQK * ES / 128;
  static constexpr int kChunksV = DV * ES / 128;
  static constexpr int kQKSteps = DQK * ES / 32;      // products of K = 32 bytes per S tile
  static constexpr int kPVSteps = kTile * ES / 32;    // products per P V (32-byte K steps)
  static constexpr int kPVKeys = 32 / ES;             // keys per P V product
  static constexpr int kStageBytes = kKBytes > kVBytes ? kKBytes : kVBytes;
  static constexpr int kQRegion = NQT * kQBytes;
  // Epilogue staging per query tile: one [128 rows x 64 columns] bf16 box of
  // O in the 128-byte swizzled layout the TMA store reads.
  static constexpr bool kSplitKV = KS > 0;
  static constexpr int kKStages = KS, kVStages = VS;
  static constexpr int kStgBytes = kSplitKV ? 0 : kTile * 64 * 2;
  // One query tile per CTA is sized so two CTAs share an SM (two softmax
  // warpgroups per SM either way); two tiles take the SM alone.
  static constexpr int kBudget = NQT == 1 ? 112 * 1024 : 226 * 1024;
  static constexpr int kStagesFit = (kBudget - kQRegion - NQT * kStgBytes) / kStageBytes;
  static constexpr int kStages = kSplitKV ? KS + VS : (kStagesFit > 4 ? 4 : kStagesFit);
  static_assert(kSplitKV ? (KS >= 1 && VS >= 1) : kStages >= 2, "K/V ring needs two stages");
  // Load ld of the K/V stream (even: K_j, odd: V_j; every unit starts on an
  // even ld): its stage, the parity of that stage's use, and the stage's
  // offset from kKVOff.
  __host__ __device__ static constexpr int stage_of(int ld) {
    return kSplitKV ? ((ld & 1) ? KS + (ld >> 1) % (VS > 0 ? VS : 1) : (ld >> 1) % (KS > 0 ? KS : 1))
                    : ld % kStages;
  }
  __host__ __device__ static constexpr uint32_t phase_of(int ld) {
    return (uint32_t)((kSplitKV ? ((ld & 1) ? (ld >> 1) / (VS > 0 ? VS : 1) : (ld >> 1) / (KS > 0 ? KS : 1))
                                : ld / kStages) & 1);
  }
  __host__ __device__ static constexpr int stage_off(int st) {
    return kSplitKV ? (st < KS ? st * kKBytes : KS * kKBytes + (st - KS) * kVBytes) : st * kStageBytes;
  }
  static constexpr int kThreads = 128 + 128 * NQT;
  static constexpr int kMinBlocks = NQT == 1 ? 2 : 1;
  // Register split (setmaxnreg): the launch gives every thread kLaunchRegs;
  // the control warpgroup drops to kCtlRegs and each softmax warpgroup rises
  // to kSmRegs.  kCtlRegs * 128 + kSmRegs * 128 * NQT == kLaunchRegs * kThreads.
  static constexpr int kLaunchRegs = NQT == 1 ? 128 : 168;
  static constexpr int kCtlRegs = NQT == 1 ? 48 : 88;
  static constexpr int kSmRegs = NQT == 1 ? 208 : 208;
  static_assert(kCtlRegs * 128 + kSmRegs * 128 * NQT == kLaunchRegs * kThreads, "register split");
  static constexpr int kKVOff = kQRegion;
  static constexpr int kStgOff = kKVOff + (kSplitKV ? KS * kKBytes + VS * kVBytes : kStages * kStageBytes);
  static constexpr int kBarOff = kStgOff + NQT * kStgBytes;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKVFull = 1;
  static constexpr int kBarKVEmpty = kBarKVFull + kStages;
  static constexpr int kBarSFull = kBarKVEmpty + kStages;
  static constexpr int kBarPFull = kBarSFull + NQT;
  static constexpr int kBarODone = kBarPFull + NQT;
  static constexpr int kBarOFree = kBarODone + NQT;    // + t: O_t read out by the epilogue (128 arrivals)
  static constexpr int kBarQEmpty = kBarOFree + NQT;   // the unit's last S products have read Q
  static constexpr int kBarMmaDone = kBarQEmpty + 1;
  static constexpr int kNumBars = kBarMmaDone + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // Tensor memory decides residency: two CTAs of 256 columns per SM, or one of
  // 512.  The shared-memory request is padded so no extra CTA lands on an SM
  // only to wait in tcgen05.alloc.
  static constexpr int kSmemMin = NQT == 1 ? 80 * 1024 : 116 * 1024;
  static constexpr int kSmemBytes = kMiscOff + 16 > kSmemMin ? kMiscOff + 16 : kSmemMin;
  static constexpr int kTmemCols = NQT == 1 ? 256 : 512;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Where-codes recorded with a timeout (role * 10 + wait).
enum : int {
  kWhereProdEmpty = 10, kWhereMmaQ = 20, kWhereMmaKV = 21, kWhereMmaP = 22, kWhereMmaO = 23,
  kWhereSmS = 30, kWhereSmO = 31, kWhereSmFinal = 32, kWhereAlign = 1
};

// SPLIT (non-causal only): each unit also takes one of p.n_splits ranges of
// p.split_tiles key tiles, keys come from a sequence of p.Nk rows, and the
// epilogue writes the range's normalised FP32 output and LSE to p.o_part /
// p.lse_part for the merge kernel (split-KV for decode-shaped problems).
// FP8 (d = 128): Q, K, V are e4m3 codes with per-tile scales p.sq,
// p.sk and a per-head scale p.sv; the products run as kind::f8f6f4; the
// softmax forms 2^8 P against a running max updated on every rise (the host
// passes tau = 0) and stores it as e4m3 over the first 32 columns of S_t.
// MASK (one query tile per CTA): keys follow p.mask (window and block map);
// each unit visits only the key tiles holding a visible pair, in ascending
// order, and masks per pair inside the tiles that are not fully visible.
template <int DQK, int DV, int NQT, bool CAUSAL, int POLY, bool PERSIST, bool SPLIT = false, bool FP8 = false,
          bool MASK = false>
__global__ void __launch_bounds__(FwdLayout<DQK, DV, NQT>::kThreads, FwdLayout<DQK, DV, NQT>::kMinBlocks)
    fwd_kernel(const __grid_constant__ FwdParams p) {
  // d_qk = 192 with one unit per CTA: two 48 KiB K stages and one 32 KiB V
  // stage instead of two 48 KiB stages that K_j and V_j take in turn (O is
  // staged in the freed Q region, so the staging tile's 32 KiB go to the
  // second K stage).  Measured on GB300 against the shared ring: +5-6 % at
  // N = 8192-16384, causal and not; one K and two V stages gave +1-2 %.
  static constexpr bool kKV21 = DQK == 192 && !PERSIST && !SPLIT && !FP8 && !MASK;
  using L = FwdLayout<DQK, DV, NQT, FP8 ? 1 : 2, kKV21 ? 2 : 0, kKV21 ? 1 : 0>;
  static_assert(!FP8 || (DQK == 128 && DV == 128 && !SPLIT), "FP8 instance: d = 128");
  static_assert(!MASK || (NQT == 1 && !CAUSAL && !SPLIT && !FP8), "masked instance: one query tile, no other mode");
  // (the FP8 instance is built with POLY = 0: the polynomial share measured
  // slower there too, and its larger error moves more P codes)
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // swizzled operand tiles need 1024-byte alignment
    if (threadIdx.x == 0) report_error(p.status, ATTN_ERR_BOUNDS, kWhereAlign);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  // ---- work units: (bh, block of NQT query tiles).  The CTA is persistent:
  // it takes units blockIdx.x, blockIdx.x + gridDim.x, ... and every role
  // runs its pipeline straight across unit boundaries (barrier phases and
  // the K/V ring position carry over), so the next unit's Q, K and V load
  // and its first products issue while this unit's epilogue runs.
  const int n_qblocks = (p.n_qtiles + NQT - 1) / NQT;
  static_assert(!(SPLIT && CAUSAL), "split-KV is non-causal");
  const int n_kv_tiles = SPLIT ? p.n_kv_tiles : p.n_qtiles;
  const int n_keys = SPLIT ? p.Nk : p.N;
  struct Unit {
    int bh, qblock, nkv[NQT], nkv_max, j0, split;
  };
  auto unit_at = [&](int u) {
    Unit w;
    w.j0 = 0;
    w.split = 0;
    int kv_len = n_kv_tiles;
    if (SPLIT) {  // the splits of one query block are neighbours
      w.split = u % p.n_splits;
      u /= p.n_splits;
      w.j0 = w.split * p.split_tiles;
      kv_len = min(n_kv_tiles - w.j0, p.split_tiles);
    }
    if (CAUSAL) {  // longest rows first, spread over heads
      const int rank = u / p.BH;
      w.bh = u - rank * p.BH;
      w.qblock = n_qblocks - 1 - rank;
    } else {  // head-major keeps one head's K/V hot in L2
      w.bh = u / n_qblocks;
      w.qblock = u - w.bh * n_qblocks;
    }
    w.nkv_max = 0;
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
      const int qt = w.qblock * NQT + t;
      w.nkv[t] = qt < p.n_qtiles ? (CAUSAL ? qt + 1 : kv_len) : 0;
      if (MASK && qt < p.n_qtiles) {  // visible key tiles; the first one in j0
        int cnt = 0;
        w.j0 = p.n_qtiles;
        for (int kt = 0; kt < p.n_qtiles; ++kt)
          if (mask_tile_visible(p.mask, qt, kt)) {
            if (cnt == 0) w.j0 = kt;
            ++cnt;
          }
        w.nkv[t] = cnt;
      }
      w.nkv_max = w.nkv[t] > w.nkv_max ? w.nkv[t] : w.nkv_max;
    }
    return w;
  };
  // CTA b takes, in round r, unit r*G + b (r even) or r*G + G-1-b (r odd):
  // with the units sorted longest first (causal), the serpentine order hands
  // every CTA a similar total.
  // Without PERSIST the grid has one CTA per unit and all of this folds away.
  const int n_units = PERSIST ? p.n_blocks : (int)gridDim.x;
  const int G = gridDim.x;
  const int n_rounds = PERSIST ? (n_units + G - 1) / G : 1;
  auto unit_of_round = [&](int r) {
    return PERSIST ? r * G + ((r & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x) : (int)blockIdx.x;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarQFull), 1);
    mbar_init(bar(L::kBarQEmpty), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarKVFull + s), 1);
      mbar_init(bar(L::kBarKVEmpty + s), 1);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(bar(L::kBarSFull + t), 1);
      mbar_init(bar(L::kBarPFull + t), 128);
      mbar_init(bar(L::kBarODone + t), 1);
      mbar_init(bar(L::kBarOFree + t), 128);
    }
    mbar_init(bar(L::kBarMmaDone), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the merge kernel (a programmatic dependent launch) may be scheduled now;
  // it waits for this grid's completion before reading the partials
  if (SPLIT && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp < 4) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(L::kCtlRegs));
   if (warp == 0) {
    // =========================== producer ===========================
    if (lane == 0) {
      prefetch_tensormap(&p.tm_q);
      prefetch_tensormap(&p.tm_k);
      prefetch_tensormap(&p.tm_v);
      int issued = 0;  // K/V loads so far (K_j and V_j alternate through the ring)
      int qn = 0;      // units started
      bool ok = true;
      for (int r = 0; ok && r < n_rounds; ++r) {
        const int u = unit_of_round(r);
        if (u >= n_units) continue;
        const Unit w = unit_at(u);
        if (PERSIST && qn > 0 && !mbar_wait(bar(L::kBarQEmpty), (qn - 1) & 1, ctl, kWhereProdEmpty)) break;
        mbar_arrive_expect_tx(bar(L::kBarQFull), NQT * L::kQBytes);
#pragma unroll
        for (int t = 0; t < NQT; ++t)
#pragma unroll
          for (int c = 0; c < L::kChunksQK; ++c)
            tma_load_3d(sbase + t * L::kQBytes + c * kSubTile, &p.tm_q, c * L::kChunkElems,
                        (w.qblock * NQT + t) * kTile, w.bh, bar(L::kBarQFull));
        ++qn;
        // K/V head of this unit (grouped-query attention shares one among kv_group query heads)
        const int kv_bh =
            p.kv_group <= 1 ? w.bh : (w.bh / p.h_q) * (p.h_q / p.kv_group) + (w.bh % p.h_q) / p.kv_group;
        int kt = w.j0;  // key tile of step j (masked instance: the visible ones in order)
        for (int j = 0; ok && j < w.nkv_max; ++j, kt = MASK ? mask_next_key_tile(p.mask, w.qblock, kt) : kt + 1) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ld = issued;
            const int s = L::stage_of(ld);
            if (!mbar_wait(bar(L::kBarKVEmpty + s), L::phase_of(ld) ^ 1, ctl, kWhereProdEmpty)) {
              ok = false;
              break;
            }
            const uint32_t dst = sbase + L::kKVOff + L::stage_off(s);
            ATTN_TRACE_AT(blockIdx.x, j, 13 + h);
            if (h == 0) {
              mbar_arrive_expect_tx(bar(L::kBarKVFull + s), L::kKBytes);
#pragma unroll
              for (int c = 0; c < L::kChunksQK; ++c)
                tma_load_3d(dst + c * kSubTile, &p.tm_k, c * L::kChunkElems, kt * kTile, kv_bh,
                            bar(L::kBarKVFull + s));
            } else {
              mbar_arrive_expect_tx(bar(L::kBarKVFull + s), L::kVBytes);
#pragma unroll
              for (int c = 0; c < L::kChunksV; ++c)
                tma_load_3d(dst + c * kSubTile, &p.tm_v, c * L::kChunkElems, kt * kTile, kv_bh,
                            bar(L::kBarKVFull + s));
            }
            issued = ld + 1;
          }
        }
      }
      // copies still in flight must land before the CTA can exit
      if (qn > 0) mbar_wait_drain(bar(L::kBarQFull), (qn - 1) & 1, p.timeout_ns);
      // (the last use of every stage: the last kStages loads of one ring, or
      // the last KS K loads and VS V loads of split rings)
      if constexpr (L::kSplitKV) {
        for (int ld = issued > 2 * L::kKStages ? issued - 2 * L::kKStages : 0; ld < issued; ld += 2)  // K (issued is even)
          mbar_wait_drain(bar(L::kBarKVFull + L::stage_of(ld)), L::phase_of(ld), p.timeout_ns);
        for (int ld = issued > 2 * L::kVStages ? issued - 2 * L::kVStages + 1 : 1; ld < issued; ld += 2)  // V
          mbar_wait_drain(bar(L::kBarKVFull + L::stage_of(ld)), L::phase_of(ld), p.timeout_ns);
      } else {
        for (int ld = issued > L::kStages ? issued - L::kStages : 0; ld < issued; ++ld)
          mbar_wait_drain(bar(L::kBarKVFull + L::stage_of(ld)), L::phase_of(ld), p.timeout_ns);
      }
    }
    __syncwarp();  // lanes 1-31 wait for lane 0 before the final barrier
  } else if (warp == 1) {
    // =========================== MMA issuer =========================
    // The whole warp runs this loop in step (waits included); one elected
    // lane issues every product and commit.
    constexpr uint32_t kIdescQK = FP8 ? idesc_e4m3_f32(128, 128, false, false) : idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdescPV = FP8 ? idesc_e4m3_f32(128, DV, false, true) : idesc_bf16_f32(128, DV, false, true);
    auto wait_all = [&](uint32_t b, uint32_t parity, int where) -> bool {
      const bool r = __all_sync(0xffffffffu, mbar_wait(b, parity, ctl, where));
      tc_fence_after();
      return r;
    };
    auto wait_load = [&](int ld) -> bool {
      return wait_all(bar(L::kBarKVFull + L::stage_of(ld)), L::phase_of(ld), kWhereMmaKV);
    };
    auto issue_qk = [&](int t, int stage) {
      const uint64_t da = sdesc_sw128(sbase + t * L::kQBytes, 16, 1024);
      const uint64_t db = sdesc_sw128(sbase + L::kKVOff + L::stage_off(stage), 16, 1024);
      if constexpr (!FP8) {  // statements of four products: one 64-column chunk each
        constexpr int kC = kSubTile / 16;
        static_assert(L::kQKSteps % 4 == 0 && L::kQKSteps <= 12, "K steps per S product");
        mma_ss_x4<0, 2, 4, 6>(tmem + t * 256, da, db, kIdescQK, 0u);
        if constexpr (L::kQKSteps >= 8) mma_ss_x4<kC, kC + 2, kC + 4, kC + 6>(tmem + t * 256, da, db, kIdescQK, 1u);
        if constexpr (L::kQKSteps >= 12)
          mma_ss_x4<2 * kC, 2 * kC + 2, 2 * kC + 4, 2 * kC + 6>(tmem + t * 256, da, db, kIdescQK, 1u);
      } else {
#pragma unroll
        for (int kk = 0; kk < L::kQKSteps; ++kk) {
          const uint32_t off = (kk / 4) * kSubTile + (kk % 4) * 32;
          mma_ss_elect_f8(tmem + t * 256, sdesc_advance(da, off), sdesc_advance(db, off), kIdescQK, kk > 0);
        }
      }
    };
    auto issue_pv = [&](int t, int stage, bool acc) {
      const uint64_t db = sdesc_sw128(sbase + L::kKVOff + L::stage_off(stage), kSubTile, 1024);
      if constexpr (!FP8) {  // two statements of four products; A: P over 8 tensor-memory columns per step
        static_assert(L::kPVSteps == 8, "K steps per P V product");
        constexpr int kBS = L::kPVKeys * 128 / 16;
        mma_ts_x4<0, kBS>(tmem + t * 256 + 128, tmem + t * 256, db, kIdescPV, acc ? 1u : 0u);
        mma_ts_x4<4, kBS>(tmem + t * 256 + 128, tmem + t * 256, db, kIdescPV, 1u);
      } else {
#pragma unroll
        for (int kk = 0; kk < L::kPVSteps; ++kk)  // A: P over 8 tensor-memory columns per step; B: kPVKeys V rows
          mma_ts_elect_f8(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, sdesc_advance(db, kk * L::kPVKeys * 128),
                          kIdescPV, (acc || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = true;
    int ld0 = 0;  // ring position of this unit's K_0
    int qn = 0;   // units started
    // parity of the P-ready phases consumed so far per tile, and whether the
    // tile's O columns still hold an output the epilogue has not read
    uint32_t pbit[NQT], obit[NQT];
    bool owed[NQT];
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
      pbit[t] = obit[t] = 0;
      owed[t] = false;
    }
    for (int r = 0; ok && r < n_rounds; ++r) {
      const int u = unit_of_round(r);
      if (u >= n_units) continue;
      const Unit w = unit_at(u);
      if (!(ok = wait_all(bar(L::kBarQFull), qn & 1, kWhereMmaQ))) break;
      ++qn;
      if (w.nkv_max > 0) {
        if (!(ok = wait_load(ld0))) break;
#pragma unroll
        for (int t = 0; t < NQT; ++t)
          if (w.nkv[t] > 0) {
            issue_qk(t, L::stage_of(ld0));
            tc_commit_elect(bar(L::kBarSFull + t));
          }
        tc_commit_elect(bar(L::kBarKVEmpty + L::stage_of(ld0)));
        // Q may be reloaded for the next unit once this unit's last S
        // products complete (here, or inside the loop below)
        if (PERSIST && w.nkv_max == 1) tc_commit_elect(bar(L::kBarQEmpty));
      }
      // O_t is overwritten by this unit's first P V product: the previous
      // unit's epilogue must have read it out
#pragma unroll
      for (int t = 0; t < NQT; ++t)
        if (PERSIST && ok && owed[t] && w.nkv[t] > 0) {
          ok = wait_all(bar(L::kBarOFree + t), obit[t], kWhereMmaO);
          obit[t] ^= 1;
          owed[t] = false;
        }
      if (!ok) break;
      // the steady-state loop (as for a single unit; ring positions and
      // phases offset by this unit's start)
      for (int j = 0; ok && j < w.nkv_max; ++j) {
        const int ldv = ld0 + 2 * j + 1;
        const int ldk = ldv + 1;
        if (!(ok = wait_load(ldv))) break;
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, j, 0);
        bool k_ready = false;
        constexpr bool kEarlyV = L::kSplitKV || L::kStages <= 2;
        int last_pv = 0;  // the last tile whose P V product reads V_j
#pragma unroll
        for (int t = 0; t < NQT; ++t)
          if (j < w.nkv[t]) last_pv = t;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (ok && j < w.nkv[t]) {
            ok = wait_all(bar(L::kBarPFull + t), pbit[t] ^ (j & 1), kWhereMmaP);
            if (lane == 0) ATTN_TRACE_AT(blockIdx.x, j, 1 + 4 * t);
            if (ok) {
              issue_pv(t, L::stage_of(ldv), j > 0);
              tc_commit_elect(bar(L::kBarODone + t));
              // With a two-stage ring (d_qk = 192) V_j's stage is released
              // as soon as its last P V product completes (the commit tracks
              // the products issued so far, not the next S products), so
              // V_{j+1} loads a product earlier: measured +10-12 % at 16K.
              // With four stages the later release is hidden, and the extra
              // commit between the products measured ~1 % slower.
              if (kEarlyV && t == last_pv) tc_commit_elect(bar(L::kBarKVEmpty + L::stage_of(ldv)));
              if (lane == 0) ATTN_TRACE_AT(blockIdx.x, j, 2 + 4 * t);
            }
          }
          if (ok && j + 1 < w.nkv[t]) {
            if (!k_ready) {
              ok = k_ready = wait_load(ldk);
              if (lane == 0) ATTN_TRACE_AT(blockIdx.x, j, 3);
            }
            if (ok) {
              issue_qk(t, L::stage_of(ldk));
              tc_commit_elect(bar(L::kBarSFull + t));
              if (lane == 0) ATTN_TRACE_AT(blockIdx.x, j, 4 + 4 * t);
            }
          }
        }
        if (!ok) break;
        if (PERSIST && j + 2 == w.nkv_max) tc_commit_elect(bar(L::kBarQEmpty));
        if (!kEarlyV) tc_commit_elect(bar(L::kBarKVEmpty + L::stage_of(ldv)));
        if (k_ready) tc_commit_elect(bar(L::kBarKVEmpty + L::stage_of(ldk)));
      }
      if (!ok) break;
      if (PERSIST && w.nkv_max == 0) tc_commit_elect(bar(L::kBarQEmpty));
#pragma unroll
      for (int t = 0; t < NQT; ++t)
        if (w.nkv[t] > 0) {
          pbit[t] ^= (uint32_t)(w.nkv[t] & 1);
          owed[t] = true;
        }
      ld0 += 2 * w.nkv_max;
    }
    // every product issued above completes before tensor memory is freed
    tc_commit_elect(bar(L::kBarMmaDone));
    mbar_wait_drain(bar(L::kBarMmaDone), 0, p.timeout_ns);
    __syncwarp();
   }
#ifdef ATTN_TRACE
   else if (warp == 2) {
    // debug only: completion times of the product groups, seen by polling
    if (lane == 0 && blockIdx.x < kTraceCtas && unit_of_round(0) < n_units) {
      const Unit w0 = unit_at(unit_of_round(0));  // the first unit only
      bool live = true;
      auto seen = [&](uint32_t b, uint32_t par) {
        for (int i = 0; live && i < (1 << 22); ++i)
          if (mbar_test(b, par)) return;
        live = false;
      };
      for (int j = 0; live && j < w0.nkv_max && j < kTraceIters; ++j)
        for (int t = 0; t < NQT; ++t) {
          if (j < w0.nkv[t]) {
            seen(bar(L::kBarODone + t), j & 1);
            ATTN_TRACE_AT(blockIdx.x, j, 16 + 2 * t);
          }
          if (j + 1 < w0.nkv[t]) {
            seen(bar(L::kBarSFull + t), (j + 1) & 1);
            ATTN_TRACE_AT(blockIdx.x, j, 17 + 2 * t);
          }
        }
    }
    __syncwarp();
   } else if (warp == 3) {
    // debug only: landing times of the K_j / V_j tiles
    if (lane == 0 && blockIdx.x < kTraceCtas && unit_of_round(0) < n_units) {
      const Unit w0 = unit_at(unit_of_round(0));  // the first unit only
      bool live = true;
      for (int ld = 0; live && ld < 2 * w0.nkv_max && ld / 2 < kTraceIters; ++ld) {
        int i = 0;
        for (; i < (1 << 22); ++i)
          if (mbar_test(bar(L::kBarKVFull + L::stage_of(ld)), L::phase_of(ld))) break;
        live = i < (1 << 22);
        ATTN_TRACE_AT(blockIdx.x, ld / 2, 20 + (ld & 1));
      }
    }
    __syncwarp();
   }
#endif
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kSmRegs));
    // ====================== softmax warpgroups =======================
    const int t = (warp - 4) >> 2;
    const int quad = warp & 3;  // this warp may touch tensor-memory lanes 32*quad .. 32*quad+31
    const uint32_t tS = tmem + ((uint32_t)(quad * 32) << 16) + t * 256;
    const uint32_t tO = tS + 128;
    // FP8: 2^(8 - tau) P is stored (P <= 2^tau against the stale max), so
    // the exponent is taken against m - (8 - tau)
    const float kPOff = FP8 ? p.p_off : 0.f;
    unsigned rescales = 0;
    bool ok = true;
    uint32_t cbit = 0;  // parity of the S / P / O-done phases of this tile in earlier units
    for (int r = 0; ok && r < n_rounds; ++r) {
    const int u = unit_of_round(r);
    if (u >= n_units) continue;
    const Unit w = unit_at(u);
    const int n = w.nkv[t];
    if constexpr (MASK) {
      // a live tile whose rows see no key at all: O = 0, LSE = -inf
      const int qt = w.qblock * NQT + t;
      const int q_row = qt * kTile + quad * 32 + lane;
      if (n == 0 && qt < p.n_qtiles && q_row < p.N) {
        uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)w.bh * p.N + q_row) * DV);
#pragma unroll
        for (int c = 0; c < DV / 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
        p.lse[(size_t)w.bh * p.N + q_row] = -INFINITY;
      }
    }
    if (n == 0) continue;
    const int bh = w.bh;
    const int qt = w.qblock * NQT + t;
    const int q_row = qt * kTile + quad * 32 + lane;
    int kt = w.j0;  // key tile of step j
    float m = -INFINITY;  // running (possibly stale) max, log2 units
    float l = 0.f;        // running sum of 2^(s*c - m + kPOff)
    // FP8: the scores carry the query tile's and the key tile's scales
    const float c_q = FP8 ? p.scale_log2 * p.sq[(size_t)bh * p.n_qtiles + qt] : p.scale_log2;
    for (int j = 0; j < n; ++j, kt = MASK ? mask_next_key_tile(p.mask, qt, kt) : kt + 1) {
      const float c_log2 = FP8 ? c_q * p.sk[(size_t)bh * n_kv_tiles + kt] : c_q;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull + t), cbit ^ (j & 1), ctl, kWhereSmS));
      if (!ok) break;
      if (quad == 0 && lane == 0) ATTN_TRACE_AT(blockIdx.x, j, 9 + 2 * t);
      tc_fence_after();
      float s[128];
      if constexpr (NQT == 1) {  // 128 registers per thread: load in 32-column pieces
        tmem_ld32p(tS + 0, s + 0);
        tmem_ld32p(tS + 32, s + 32);
        tmem_ld32p(tS + 64, s + 64);
        tmem_ld32p(tS + 96, s + 96);
      } else {
        tmem_ld128(tS, s);
      }
      const int kbase = kt * kTile;
      if constexpr (MASK) {
        if (!mask_tile_full(p.mask, qt, kt)) {
          // keys lo .. hi are visible from this row
          const int lo = p.mask.left >= 0 ? q_row - p.mask.left : 0;
          const int hi = p.mask.right >= 0 ? min(q_row + p.mask.right, p.N - 1) : p.N - 1;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (kbase + c < lo || kbase + c > hi) s[c] = -INFINITY;
        }
      } else if ((CAUSAL && j == qt) || kbase + kTile > n_keys) {
        const int lim = CAUSAL ? min(q_row + 1, p.N) : n_keys;  // keys < lim are visible
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (kbase + c >= lim) s[c] = -INFINITY;
      }
      // row max with three-input max: eight independent chains, two new
      // scores per instruction
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmax3(s[i], s[i + 8], s[i + 16]);
#pragma unroll
      for (int c = 24; c < 120; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + i + 8]);
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[120 + i]);
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      if (t == 0 && quad == 0 && lane == 0) ATTN_TRACE_AT(blockIdx.x, j, 15);
      const float m_new = fmaxf(m, mx * c_log2);
      const bool need = m_new > m + p.tau;
      if (__any_sync(0xffffffffu, need)) {
        // the warp moves every row to its current max (valid for all rows,
        // since m_new >= m), so tensor-memory traffic stays warp-uniform
        const float alpha = (m == -INFINITY) ? 0.f : ex2_mufu(m - m_new);
        rescales += (j > 0 && need) ? 1u : 0u;
        l *= alpha;
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarODone + t), cbit ^ ((j - 1) & 1), ctl, kWhereSmO));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < DV; c0 += 32) {
            float o[32];
            tmem_ld32(tO + c0, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tO + c0, o);
          }
        }
        m = m_new;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      // x = s * scale * log2(e) - m on pairs (packed FP32 FMA), then 2^x
      const float2 c2 = make_float2(c_log2, c_log2);
      const float2 nm2 = make_float2(kPOff - m_use, kPOff - m_use);
      float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      if constexpr (FP8) {
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float2 x0 = __ffma2_rn(make_float2(s[c0 + i], s[c0 + i + 1]), c2, nm2);
            const float2 x1 = __ffma2_rn(make_float2(s[c0 + i + 2], s[c0 + i + 3]), c2, nm2);
            const float2 e0 = make_float2(i < POLY ? ex2_poly3(x0.x) : ex2_mufu(x0.x),
                                          i + 1 < POLY ? ex2_poly3(x0.y) : ex2_mufu(x0.y));
            const float2 e1 = make_float2(i + 2 < POLY ? ex2_poly3(x1.x) : ex2_mufu(x1.x),
                                          i + 3 < POLY ? ex2_poly3(x1.y) : ex2_mufu(x1.y));
            ls[(i >> 2) & 3] = __fadd2_rn(ls[(i >> 2) & 3], __fadd2_rn(e0, e1));
            pk[i >> 2] = pack_e4m3x4(e0.x, e0.y, e1.x, e1.y);
          }
          tmem_st8(tS + c0 / 4, pk);  // P (e4m3, four per column) over the first 32 columns of S
        }
      } else {
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = __ffma2_rn(make_float2(s[c0 + i], s[c0 + i + 1]), c2, nm2);
          const float e0 = (i < POLY) ? ex2_poly3(x.x) : ex2_mufu(x.x);
          const float e1 = (i + 1 < POLY) ? ex2_poly3(x.y) : ex2_mufu(x.y);
          ls[(i >> 1) & 3] = __fadd2_rn(ls[(i >> 1) & 3], make_float2(e0, e1));
          pk[i >> 1] = pack_bf16(e0, e1);
        }
        tmem_st16(tS + c0 / 2, pk);  // P (bf16 pairs) over the first 64 columns of S
      }
      }
      const float2 lsum = __fadd2_rn(__fadd2_rn(ls[0], ls[1]), __fadd2_rn(ls[2], ls[3]));
      l += lsum.x + lsum.y;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::kBarPFull + t));
      if (quad == 0 && lane == 0) ATTN_TRACE_AT(blockIdx.x, j, 10 + 2 * t);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarODone + t), cbit ^ ((n - 1) & 1), ctl, kWhereSmFinal));
    // the four warps of the warpgroup agree (the epilogue's named barriers
    // need all of them, and after a timeout all of them leave together)
    ok = named_bar_and(1 + t, 128, ok);
    {
      if (ok) {
        tc_fence_after();
        const float inv_l = l > 0.f ? (FP8 ? p.sv[bh] : 1.f) / l : 0.f;
        const bool live = q_row < p.N;
        if constexpr (SPLIT) {  // this key range's normalised output and LSE, FP32
          const size_t prow = ((size_t)w.split * p.BH + bh) * p.N + (live ? q_row : 0);
          float4* orow4 = reinterpret_cast<float4*>(p.o_part + prow * DV);
#pragma unroll
          for (int c0 = 0; c0 < DV; c0 += 32) {
            float o[32];
            tmem_ld32(tO + c0, o);
            if (live) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                orow4[c0 / 4 + v] = make_float4(o[4 * v] * inv_l, o[4 * v + 1] * inv_l, o[4 * v + 2] * inv_l,
                                                o[4 * v + 3] * inv_l);
            }
          }
          if (PERSIST) {
            tc_fence_before();
            mbar_arrive(bar(L::kBarOFree + t));
          }
          if (live) p.lse_part[prow] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
          float o[DV];
#pragma unroll
          for (int c0 = 0; c0 < DV; c0 += 32) tmem_ld32p(tO + c0, o + c0);
          // O_t has been read out: the next unit's products may overwrite it
          if (PERSIST) {
            tc_fence_before();
            mbar_arrive(bar(L::kBarOFree + t));
          }
          // O / l as bf16, one 64-column box at a time: each thread writes its
          // row into the staging tile in the 128-byte swizzled layout (16-byte
          // unit c of row r at unit c ^ (r % 8): a quarter warp covers all 32
          // banks), then one thread hands the box to the copy engine, whose
          // TMA store writes whole rows to global memory and leaves out the
          // rows past N.  The staging tile is reused once the previous box's
          // store has read it.
          // Without persistent CTAs the tile's Q region is free by now (its
          // last S product has completed) and, when it holds all of O's
          // boxes, takes them side by side: no box waits for another's store.
          constexpr bool kInQ = !PERSIST && L::kQBytes >= DV * kTile * 2;
          static_assert(kInQ || !L::kSplitKV, "split K/V rings leave no O staging tile");
          constexpr uint32_t kBoxStride = kInQ ? kTile * 128 : 0;
          const uint32_t s_off = kInQ ? (uint32_t)(t * L::kQBytes) : (uint32_t)(L::kStgOff + t * L::kStgBytes);
          const int r_in = quad * 32 + lane;
          const bool issuer = quad == 0 && lane == 0;
#pragma unroll
          for (int b = 0; b < DV / 64; ++b) {
            uint8_t* srow = smem + s_off + b * kBoxStride + r_in * 128;
            if (!kInQ) {  // the previous box's store has read the staging tile
              if (issuer) bulk_wait_read<0>();
              named_bar_sync(1 + t, 128);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const float* v = o + b * 64 + 8 * c;
              *reinterpret_cast<uint4*>(srow + ((c ^ (r_in & 7)) * 16)) =
                  make_uint4(pack_bf16(v[0] * inv_l, v[1] * inv_l), pack_bf16(v[2] * inv_l, v[3] * inv_l),
                             pack_bf16(v[4] * inv_l, v[5] * inv_l), pack_bf16(v[6] * inv_l, v[7] * inv_l));
            }
            if (!kInQ || b == DV / 64 - 1) {
              fence_proxy_async_smem();
              named_bar_sync(1 + t, 128);
              if (issuer) {
                for (int bb = kInQ ? 0 : b; bb <= b; ++bb)
                  tma_store_3d(&p.tm_o, sbase + s_off + bb * kBoxStride, bb * 64, qt * kTile, bh);
                bulk_commit();
              }
            }
          }
          if (live)
            p.lse[(size_t)bh * p.N + q_row] = l > 0.f ? (m - kPOff + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
      }
    }
    cbit ^= (uint32_t)(n & 1);
    }  // units
    // the epilogue's TMA stores have read the staging tile before the CTA
    // exits (their global writes complete on their own)
    if (quad == 0 && lane == 0) bulk_wait_read<0>();
    __syncwarp();
    if (p.rescale_counter != nullptr) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) rescales += __shfl_xor_sync(0xffffffffu, rescales, off);
      if (lane == 0 && rescales) atomicAdd(p.rescale_counter, (unsigned long long)rescales);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Split-KV forward (persistent, non-causal, hardware exponentials) followed
// by the merge kernel (attn_merge.cuh).
template <int DQK, int DV, int NQT>
cudaError_t launch_fwd_split_instance(const FwdParams& p, cudaStream_t stream) {
  using L = FwdLayout<DQK, DV, NQT>;
  auto kernel = fwd_kernel<DQK, DV, NQT, false, 0, true, true>;
  int sms = 0;
  cudaError_t e = prepare_kernel((const void*)kernel, L::kSmemBytes, L::kLaunchRegs, &sms);
  if (e != cudaSuccess) return e;
  int grid = sms * L::kMinBlocks;
  if (grid > p.n_blocks) grid = p.n_blocks;
  kernel<<<grid, L::kThreads, L::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int DQK, int DV, int NQT, bool CAUSAL, int POLY, bool FP8 = false, bool MASK = false>
cudaError_t launch_fwd_instance(const FwdParams& p, cudaStream_t stream) {
  using L = FwdLayout<DQK, DV, NQT, FP8 ? 1 : 2>;
  constexpr bool kKV21 = DQK == 192 && !FP8 && !MASK;  // the one-unit-per-CTA instance's split rings
  using L1 = FwdLayout<DQK, DV, NQT, FP8 ? 1 : 2, kKV21 ? 2 : 0, kKV21 ? 1 : 0>;
  // Persistent CTAs pay off when units are short (few K/V tiles each); with
  // long units the one-unit-per-CTA kernel is leaner and the launch order
  // already balances.  p.max_ctas > 0 forces the persistent grid.
  const bool persist = p.max_ctas > 0 || p.persist;
  auto kernel = persist ? fwd_kernel<DQK, DV, NQT, CAUSAL, POLY, true, false, FP8, MASK>
                        : fwd_kernel<DQK, DV, NQT, CAUSAL, POLY, false, false, FP8, MASK>;
  // setmaxnreg.inc waits until the registers it asks for are free, so the
  // split must add up to what the launch actually hands out
  int sms = 0;
  const int smem = persist ? L::kSmemBytes : L1::kSmemBytes;
  cudaError_t e = prepare_kernel((const void*)kernel, smem, L::kLaunchRegs, &sms);
  if (e != cudaSuccess) return e;
  // persistent grid: as many CTAs as fit on the device at once, each looping
  // over work units (p.max_ctas > 0 sets the grid instead, e.g. one unit per
  // CTA when it is at least the number of units)
  int grid = !persist ? p.n_blocks : p.max_ctas > 0 ? p.max_ctas : sms * L::kMinBlocks;
  if (grid > p.n_blocks) grid = p.n_blocks;
  kernel<<<grid, L::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
