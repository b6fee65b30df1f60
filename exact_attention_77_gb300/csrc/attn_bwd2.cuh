// Backward attention kernel on CTA pairs for sm_103a, d = 128 (template;
// instantiated in attn_bwd_d128.cu).
//
// What it computes: the same dQ, dK, dV as the one-CTA kernel in
// attn_bwd.cuh (five products and two elementwise steps per key tile x
// query tile, "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design
// for Asymmetric Hardware Scaling", Figure 2), with the pairing of the
// backward's 2-CTA mode (same paper, Table 3 and Figure 3): two CTAs of a
// cluster take key tiles j0 = 2p and j1 = 2p + 1 of one head and walk the
// query tiles together; every product is one tcgen05.mma.cta_group::2
// issued by the even CTA, with M = 256 (each CTA's 128 keys) for S^T, dP^T,
// dV and dK, so each CTA reads only half of the B operand from its shared
// memory; and dQ of the query tile is one M = 128 pair product whose
// reduction runs over both key tiles (256 keys), after each CTA has written
// the half of its dS that the other needs into the other's shared memory.
// The pair thus reads a quarter less operand data from shared memory per
// tile and writes half as many dQ partials.
//
// The pair product shares its K dimension between the two CTAs (only A's
// rows and B's columns are split), so both CTAs keep every operand in the
// same natural order at the same shared-memory offsets.  Per CTA r (own
// queries 64r..64r+63, own d-half r):
//   K, V         this CTA's key tile, [d 0..63 | d 64..127]       (S^T, dP^T: A)
//   KQ           both key tiles' rows, own d-half                 (dQ: B)
//   QA, dOA      own 64 queries, [d 0..63 | d 64..127]            (S^T, dP^T: B)
//   QB, dOB      all 128 queries, own d-half                      (dK, dV: B)
//   dS           both key tiles' rows x own 64 queries            (dQ: A)
// Each of QA, QB, dOA, dOB has one stage with its own full / empty
// barriers: a part is reloaded for the next query tile as soon as its one
// product has read it, about a tile ahead of its next use.
//
// Roles (512 threads): warp 0 loads (own CTA); warp 1 of the even CTA issues
// every product; warp 2 of the odd CTA relays its load completions to the
// even CTA; warp 3 moves the other CTA's dS half with the copy engine and (odd
// CTA) relays the compute signals, so the compute warps only ever touch their
// own CTA's memory (measured: a cluster-scope release arrive or remote store
// from a compute warp stalled it ~900 cycles); two compute warpgroups (keys on
// tensor-memory lanes, warpgroup h takes queries 64h..64h+63); one dQ
// warpgroup (reads this CTA's 64 dQ rows, has the copy engine add them into
// the FP32 accumulator).
//
// Every wait is bounded; a timeout raises the CTA's abort flag and every
// role falls through to the teardown, which both CTAs of a pair always reach.
#pragma once

#include "attn_bwd.cuh"

namespace attn {

// ------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t mapa_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// arrive on an mbarrier given by its shared::cluster address.  Used only by
// the relay threads, each after it has waited for the local phase that
// records the work as complete (copies landed, tensor-memory stores or loads
// waited for with tcgen05.wait, shared-memory writes fenced to the async
// proxy); relaxed, since a cluster-scope release measured about a thousand
// cycles per arrive on GB300 and serialised the relays.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait with cluster-scope acquire, for phases the other CTA of the pair
// may complete.  It polls with test_wait: measured on GB300, a thread
// suspended in try_wait on such a phase woke a thousand or more cycles after
// a remote arrive completed it.
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, const WaitCtl& ctl, int where) {
  if (mbar_test_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_test_cluster(bar, parity)) return true;
    if (*ctl.abort) return false;
    if (globaltimer_ns() - t0 > ctl.timeout_ns) {
      *ctl.abort = 1;
      report_error(ctl.status, ATTN_ERR_TIMEOUT, where);
      return false;
    }
  }
}

// copy engine: bytes of this CTA's shared memory into the other CTA's,
// completing the transaction count of the barrier at dst_bar (other CTA)
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                  uint32_t dst_bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(src_cta), "r"(bytes), "r"(dst_bar_cluster)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_cluster() {
  asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] B[smem] over the pair: A rows split by CTA (M/2 each),
// B's N columns split by CTA (N/2 each), D rows in each CTA's tensor memory
__device__ __forceinline__ void mma_pair_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// elect.sync forms for an issue loop the whole warp runs in step
__device__ __forceinline__ void mma_pair_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_pair_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
          bar),
      "h"((uint16_t)3)
      : "memory");
}

// the same with A read from each CTA's tensor memory
__device__ __forceinline__ void mma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// arrive on the barrier at this shared-memory offset in both CTAs once every
// product issued so far completes
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

// ------------------------------------------------------------------ layout
struct Bwd2Layout {
  static constexpr int D = 128;
  static constexpr int kHalf = 64 * 128;   // 8 KiB: 64 rows x one 128-byte d-half
  static constexpr int kSub = 128 * 128;   // 16 KiB: 128 rows x one d-half
  static constexpr int kKOff = 0;          // K_j: [d-half 0 | d-half 1]
  static constexpr int kVOff = kKOff + 2 * kSub;
  static constexpr int kKQOff = kVOff + 2 * kSub;  // key tiles 2p, 2p+1 x own d-half
  static constexpr int kQAOff = kKQOff + 2 * kSub;  // own queries: [d-half 0 | d-half 1]
  static constexpr int kQBOff = kQAOff + kSub;      // all queries x own d-half
  static constexpr int kOAOff = kQBOff + kSub;
  static constexpr int kOBOff = kOAOff + kSub;
  static constexpr int kDSOff = kOBOff + kSub;      // 256 key rows x own 64 queries (MN-major)
  static constexpr int kDSXOff = kDSOff + 2 * kSub;  // own keys x the other CTA's 64 queries
  static constexpr int kStgOff = kDSXOff + kSub;      // dQ staging: own 64 rows x one d-half, fp32
  static constexpr int kStgBytes = 16 * 1024;
  static constexpr int kVecOff = kStgOff + kStgBytes;  // per buffer: -LSE2[128], -D[128]
  static constexpr int kVecBytes = 2 * 128 * 4;
  static constexpr int kBarOff = kVecOff + 2 * kVecBytes;
  enum : int {
    kBarKV = 0,     // K, V, KQ landed
    kBarQAFull, kBarQAEmpty, kBarQBFull, kBarQBEmpty,
    kBarOAFull, kBarOAEmpty, kBarOBFull, kBarOBEmpty,
    kBarVecFull,    // + buffer
    kBarSFull = kBarVecFull + 2, kBarDPFull,
    kBarPReady,     // + half: P^T half in tensor memory (8 warp arrivals)
    kBarDSFull = kBarPReady + 2,  // + half: dS^T half in tensor memory (8 warp arrivals)
    kBarDSmem = kBarDSFull + 2,   // dS written to shared memory (8 warp arrivals)
    kBarDSIn,       // the other CTA's dS half copied in (transaction count + 1 arrival)
    kBarDQFull, kBarDQFree,       // DQFree: 4 warp arrivals
    kBarAccDone,
    // even CTA only: the odd CTA's loads and signals, relayed
    kBarKVPeer, kBarQAPeer, kBarQBPeer, kBarOAPeer, kBarOBPeer,
    kBarPReadyPeer, kBarDSFullPeer = kBarPReadyPeer + 2, kBarDSBufPeer = kBarDSFullPeer + 2, kBarDQFreePeer,
    kBarStgFull,    // 128 arrivals
    kBarStgFree,
    kNumBars
  };
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static constexpr int kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
  static constexpr int kColDQ = 128;  // 64 columns; shares the dP^T columns
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128;
  static constexpr int kCtlRegs = 112;
  static constexpr int kComputeRegs = 128;
  static constexpr int kDqRegs = 144;
  static_assert(kCtlRegs * 128 + kComputeRegs * 256 + kDqRegs * 128 <= kLaunchRegs * kThreads, "register split");
};

template <bool CAUSAL, bool DETERMINISTIC>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(512, 1)
    bwd2_kernel(const __grid_constant__ BwdParams p) {
  using L = Bwd2Layout;
  constexpr int D = L::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  const int own = (int)rank;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };
  auto bar0 = [&](int i) -> uint32_t { return mapa_rank(sbase + L::kBarOff + 8u * i, 0); };  // the even CTA's
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  // work unit: key-tile pair pr of head bh; this CTA takes key tile 2pr + rank
  const int n = p.n_tiles;
  const int n_pairs = (n + 1) >> 1;
  const int unit = blockIdx.x >> 1;
  int pr, bh;
  if (DETERMINISTIC) {  // pair-major: a CTA waits only on pairs launched before it
    pr = unit / p.BH;
    bh = unit - pr * p.BH;
  } else {  // head-major: resident CTAs share one or two heads' dQ accumulators in L2
    bh = unit / n_pairs;
    pr = unit - bh * n_pairs;
  }
  const int j = 2 * pr + own;  // own key tile (== n for the odd CTA of a ragged last pair: no keys)
  const int i_lo = CAUSAL ? 2 * pr : 0;  // both CTAs walk query tiles n-1 .. i_lo together
  const int n_it = n - i_lo;
  auto tile_of = [&](int it) { return n - 1 - it; };

  if (threadIdx.x == 0) {
    for (int b = 0; b < L::kNumBars; ++b) {
      uint32_t cnt = 1;
      if (b == L::kBarPReady || b == L::kBarPReady + 1 || b == L::kBarDSFull || b == L::kBarDSFull + 1 ||
          b == L::kBarDSmem)
        cnt = 8;
      if (b == L::kBarDQFree) cnt = 4;
      if (b == L::kBarStgFull) cnt = 128;
      mbar_init(bar(b), cnt);
    }
    *abort_flag = (sbase & 1023u) ? 1 : 0;  // swizzled tiles need 1024-byte alignment
    if (sbase & 1023u) report_error(p.status, ATTN_ERR_BOUNDS, 3);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or pair commit
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool live_cta = *abort_flag == 0;

  if (warp < 4) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(L::kCtlRegs));
   if (warp == 0) {
    // ============================ producer ============================
    if (lane == 0 && live_cta) {
      prefetch_tensormap(&p.tm_q_half);
      prefetch_tensormap(&p.tm_do_half);
      prefetch_tensormap(&p.tm_q);
      prefetch_tensormap(&p.tm_do);
      prefetch_tensormap(&p.tm_k);
      prefetch_tensormap(&p.tm_v);
      mbar_arrive_expect_tx(bar(L::kBarKV), 6 * L::kSub);
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(sbase + L::kKOff + c * L::kSub, &p.tm_k, 64 * c, j * kBTile, bh, bar(L::kBarKV));
        tma_load_3d(sbase + L::kVOff + c * L::kSub, &p.tm_v, 64 * c, j * kBTile, bh, bar(L::kBarKV));
        tma_load_3d(sbase + L::kKQOff + c * L::kSub, &p.tm_k, 64 * own, (2 * pr + c) * kBTile, bh, bar(L::kBarKV));
      }
      int issued = 0;
      bool ok = true;
      for (int it = 0; ok && it < n_it; ++it) {
        const int i = tile_of(it);
        const uint32_t pe = (it & 1) ^ 1;  // parity of the empty phase to wait for (it > 0)
        // QA + vec (after the previous S^T)
        if (it > 0 && !(ok = mbar_wait_cl(bar(L::kBarQAEmpty), pe, ctl, kBWhereProd))) break;
        ATTN_TRACE_AT(blockIdx.x, it, 13);
        mbar_arrive_expect_tx(bar(L::kBarQAFull), L::kSub);
        tma_load_3d(sbase + L::kQAOff, &p.tm_q_half, 0, i * kBTile + 64 * own, bh, bar(L::kBarQAFull));
        tma_load_3d(sbase + L::kQAOff + L::kHalf, &p.tm_q_half, 64, i * kBTile + 64 * own, bh, bar(L::kBarQAFull));
        const int vb = it & 1;
        const size_t vrow = (size_t)bh * p.Npad + (size_t)i * kBTile;
        mbar_arrive_expect_tx(bar(L::kBarVecFull + vb), L::kVecBytes);
        bulk_load(sbase + L::kVecOff + vb * L::kVecBytes, p.row_lse2 + vrow, kBTile * 4, bar(L::kBarVecFull + vb));
        bulk_load(sbase + L::kVecOff + vb * L::kVecBytes + kBTile * 4, p.row_d + vrow, kBTile * 4,
                  bar(L::kBarVecFull + vb));
        // dOA (after the previous dP^T)
        if (it > 0 && !(ok = mbar_wait_cl(bar(L::kBarOAEmpty), pe, ctl, kBWhereProd + 1))) break;
        mbar_arrive_expect_tx(bar(L::kBarOAFull), L::kSub);
        tma_load_3d(sbase + L::kOAOff, &p.tm_do_half, 0, i * kBTile + 64 * own, bh, bar(L::kBarOAFull));
        tma_load_3d(sbase + L::kOAOff + L::kHalf, &p.tm_do_half, 64, i * kBTile + 64 * own, bh, bar(L::kBarOAFull));
        // dOB (after the previous dV)
        if (it > 0 && !(ok = mbar_wait_cl(bar(L::kBarOBEmpty), pe, ctl, kBWhereProd + 2))) break;
        mbar_arrive_expect_tx(bar(L::kBarOBFull), L::kSub);
        tma_load_3d(sbase + L::kOBOff, &p.tm_do, 64 * own, i * kBTile, bh, bar(L::kBarOBFull));
        // QB (after the previous dK)
        if (it > 0 && !(ok = mbar_wait_cl(bar(L::kBarQBEmpty), pe, ctl, kBWhereProd + 3))) break;
        ATTN_TRACE_AT(blockIdx.x, it, 14);
        mbar_arrive_expect_tx(bar(L::kBarQBFull), L::kSub);
        tma_load_3d(sbase + L::kQBOff, &p.tm_q, 64 * own, i * kBTile, bh, bar(L::kBarQBFull));
        issued = it + 1;
      }
      // copies in flight land before the CTA exits
      mbar_wait_drain(bar(L::kBarKV), 0, p.timeout_ns);
      if (issued > 0) {
        const uint32_t pl = (issued - 1) & 1;
        mbar_wait_drain(bar(L::kBarQAFull), pl, p.timeout_ns);
        mbar_wait_drain(bar(L::kBarOAFull), pl, p.timeout_ns);
        mbar_wait_drain(bar(L::kBarOBFull), pl, p.timeout_ns);
        mbar_wait_drain(bar(L::kBarQBFull), pl, p.timeout_ns);
        mbar_wait_drain(bar(L::kBarVecFull + ((issued - 1) & 1)), ((issued - 1) >> 1) & 1, p.timeout_ns);
        if (issued > 1) mbar_wait_drain(bar(L::kBarVecFull + (issued & 1)), ((issued - 2) >> 1) & 1, p.timeout_ns);
      }
    }
    __syncwarp();
   } else if (warp == 2 && rank == 1) {
    // ============ relay: the odd CTA's loads, announced to the even CTA ============
    if (lane == 0 && live_cta) {
      bool ok = mbar_wait_cl(bar(L::kBarKV), 0, ctl, kBWhereProd + 4);
      if (ok) mbar_arrive_cluster(bar0(L::kBarKVPeer));
      for (int it = 0; ok && it < n_it; ++it) {
        const uint32_t pf = it & 1;
        if (!(ok = mbar_wait_cl(bar(L::kBarQAFull), pf, ctl, kBWhereProd + 5))) break;
        mbar_arrive_cluster(bar0(L::kBarQAPeer));
        ATTN_TRACE_AT(blockIdx.x, it, 15);
        if (!(ok = mbar_wait_cl(bar(L::kBarOAFull), pf, ctl, kBWhereProd + 6))) break;
        mbar_arrive_cluster(bar0(L::kBarOAPeer));
        if (!(ok = mbar_wait_cl(bar(L::kBarOBFull), pf, ctl, kBWhereProd + 7))) break;
        mbar_arrive_cluster(bar0(L::kBarOBPeer));
        if (!(ok = mbar_wait_cl(bar(L::kBarQBFull), pf, ctl, kBWhereProd + 8))) break;
        mbar_arrive_cluster(bar0(L::kBarQBPeer));
      }
    }
    __syncwarp();
   } else if (warp == 3) {
    // ===== signals: dS exchange (both CTAs); the odd CTA's compute signals, relayed =====
    // The compute warps only touch this CTA's memory; this thread moves the
    // other CTA's dS half with the copy engine and forwards the odd CTA's
    // readiness to the even CTA (whose thread issues the products).
    if (lane == 0 && live_cta) {
      bool ok = true;
      const uint32_t peer = 1u - rank;
      for (int it = 0; ok && it < n_it; ++it) {
        const uint32_t pf = it & 1;
        if (own == 1) {
#pragma unroll
          for (int m = 0; m < 2 && ok; ++m) {
            if (!(ok = mbar_wait_cl(bar(L::kBarPReady + m), pf, ctl, kBWhereEw + 6))) break;
            mbar_arrive_cluster(bar0(L::kBarPReadyPeer + m));
            if (m == 0) ATTN_TRACE_AT(blockIdx.x, it, 28);
          }
#pragma unroll
          for (int m = 0; m < 2 && ok; ++m) {
            if (!(ok = mbar_wait_cl(bar(L::kBarDSFull + m), pf, ctl, kBWhereEw + 7))) break;
            mbar_arrive_cluster(bar0(L::kBarDSFullPeer + m));
            if (m == 1) ATTN_TRACE_AT(blockIdx.x, it, 29);
          }
          if (!ok) break;
        }
        // this iteration's incoming half: one local arrival plus its bytes
        mbar_arrive_expect_tx(bar(L::kBarDSIn), L::kSub);
        if (!(ok = mbar_wait_cl(bar(L::kBarDSmem), pf, ctl, kBWhereEw + 8))) break;
        // own keys x the other CTA's queries -> its dS rows 128*rank ..
        bulk_copy_to_peer(mapa_rank(sbase + L::kDSOff + (uint32_t)own * L::kSub, peer), sbase + L::kDSXOff, L::kSub,
                          mapa_rank(bar(L::kBarDSIn), peer));
        ATTN_TRACE_AT(blockIdx.x, it, 30);
        // the incoming half must land before the barrier is armed again
        if (!(ok = mbar_wait_cl(bar(L::kBarDSIn), pf, ctl, kBWhereEw + 9))) break;
        ATTN_TRACE_AT(blockIdx.x, it, 31);
        if (own == 1) {
          mbar_arrive_cluster(bar0(L::kBarDSBufPeer));
          if (!(ok = mbar_wait_cl(bar(L::kBarDQFree), pf, ctl, kBWhereEw + 10))) break;
          mbar_arrive_cluster(bar0(L::kBarDQFreePeer));
        }
      }
    }
    __syncwarp();
   }
#ifdef ATTN_TRACE
   else if (warp == 2 && rank == 0) {
    // debug only: completion times of the products, seen by polling
    if (lane == 0 && blockIdx.x < kTraceCtas) {
      bool live = true;
      auto seen = [&](uint32_t b, uint32_t par) {
        for (int q = 0; live && q < (1 << 22); ++q)
          if (mbar_test(b, par)) return;
        live = false;
      };
      for (int it = 0; live && it < n_it && it < kTraceIters; ++it) {
        seen(bar(L::kBarSFull), it & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 16);
        seen(bar(L::kBarDPFull), it & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 17);
        seen(bar(L::kBarOBEmpty), it & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 18);
        seen(bar(L::kBarQBEmpty), it & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 19);
        seen(bar(L::kBarDQFull), it & 1);
        ATTN_TRACE_AT(blockIdx.x, it, 20);
      }
    }
    __syncwarp();
   }
#endif
   else if (warp == 1 && rank == 0) {
    // ======================= products (even CTA) =======================
    // the whole warp runs this loop in step; elect.sync picks the issuing lane
    if (live_cta) {
      constexpr uint32_t kIdSq = idesc_bf16_f32(256, 128, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(256, 128, false, true);  // dV, dK (A in tensor memory)
      constexpr uint32_t kIdDq = idesc_bf16_f32(128, 128, true, true);    // dQ (A = dS, MN-major)
      // S^T / dP^T: A = the key tile (K-major), B = own 64 queries (K-major)
      auto mma_scores = [&](uint32_t d_col, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t da = sdesc_sw128(a_base + (kk / 4) * L::kSub, 16, 1024);
          const uint64_t db = sdesc_sw128(b_base + (kk / 4) * L::kHalf, 16, 1024);
          mma_pair_ss_elect(tmem + d_col, sdesc_advance(da, (kk % 4) * 32), sdesc_advance(db, (kk % 4) * 32), kIdSq, kk > 0);
        }
      };
      // dV / dK half m: A = P^T / dS^T (queries 64h..64h+63 packed in columns
      // 64h..64h+31), B = all queries x own d-half (MN-major)
      auto mma_acc_half = [&](uint32_t d_col, uint32_t a_col, uint32_t b_base, bool acc, int m) {
        const uint64_t db = sdesc_sw128(b_base, L::kSub, 1024);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int kk = 4 * hh + 2 * m + u;
            mma_pair_ts_elect(tmem + d_col, tmem + a_col + (kk / 4) * 64 + (kk % 4) * 8, sdesc_advance(db, kk * 2048),
                        kIdAcc, (acc || m > 0 || hh > 0 || u > 0) ? 1u : 0u);
          }
      };
      auto both = [&](int b_local, int b_peer, uint32_t parity, int where) -> bool {
        return __all_sync(0xffffffffu, mbar_wait_cl(bar(b_local), parity, ctl, where) &&
                                           mbar_wait_cl(bar(b_peer), parity, ctl, where));
      };
      bool ok = both(L::kBarKV, L::kBarKVPeer, 0, kBWhereMma);
      tc_fence_after();
      for (int it = 0; ok && it < n_it; ++it) {
        const uint32_t pf = it & 1;
        if (!(ok = both(L::kBarQAFull, L::kBarQAPeer, pf, kBWhereMma + 1))) break;
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 0);
        tc_fence_after();
        mma_scores(L::kColS, sbase + L::kKOff, sbase + L::kQAOff);
        tc_commit_pair_elect(bar(L::kBarSFull));
        tc_commit_pair_elect(bar(L::kBarQAEmpty));
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 1);
        if (!(ok = both(L::kBarOAFull, L::kBarOAPeer, pf, kBWhereMma + 3))) break;
        if (it > 0 && !(ok = both(L::kBarDQFree, L::kBarDQFreePeer, (it - 1) & 1, kBWhereMma + 2))) break;
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 2);
        tc_fence_after();
        mma_scores(L::kColDP, sbase + L::kVOff, sbase + L::kOAOff);  // runs while P is computed
        tc_commit_pair_elect(bar(L::kBarDPFull));
        tc_commit_pair_elect(bar(L::kBarOAEmpty));
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 3);
        if (!(ok = both(L::kBarOBFull, L::kBarOBPeer, pf, kBWhereMma + 4))) break;
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 4);
#pragma unroll
        for (int m = 0; m < 2 && ok; ++m) {
          if (!(ok = both(L::kBarPReady + m, L::kBarPReadyPeer + m, pf, kBWhereMma + 5))) break;
          if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 5 + m);
          tc_fence_after();
          mma_acc_half(L::kColDV, L::kColS, sbase + L::kOBOff, it > 0, m);
        }
        if (!ok) break;
        tc_commit_pair_elect(bar(L::kBarOBEmpty));
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 7);
        if (!(ok = both(L::kBarQBFull, L::kBarQBPeer, pf, kBWhereMma + 6))) break;
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 8);
#pragma unroll
        for (int m = 0; m < 2 && ok; ++m) {
          if (!(ok = both(L::kBarDSFull + m, L::kBarDSFullPeer + m, pf, kBWhereMma + 7))) break;
          if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 9 + m);
          tc_fence_after();
          mma_acc_half(L::kColDK, L::kColDP, sbase + L::kQBOff, it > 0, m);
        }
        if (!ok) break;
        tc_commit_pair_elect(bar(L::kBarQBEmpty));
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 11);
        // dQ of this query tile over both key tiles: A = dS (key rows of tile
        // 2pr, then 2pr+1), B = KQ (the same key rows x own d-half).  Both
        // CTAs' dS tiles must be complete: own rows, the copied-in rows, and
        // the odd CTA's (relayed).
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(L::kBarDSmem), pf, ctl, kBWhereMma + 8)) &&
                   both(L::kBarDSIn, L::kBarDSBufPeer, pf, kBWhereMma + 8)))
          break;
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 27);
        tc_fence_after();
        {
          const uint64_t da = sdesc_sw128(sbase + L::kDSOff, L::kSub, 1024);
          const uint64_t db = sdesc_sw128(sbase + L::kKQOff, L::kSub, 1024);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_pair_ss_elect(tmem + L::kColDQ, sdesc_advance(da, kk * 2048), sdesc_advance(db, kk * 2048), kIdDq, kk > 0);
        }
        tc_commit_pair_elect(bar(L::kBarDQFull));
        if (lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 12);
      }
      tc_commit_pair_elect(bar(L::kBarAccDone));
      mbar_wait_drain(bar(L::kBarAccDone), 0, p.timeout_ns);
    }
    __syncwarp();
   }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kComputeRegs));
    // ================= two compute warpgroups (h = 0, 1) =================
    // Keys on tensor-memory lanes; warpgroup h takes queries 64h..64h+63.
    const int h = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int lrow = quad * 32 + lane;
    const int k_glob = j * kBTile + lrow;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::kColS;
    const uint32_t tDP = tmem + lane_base + L::kColDP;
    const float c_log2 = p.scale_log2;
    const bool key_dead = k_glob >= p.N;
    // dS rows of these queries belong to CTA h (whose dQ rows they are): own
    // queries go to this CTA's dS tile at key row 128*rank + lrow, the other
    // CTA's to the local half tile that the copy engine moves over (its row
    // lrow lands on row 128*rank + lrow there; the swizzle phase is the same)
    uint8_t* ds_row = smem + (h == own ? L::kDSOff + own * L::kSub : L::kDSXOff) + (lrow >> 3) * 1024 + (lrow & 7) * 128;
    bool ok = live_cta;
    auto arrive_local = [&](int b_idx) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(b_idx));
    };
    for (int it = 0; ok && it < n_it; ++it) {
      const int i = tile_of(it);
      const int vb = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarVecFull + vb), (it >> 1) & 1, ctl, kBWhereEw + 3));
      if (!ok) break;
      const float* vec = reinterpret_cast<const float*>(smem + L::kVecOff + vb * L::kVecBytes);
      const bool diag = CAUSAL && i <= j;  // keys above the queries are masked
      const bool mask_tile = diag || (j * kBTile + kBTile > p.N);
      ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(L::kBarSFull), it & 1, ctl, kBWhereEw));
      if (!ok) break;
      if (warp == 4 && lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 21);
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
        tmem_st16(tS + 64 * h + 16 * m, pk);  // P^T (bf16) inside the columns just read
      };
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (mask_tile) p_chunk(m, std::true_type{});
        else p_chunk(m, std::false_type{});
        tmem_wait_st();
        tc_fence_before();
        arrive_local(L::kBarPReady + m);
      }
      if (warp == 4 && lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 22);

      ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(L::kBarDPFull), it & 1, ctl, kBWhereEw + 1));
      if (!ok) break;
      if (warp == 4 && lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 23);
      tc_fence_after();
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
        tmem_st16(tDP + 64 * h + 16 * m, dk);  // dS^T (bf16)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (4 * m + u) ^ (lrow & 7);
          *reinterpret_cast<uint4*>(ds_row + unit * 16) = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
        tmem_wait_st();
        tc_fence_before();
        arrive_local(L::kBarDSFull + m);
      }
      fence_proxy_async_smem();  // the dS tiles are read by the products and the copy engine
      arrive_local(L::kBarDSmem);
      if (warp == 4 && lane == 0) ATTN_TRACE_AT(blockIdx.x, it, 24);
    }
    // epilogue: dV and dK rows of this key tile; warpgroup h writes columns
    // [h*D/2, (h+1)*D/2)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(L::kBarAccDone), 0, ctl, kBWhereFin));
    if (ok) {
      tc_fence_after();
      const bool live = !key_dead;
      const size_t row = (size_t)bh * p.N + (live ? k_glob : 0);
      uint4* dvrow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dv) + row * D);
      uint4* dkrow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dk) + row * D);
#pragma unroll
      for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
        float a[32], bb[32];
        tmem_ld32(tmem + lane_base + L::kColDV + c0, a);
        tmem_ld32(tmem + lane_base + L::kColDK + c0, bb);
        uint32_t pa[16], pb[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          pa[q] = pack_bf16(a[2 * q], a[2 * q + 1]);
          pb[q] = pack_bf16(bb[2 * q] * p.scale, bb[2 * q + 1] * p.scale);
        }
        if (live) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            dvrow[c0 / 8 + v] = make_uint4(pa[4 * v], pa[4 * v + 1], pa[4 * v + 2], pa[4 * v + 3]);
            dkrow[c0 / 8 + v] = make_uint4(pb[4 * v], pb[4 * v + 1], pb[4 * v + 2], pb[4 * v + 3]);
          }
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kDqRegs));
    // ========================== dQ warpgroup ===========================
    // This CTA's dQ rows (queries 64*rank + (lane % 64)) arrive as 128 lanes
    // x 64 columns: lanes 0-63 hold d 0..63, lanes 64-127 d 64..127.  They
    // are staged in the accumulator's [D/4][64][4] order (this CTA's row half
    // of the tile) and added by the copy engine, one 16 KiB round per d-half.
    const int quad = warp & 3;
    const int tl = quad * 32 + lane;  // tensor-memory lane
    const int lr = tl & 63, ch = tl >> 6;
    const int tid = threadIdx.x - 384;
    const uint32_t tDQ = tmem + ((uint32_t)(quad * 32) << 16) + L::kColDQ;
    float* stg = reinterpret_cast<float*>(smem + L::kStgOff);
    bool ok = live_cta;
    for (int it = 0; ok && it < n_it; ++it) {
      const int i = tile_of(it);
      ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(L::kBarDQFull), it & 1, ctl, kBWhereDq));
      if (!ok) break;
      if (tl == 0) ATTN_TRACE_AT(blockIdx.x, it, 25);
      tc_fence_after();
      float dq[64];
      tmem_ld64(tDQ, dq);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kBarDQFree));  // the tensor-memory dQ columns may be overwritten
      float* gdst = p.dq_acc + ((size_t)bh * p.n_tiles + i) * (size_t)(D * kBTile) + (size_t)own * (64 * D);
      int* ticket = DETERMINISTIC ? p.tickets + (size_t)bh * p.n_tiles + i : nullptr;
#pragma unroll
      for (int r = 0; r < 2 && ok; ++r) {
        const int rc = 2 * it + r;  // staging rounds so far
        if (rc > 0)  // the copy engine has read the previous round
          ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarStgFree), (rc - 1) & 1, ctl, kBWhereDq + 2));
        if (!ok) break;
        if (ch == r) {  // round r: d-half r, held by lanes 64r .. 64r+63
#pragma unroll
          for (int g = 0; g < 16; ++g)
            *reinterpret_cast<float4*>(stg + (g * 64 + lr) * 4) =
                make_float4(dq[4 * g], dq[4 * g + 1], dq[4 * g + 2], dq[4 * g + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(L::kBarStgFull));
        if (tid == 0) {
          bool go = mbar_wait(bar(L::kBarStgFull), rc & 1, ctl, kBWhereDq + 1);
          if (go && DETERMINISTIC && r == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(ticket) < 2 * pr) {  // pairs add into tile i in ascending order
              if (*ctl.abort || globaltimer_ns() - t0 > ctl.timeout_ns) {
                if (!*ctl.abort) report_error(ctl.status, ATTN_ERR_TIMEOUT, kBWhereTicket);
                *ctl.abort = 1;
                go = false;
                break;
              }
            }
            fence_proxy_async_global();
          }
          if (go && !*ctl.abort) {
            bulk_reduce_add_f32(gdst + (size_t)r * 16 * 64 * 4, smem_u32(stg), L::kStgBytes);
            bulk_commit();
          }
          if (DETERMINISTIC && r == 1) {
            bulk_wait_all<0>();  // the additions are performed before the ticket moves on
            fence_proxy_async_global();
            if (go && !*ctl.abort) red_release_gpu_add(ticket, 1);
          } else {
            bulk_wait_read<0>();
          }
          mbar_arrive(bar(L::kBarStgFree));
          ATTN_TRACE_AT(blockIdx.x, it, 26);
        }
        __syncwarp();
      }
    }
    if (tid == 0) bulk_wait_all<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the even CTA's last products wrote this CTA's tensor memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace attn
