// Persistent variant of the backward main kernel (attn_bwd.cuh): one CTA per
// SM takes the (head, key tile) units in rounds, and every role runs its
// pipeline across unit boundaries (ring positions and barrier phases carry
// over); the next unit's K/V load waits only for the last products that read
// the previous K/V, and its first dV / dK products for the previous
// epilogue's read-out of the accumulators.  Short sequences (few query tiles
// per unit) gain the per-CTA setup, the first loads and the epilogue.  It is
// kept apart from the one-unit kernel, whose code generation it would
// otherwise perturb (measured: merging the two cost that kernel 2-3 % at
// N = 16384).
#pragma once

#include "attn_bwd.cuh"

namespace attn {

// Three more barriers: K/V of a unit read for the last time (commit), the
// accumulators read out by the epilogue (256 arrivals), every product done.
template <int D>
struct BwdPLayout : BwdLayout<D> {
  using B = BwdLayout<D>;
  static constexpr int kBarKVEmpty = B::kNumBars;
  static constexpr int kBarAccFree = kBarKVEmpty + 1;
  static constexpr int kBarMmaDrain = kBarAccFree + 1;
  static constexpr int kNumBars = kBarMmaDrain + 1;
  static constexpr int kMiscOff = B::kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int D, bool CAUSAL, bool DETERMINISTIC>
__global__ void __launch_bounds__(512, 1) bwd_persist_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdPLayout<D>;
  // (the unit walk below is written for the general case; this kernel is
  // the plain one: no mask map, one K/V head per query head)
  constexpr bool MASK = false, GQA = false, PERSIST = true;
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
  // work unit u: key tile j of K/V head bh.  Key-tile-major in groups of
  // heads in deterministic mode (a unit waits only on units ordered before
  // it), and over all heads under the causal mask when a round of G units
  // holds two or more units of every head (2 x heads <= G: the rounds then
  // go from the longest units to the shortest, and a head's units in a
  // round share its Q / dO reads in L2); head-major otherwise (resident
  // CTAs share one or two heads' Q, dO and dQ accumulators in L2).  Causal
  // key tiles with small j are the longest and go first in either order.
  // GQA: walk position qi = g * n + i over query head g of the group and
  // query tile i (from n-1 down to i_lo, head after head); the first query
  // head of K/V head bh is qh0.  Deterministic and non-causal: the rotated
  // walk of det_order.h (every CTA is resident, the kernel being launched
  // cooperatively), unit jj starting at query tile (n - 1 - sigma jj) mod n
  // and wrapping from 0 to n - 1.
  constexpr bool kRot = DETERMINISTIC && !CAUSAL && !MASK && !GQA;
  const bool causal_ktm = 2 * n_heads <= (int)gridDim.x;
  // persistent CTAs take unit r G + b in round r (G - 1 - b on odd rounds, so
  // that with the longest units first every CTA gets a similar total); each
  // CTA's units increase from round to round.
  // Cut tail (atomic dQ, no causal mask; the units are all equal): when the
  // last round is partial, rem units for G CTAs, every CTA but rem would idle
  // for a whole unit.  Instead its units are cut into s = min(G / rem, n)
  // pieces of contiguous query tiles, one per CTA (CTA b takes piece b mod s
  // of tail unit b / s), and the round takes about 1/s of a unit.  Each piece
  // leaves FP32 dV / dK partials in slot b of p.tail_part, and the dQ
  // conversion that follows the kernel sums each unit's slots in piece order
  // into dV and dK.  (Measured on GB300, d = 128, H = 16: 2048 units are
  // 13.47 rounds and ran at 1316 TFLOP/s against ~1360 for unit counts that
  // fill their last round.)
  constexpr bool kTail = !DETERMINISTIC && !CAUSAL && !MASK && !GQA;
  const int n_units = PERSIST ? n_heads * n : (int)gridDim.x;
  const int G = gridDim.x;
  const int n_rounds = PERSIST ? (n_units + G - 1) / G : 1;
  const int n_full = n_units / G;
  const int rem = n_units - n_full * G;
  const int tail_s = (kTail && PERSIST && p.tail_s > 1) ? p.tail_s : 1;  // the launch's plan
  struct BUnit {
    int j, bh, i_lo, n_it, qh0, i_first;
    int piece;  // piece of a cut unit (-1: the whole unit)
  };
  auto unit_at = [&](int u, int piece) {
    BUnit w;
    w.piece = piece;
    if (DETERMINISTIC) {
      det_unit(u, n_heads, n, p.det_group, p.det_desc, w.j, w.bh);
    } else if (CAUSAL && causal_ktm) {
      det_unit(u, n_heads, n, n_heads, 0, w.j, w.bh);
    } else {
      w.bh = u / n;
      w.j = u - w.bh * n;
    }
    w.i_lo = CAUSAL ? w.j : 0;  // query tiles i_lo .. n-1, visited from n-1 down
    w.n_it = n - w.i_lo;
    w.qh0 = w.bh;
    if (GQA) {
      const int h_kv = p.h_q / p.kv_group;
      w.qh0 = (w.bh / h_kv) * p.h_q + (w.bh % h_kv) * p.kv_group;
      w.n_it *= p.kv_group;
    }
    if (MASK) {  // only the query tiles holding a visible pair with key tile j
      w.n_it = 0;
      for (int i = 0; i < n; ++i) w.n_it += mask_tile_visible(p.mask, i, w.j) ? 1 : 0;
    }
    // every role walks the same query tiles, from the last down
    w.i_first = MASK ? mask_prev_query_tile(p.mask, w.j, n) : n - 1;
    if (kRot) {
      const DetRot d = det_rot(u, (int)gridDim.x, n_heads, n, p.det_group, p.det_desc);
      w.i_first = det_rot_first(d.jj, n, d.sigma);
    }
    if (kTail && piece >= 0) {  // query tiles [lo, hi), from hi - 1 down
      const int lo = piece * n / tail_s, hi = (piece + 1) * n / tail_s;
      w.i_first = hi - 1;
      w.n_it = hi - lo;
    }
    return w;
  };
  auto tile_i = [&](int qi) { return GQA ? qi % n : qi; };
  auto head_q = [&](const BUnit& w, int qi) { return GQA ? w.qh0 + qi / n : w.bh; };
  auto i_next = [&](const BUnit& w, int i) {
    if (GQA) return (i % n) > w.i_lo ? i - 1 : (i / n + 1) * n + (n - 1);
    if (kRot) return i > 0 ? i - 1 : n - 1;
    return MASK ? mask_prev_query_tile(p.mask, w.j, i) : i - 1;
  };
  // the unit (n_units: none) and piece (-1: whole) of this CTA's round rd
  auto unit_of_round = [&](int rd, int& piece) {
    const int b = (int)blockIdx.x;
    piece = -1;
    if (!PERSIST) return b;
    if (kTail && tail_s > 1 && rd == n_full) {
      piece = b % tail_s;
      return b < rem * tail_s ? n_full * G + b / tail_s : n_units;
    }
    return rd * G + ((rd & 1) ? G - 1 - b : b);
  };

  if (threadIdx.x == 0) {
    for (int b = 0; b < L::kNumBars; ++b) {
      uint32_t cnt = 1;
      if ((b >= L::kBarPReady && b < L::kBarPReady + 2) || (b >= L::kBarDSFull && b < L::kBarDSFull + 2))
        cnt = 256;  // both compute warpgroups
      if (b == L::kBarDQFree) cnt = 128;  // the dQ warpgroup
      if (b == L::kBarAccFree) cnt = 256;  // both compute warpgroups
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
      int issued_q = 0, issued_do = 0;  // loads issued per ring (over all units)
      int t = 0, ucnt = 0;              // tiles and units started
      bool ok = true;
      for (int rd = 0; ok && rd < n_rounds; ++rd) {
        int pc;
        const int u = unit_of_round(rd, pc);
        if (PERSIST && u >= n_units) continue;
        const BUnit w = unit_at(u, pc);
        // K and V of the previous unit are read until its last products complete
        if (PERSIST && ucnt > 0 && !(ok = mbar_wait(bar(L::kBarKVEmpty), (ucnt - 1) & 1, ctl, kBWhereProd + 2)))
          break;
        mbar_arrive_expect_tx(bar(L::kBarKV), 2 * L::kTileBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(sbase + L::kKOff + c * kBSub, &p.tm_k, c * 64, w.j * kBTile, w.bh, bar(L::kBarKV));
          tma_load_3d(sbase + L::kVOff + c * kBSub, &p.tm_v, c * 64, w.j * kBTile, w.bh, bar(L::kBarKV));
        }
        ++ucnt;
        for (int it = 0, qi = w.i_first; it < w.n_it; ++it, qi = i_next(w, qi)) {
          const int tt = t + it;
          const int i = tile_i(qi);
          const int qh = head_q(w, qi);
          const int s = tt % L::kQStages;
          const uint32_t ph = ((tt / L::kQStages) & 1) ^ 1;
          const int sd = tt % L::kDOStages;
          const uint32_t phd = ((tt / L::kDOStages) & 1) ^ 1;
          if (!(ok = mbar_wait(bar(L::kBarQEmpty + s), ph, ctl, kBWhereProd))) break;
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
          issued_q = tt + 1;
          if (!(ok = mbar_wait(bar(L::kBarDOEmpty + sd), phd, ctl, kBWhereProd + 1))) break;
          mbar_arrive_expect_tx(bar(L::kBarDOFull + sd), L::kTileBytes);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sbase + L::kDOOff + sd * L::kTileBytes + c * kBSub, &p.tm_do, c * 64, i * kBTile, qh,
                        bar(L::kBarDOFull + sd));
          ATTN_TRACE_AT(blockIdx.x, it, 14);
          issued_do = tt + 1;
        }
        t += w.n_it;
      }
      // loads still in flight land before the CTA exits: the last unit's K/V
      // and each ring's last (stage count) loads, each on the newest phase of
      // its stage
      if (ucnt > 0) mbar_wait_drain(bar(L::kBarKV), (ucnt - 1) & 1, p.timeout_ns);
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
      bool ok = true;
      int t = 0, ucnt = 0;  // tiles and units done
      for (int rd = 0; ok && rd < n_rounds; ++rd) {
      int pc;
      const int u = unit_of_round(rd, pc);
      if (PERSIST && u >= n_units) continue;
      const BUnit w = unit_at(u, pc);
      if (!(ok = mbar_wait(bar(L::kBarKV), ucnt & 1, ctl, kBWhereMma))) break;
      tc_fence_after();
      for (int it = 0; ok && it < w.n_it; ++it) {
        const int tt = t + it;
        const int s = tt % L::kQStages;
        const uint32_t ph = (tt / L::kQStages) & 1;
        const int sd = tt % L::kDOStages;
        const uint32_t phd = (tt / L::kDOStages) & 1;
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
        if (L::kColDQ == L::kColDP && tt > 0)  // dP^T columns still hold dQ of the previous tile
          if (!(ok = mbar_wait(bar(L::kBarDQFree), (tt - 1) & 1, ctl, kBWhereMma + 2))) break;
        ATTN_TRACE_AT(blockIdx.x, it, 1);
        tc_fence_after();
        mma_kmajor(L::kColDP, sbase + L::kVOff, dos);  // runs while P is computed
        tc_commit(bar(L::kBarDPFull));
        // dV on each half of P^T as it lands (runs while dS is computed)
#pragma unroll
        for (int m = 0; m < 2 && ok; ++m) {
          if (!(ok = mbar_wait(bar(L::kBarPReady + m), tt & 1, ctl, kBWhereMma + 4))) break;
          // the unit's first dV / dK products overwrite the accumulators the
          // previous unit's epilogue reads
          if (PERSIST && it == 0 && m == 0 && ucnt > 0)
            if (!(ok = mbar_wait(bar(L::kBarAccFree), (ucnt - 1) & 1, ctl, kBWhereMma + 7))) break;
          if (m == 0) ATTN_TRACE_AT(blockIdx.x, it, 3);
          tc_fence_after();
          mma_tmem_a_half(L::kColDV, L::kColS, dos, it > 0, m);
        }
        if (!ok) break;
        tc_commit(bar(L::kBarDOEmpty + sd));  // dO_i's last reader: reload it early
#pragma unroll
        for (int m = 0; m < 2 && ok; ++m) {
          if (!(ok = mbar_wait(bar(L::kBarDSFull + m), tt & 1, ctl, kBWhereMma + 6))) break;
          if (m == 0) ATTN_TRACE_AT(blockIdx.x, it, 12);
          tc_fence_after();
          mma_tmem_a_half(L::kColDK, L::kColDP, qs, it > 0, m);
        }
        if (!ok) break;
        tc_commit(bar(L::kBarQEmpty + s));
        if (L::kColDQ != L::kColDP && tt > 0)
          if (!(ok = mbar_wait(bar(L::kBarDQFree), (tt - 1) & 1, ctl, kBWhereMma + 5))) break;
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
      if (!ok) break;
      if (PERSIST) tc_commit(bar(L::kBarKVEmpty));  // this unit's K and V have been read for the last time
      tc_commit(bar(L::kBarAccDone));               // this unit's dV and dK are complete
      t += w.n_it;
      ++ucnt;
      }  // units
      // every product issued above completes before tensor memory is freed
      tc_commit(bar(L::kBarMmaDrain));
      mbar_wait_drain(bar(L::kBarMmaDrain), 0, p.timeout_ns);

    }
    __syncwarp();
   } else if (DETERMINISTIC) {
    // ==================== dQ reducers (deterministic mode) ====================
    // As in bwd_kernel: warps 2 and 3 take the CTA's tiles in turn (counted
    // over all of its units), issue each tile's staged rounds in ticket order,
    // free the staging tile after each read and pass the ticket on once the
    // additions are complete, overlapping that wait with the other reducer.
    if (lane == 0) {
      const int wr = warp - 2;
      int kt = 0;  // tiles this reducer has taken
      bool ok = true;
      int t = 0;  // tiles of earlier units
      for (int rd = 0; ok && rd < n_rounds; ++rd) {
        int pc;
        const int u = unit_of_round(rd, pc);
        if (PERSIST && u >= n_units) continue;
        const BUnit w = unit_at(u, pc);
        const int j = w.j;
        const DetRot dr = kRot ? det_rot(u, (int)gridDim.x, n_heads, n, p.det_group, p.det_desc) : DetRot{};
        for (int it = 0, qi = w.i_first; ok && it < w.n_it; ++it, qi = i_next(w, qi)) {
          const int tt = t + it;
          if ((tt & 1) != wr) continue;
          const int i = tile_i(qi);
          const int qh = head_q(w, qi);
          float* gdst = p.dq_acc + ((size_t)qh * p.n_tiles + i) * (size_t)(D * kBTile);
          int* ticket = p.tickets + (size_t)qh * p.n_tiles + i;
          const int rank = kRot ? det_rot_rank(i, dr, n) : det_rank(i, j, n, CAUSAL, p.det_desc);
          constexpr int kRoundFloats = L::kSlotBytes / 4;
          for (int r = 0; ok && r < L::kRounds; ++r) {
            const int sl = r & 1;
            const uint32_t par = (uint32_t)(kt * (L::kRounds / 2) + (r >> 1)) & 1;
            if (!(ok = mbar_wait(bar(L::kBarStgFull + 2 * wr + sl), par, ctl, kBWhereDq + 2))) break;
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
        t += w.n_it;
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
      int pc0;
      const int u0 = unit_of_round(0, pc0);
      const int n_it0 = u0 < n_units ? unit_at(u0, pc0).n_it : 0;  // the first unit only
      for (int it = 0; live && it < n_it0 && it < kTraceIters; ++it) {
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
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::kColS;
    const uint32_t tDP = tmem + lane_base + L::kColDP;
    const float c_log2 = p.scale_log2;
    bool ok = true;
    int t = 0, ucnt = 0;  // tiles and units done
    for (int rd = 0; ok && rd < n_rounds; ++rd) {
    int pc;
    const int u = unit_of_round(rd, pc);
    if (PERSIST && u >= n_units) continue;
    const BUnit w = unit_at(u, pc);
    const int j = w.j;
    const int k_glob = j * kBTile + lrow;
    const bool key_dead = k_glob >= p.N;
    for (int it = 0, qi = w.i_first; it < w.n_it; ++it, qi = i_next(w, qi)) {
      const int tt = t + it;
      const int i = tile_i(qi);
      const int s = tt % L::kQStages;
      // LSE2 / D vectors arrive with Q_i on the stage's barrier
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarQFull + s), (tt / L::kQStages) & 1, ctl, kBWhereEw + 3));
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
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull), tt & 1, ctl, kBWhereEw));
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

      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDPFull), tt & 1, ctl, kBWhereEw + 1));
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
    // epilogue: dV and dK rows of this key tile; warpgroup h writes columns
    // [h*D/2, (h+1)*D/2) through 64-column boxes in the dS tile (free here:
    // the unit's last dQ product, its last reader, has completed, and this
    // warpgroup writes the next unit's dS only after this epilogue), dV then
    // dK, each stored by TMA as whole rows (measured on GB300 against direct
    // row stores from registers: +3.5 % at N = 8192, +5 % at 4096, +7-14 % at
    // 1024-2048 with atomic dQ; deterministic +3-9 % at N <= 2048).
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarAccDone), ucnt & 1, ctl, kBWhereFin));
    {
      ok = named_bar_and(2, 256, ok);  // both compute warpgroups (the stores below need every row)
      // (a piece of a cut unit is always the CTA's last: its epilogue follows
      // the loop, so that none of its addresses stay live through the tiles)
      if (kTail && w.piece >= 0) {
      } else if (ok) {
        tc_fence_after();
        constexpr int kBoxes = D / 64;
        constexpr uint32_t kBoxBytes = kBTile * 128;
        static_assert(kBoxes * kBoxBytes <= L::kDSBytes, "one tensor's boxes fit the dS tile");
        const uint32_t stg = sbase + L::kDSOff;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {  // dV, then dK
#pragma unroll
          for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
            float a[32];
            tmem_ld32(tmem + lane_base + (pass == 0 ? L::kColDV : L::kColDK) + c0, a);
            const float mul = pass == 0 ? 1.f : p.scale;
            uint32_t pa[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) pa[q] = pack_bf16(a[2 * q] * mul, a[2 * q + 1] * mul);
            const uint32_t box_off = (uint32_t)(c0 / 64) * kBoxBytes + (uint32_t)lrow * 128;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              st_shared_v4(stg + box_off + (uint32_t)(((c0 % 64) / 8 + v) ^ (lrow & 7)) * 16, pa[4 * v],
                           pa[4 * v + 1], pa[4 * v + 2], pa[4 * v + 3]);
          }
          if (pass == 1) {  // both accumulators have been read out: the next unit may overwrite them
            tc_fence_before();
            mbar_arrive(bar(L::kBarAccFree));
          }
          fence_proxy_async_smem();
          named_bar_sync(2, 256);
          if (h == 0 && tid == 0) {
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx)
              tma_store_3d(pass == 0 ? &p.tm_dv : &p.tm_dk, stg + bx * kBoxBytes, bx * 64, w.j * kBTile, w.bh);
            bulk_commit();
            bulk_wait_read<0>();  // the boxes have been read before they are written again
          }
          named_bar_sync(2, 256);
        }
      }
    }
    t += w.n_it;
    ++ucnt;
    }  // units
    if (kTail && ok && tail_s > 1) {
      // a piece of a cut unit (its accumulators complete, waited for above):
      // this thread's FP32 dV / dK partials, its key row and its warpgroup's
      // half of the columns, into the CTA's slot
      int pc;
      if (unit_of_round(n_full, pc) < n_units) {
        tc_fence_after();
        float* mine = p.tail_part + (size_t)blockIdx.x * (2 * kBTile * D);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass)
#pragma unroll
          for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
            float a[32];
            tmem_ld32(tmem + lane_base + (pass == 0 ? L::kColDV : L::kColDK) + c0, a);
            float4* dst = reinterpret_cast<float4*>(mine + (size_t)(pass * kBTile + lrow) * D + c0);
#pragma unroll
            for (int v = 0; v < 8; ++v) dst[v] = make_float4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
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
    int t = 0;  // tiles done
    for (int rd = 0; ok && rd < n_rounds; ++rd) {
    int pc;
    const int u = unit_of_round(rd, pc);
    if (PERSIST && u >= n_units) continue;
    const BUnit w = unit_at(u, pc);
    const int j = w.j;
    for (int it = 0, qi = w.i_first; it < w.n_it; ++it, qi = i_next(w, qi)) {
      const int tt = t + it;
      const int i = tile_i(qi);
      const int qh = head_q(w, qi);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDQFull), tt & 1, ctl, kBWhereDq));
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
        // the reducer warps issue the additions in ticket order; each round is
        // staged into its ring slot once the slot's previous round has been read
#pragma unroll
        for (int r = 0; r < L::kRounds && ok; ++r) {
          const int sl = r & 1;
          const int use = (tt * L::kRounds + r) >> 1;  // earlier rounds through this slot
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
          if (lane == 0) mbar_arrive(bar(L::kBarStgFull + 2 * (tt & 1) + sl));
        }
        if (!ok) break;
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
        if (tt > 0 || r > 1) {
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
      __syncwarp();
      if (tid == 0) ATTN_TRACE_AT(blockIdx.x, it, 11);
    }
    t += w.n_it;
    }  // units
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

template <int D, bool CAUSAL, bool DET>
cudaError_t launch_bwd_persist_main(BwdParams& p, cudaStream_t stream) {
  using L = BwdPLayout<D>;
  auto kernel = bwd_persist_kernel<D, CAUSAL, DET>;
  int sms = 0;
  cudaError_t e = prepare_kernel((const void*)kernel, L::kSmemBytes, L::kLaunchRegs, &sms);
  if (e != cudaSuccess) return e;
  const int n_units = p.BH * p.n_tiles;
  const int grid = n_units < sms ? n_units : sms;  // one CTA per SM
  // the cut tail (atomic dQ without the causal mask; see the kernel): the
  // last round's rem units in s = min(grid / rem, n_tiles) pieces, as many as
  // the workspace has slots for
  p.tail_s = 1;
  if (!DET && !CAUSAL && p.tail_part != nullptr) {
    const int n_full = n_units / grid, rem = n_units - n_full * grid;
    if (n_full > 0 && rem > 0) {
      int s = grid / rem;
      if (s > p.n_tiles) s = p.n_tiles;
      if (s * rem > p.tail_cap) s = p.tail_cap / rem;
      if (s > 1) {
        p.tail_s = s;
        p.tail_first = n_full * grid;
        p.tail_units = rem;
      }
    }
  }
  if constexpr (DET) {
    // Deterministic mode: a unit's dQ additions wait for lower-numbered units,
    // which on later rounds belong to other CTAs (some with a higher index),
    // so every CTA must be resident at once.  A cooperative launch guarantees
    // that even while other kernels hold part of the GPU (or fails up front).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
  }
  kernel<<<grid, L::kThreads, L::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
