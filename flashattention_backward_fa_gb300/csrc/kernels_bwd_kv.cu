// Key/value-major backward kernel on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// "FlashAttention backward", §The loop structure: the outer loop runs over
// key/value blocks and the inner loop over query blocks, so that dK_j and dV_j
// accumulate on chip and are written once. Per (query step of 64 rows, key
// block of 128 rows):
//
//   S^T  = K_j Q_i^T            (recomputed, "Lecture 7" §The recomputation trick)
//   dP~T = V_j dO_i^T
//   P^T  = exp2(S^T * scale*log2e - L_i*log2e)    masked pairs -> 0
//   P~T  = P^T o Z/(1-p),  dP^T = dP~T o Z/(1-p)  (dropout, "Lecture 7" §Dropout)
//   dS^T = P^T o (dP^T - D_i)                     ("FlashAttention backward" §The gradients)
//   dV  += P~T dO_i,   dK += dS^T Q_i             (fp32 in TMEM; dK scaled on store)
//   atomic and ordered modes: dQ_i^T = K_j^T dS^T, added into an fp32 HBM
//   accumulator ("FlashAttention backward" §The loop structure, choice (a)).
//
// Keys sit on the 128 TMEM lanes: one thread owns one key row of S^T and dP^T.
// Row-math warps wait warp-wide (warp_wait) and reconverge after per-lane
// branches, because the TMEM loads and stores are warp-collective (.aligned)
// and must not run on a split warp.
// The row math turns them into P~T and dS^T, each rounded to 16 bits plus the
// rounding residual where a tile holds probabilities above kSplitThreshold
// (see interleave_split), and writes them back over the TMEM columns it has
// just read: dV and dK take them as the A operand straight from TMEM. In
// atomic mode dS^T goes to shared memory instead, where it is the A operand
// of dK and the B operand of dQ^T.
//
// Warp roles: warp 0 issues TMA loads; warp 1 owns TMEM and issues the S^T
// MMAs, warp 3 the dP^T MMAs and warp 2 the dV / dK (and dQ^T) MMAs, so that
// the three MMA streams are issued in parallel (one thread issues at most about
// one MMA per 50 cycles); four row-math warpgroups (warps 4-19)
// take alternate query steps, warpgroup w using buffer w, and write the dV
// (warpgroup 0) / dK (warpgroup 1) epilogue.
//
// dQ (atomic and ordered modes).
//  * atomic: each row-math thread adds its 32 dQ^T values (one d row, the
//    warpgroup's 32 queries) into the fp32 accumulator with red.add straight
//    from the TMEM load; a warp's reduction covers 128 contiguous bytes.
//    Reductions of different key blocks land in any order. (Staging the tile
//    in shared memory for one TMA reduce-add, as the ordered mode does,
//    measured slower: this kernel is bound by shared-memory bandwidth, and
//    staging adds a write and a TMA read of 32 KB a step.)
//  * ordered (deterministic): the row-math warps move dQ^T from TMEM into a
//    staging tile in shared memory, laid out [32 query rows][d] fp32 per
//    warpgroup, over the dS^T image of the step (the dK and dQ^T MMAs have read
//    it by then, and the image of that buffer is not rewritten until the same
//    warpgroups' phase 2 two steps later). The TMA producer thread, which also
//    acts as the reducer, adds each staged tile into the accumulator with one
//    TMA tensor reduce-add and releases the staging area as soon as the TMA
//    unit has read it; producer and reducer duties share one polling loop
//    that never blocks on either. Every 32-row query chunk keeps a counter of the
//    contributions already added; key block j waits until its predecessors
//    (key blocks jlo .. j-1 of that chunk, in ascending order) are complete,
//    adds its own, waits for completion and publishes count + 1. The fp32 sums
//    are then formed in one fixed order ("Lecture 7" §Determinism: a
//    deterministic mode orders the reductions instead of relying on atomics).
//    CTAs take their units from a ticket counter rather than blockIdx, so a
//    key block only ever waits for one that an earlier (hence running or
//    finished) CTA took: no wait can depend on a CTA that is not resident.
//    Queries run from the last step down to the diagonal in both modes, so
//    the key blocks of a head that start together reach each query chunk at
//    the same step.
//
// TMEM columns (512): S^T buffers [0,64) and [64,128), dP^T buffers [128,192)
// and [192,256) (dS^T image, or dQ^T in atomic mode, later in the step),
// dV [256,256+d), dK [256+d,256+2d).
#include "fa_internal.h"

namespace fa {

// 4 role warps + 4 row-math warpgroups. (A 21st warp would put six warps on
// one SM sub-partition and cap every thread at 80 registers, which spills the
// row math; the dQ reducer therefore shares the TMA producer's thread.)
constexpr int kKVThreads = 640;

template <int D, bool kAtomic, bool kBias = false>
struct KVCfg {
  static constexpr int kThreads = kKVThreads;
  static constexpr int kPanels = D / 64;
  static constexpr uint32_t kKVPanel = kRowsKV * 128;          // 16 KB: 128 rows x 64 elements
  static constexpr uint32_t kKVTile = kPanels * kKVPanel;
  static constexpr uint32_t kQPanel = kStepQ * 128;            // 8 KB: 64 rows x 64 elements
  static constexpr uint32_t kQTile = kPanels * kQPanel;
  static constexpr uint32_t kPTile = kRowsKV * kStepQ * 2;     // 16 KB: 128 keys x 64 queries
  static constexpr uint32_t kImgBytes = kAtomic ? 4 * kPTile : 0;  // dS^T [buffer][rounded, residual]
  // attention bias tile of a step: 64 query rows x 128 keys, 16-bit, unswizzled
  static constexpr uint32_t kBiasTile = kBias ? kStepQ * kRowsKV * 2 : 0;
  static constexpr uint32_t kStageBytes = 2 * kQTile + 2 * kStepQ * 4 + kBiasTile;
  // (+128: alignment of the bias tiles, only when there are any; at d = 128 with
  // atomic dQ the budget holds exactly three stages without it)
  static constexpr uint32_t kFixed = 2 * kKVTile + kImgBytes + 512 + 1024 + (kBias ? 128 : 0);
  static constexpr int kNSraw = (int)((227u * 1024u - kFixed) / kStageBytes);
  static constexpr int kNS = kNSraw > 4 ? 4 : kNSraw;          // Q/dO pipeline stages
  static constexpr uint32_t oK = 0;
  static constexpr uint32_t oV = oK + kKVTile;
  static constexpr uint32_t oQ = oV + kKVTile;
  static constexpr uint32_t oDO = oQ + kNS * kQTile;
  static constexpr uint32_t oImg = oDO + kNS * kQTile;
  static constexpr uint32_t oL = oImg + kImgBytes;
  static constexpr uint32_t oD = oL + kNS * kStepQ * 4;
  static constexpr uint32_t oB = kBias ? (oD + kNS * kStepQ * 4 + 127) & ~127u : oD + kNS * kStepQ * 4;
  static constexpr uint32_t oBar = oB + kNS * kBiasTile;
  static constexpr int bKV = 0;
  static constexpr int bQFull = 1;
  static constexpr int bQEmpty = bQFull + kNS;
  static constexpr int bSFull = bQEmpty + kNS;                // [2]: S^T landed
  static constexpr int bDPFull = bSFull + 2;                   // [2]: dP^T landed
  static constexpr int bSEmpty = bDPFull + 2;
  static constexpr int bDPEmpty = bSEmpty + 2;
  static constexpr int bPFull = bDPEmpty + 2;
  static constexpr int bDSFull = bPFull + 2;                   // [2]: dS^T image written
  static constexpr int bDQFull = bDSFull + 2;                  // [2]: dQ^T MMAs (and dK) done
  static constexpr int bStaged = bDQFull + 2;                  // [2]: dQ^T staged over the image
  static constexpr int bStageFree = bStaged + 2;               // [2]: staging read by the TMA unit
  static constexpr int bAcc = bStageFree + 2;
  static constexpr int bDrain = bAcc + 1;                      // one per MMA-issuing warp
  // CTA pairs: the peer's K/V tiles and Q/dO stages landed (leader's barriers)
  static constexpr int bPeerKV = bDrain + 3;
  static constexpr int bPeerQFull = bPeerKV + 1;
  static constexpr int kBars = bPeerQFull + kNS;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = oAbort + 8;               // [buffer][CTA of the pair][warp] split votes
  static constexpr uint32_t kSmem = oFlags + 128 + 1024;       // + slack for 1024-byte alignment
  static_assert(kNS >= 2, "shared memory budget leaves fewer than two Q/dO stages");
  static_assert(kBias || kNS >= (kAtomic && D == 128 ? 3 : 4), "Q/dO pipeline shallower than designed");
  static_assert(kSmem <= 227u * 1024u, "shared memory budget exceeded");
};

// One row of a 128-row x 64-element, 128-byte-swizzled shared tile: chunk t of
// the 32 elements [32c, 32c+32) goes to 16-byte slot (4c + t) ^ (row & 7).
__device__ __forceinline__ void store_tile_row_chunk(uint32_t row_addr, int row, int c, const uint32_t (&v)[16]) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t slot = (uint32_t)((4 * c + t) ^ (row & 7)) << 4;
    st_shared_v4(row_addr + slot, v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
  }
}

// kPair: the CTA pair form (a cluster of two CTAs on two adjacent key blocks
// of one head; see the comment at launch_dkdv_t). tmQ32 / tmDO32 are the
// 32-row maps of the pair's split Sᵀ / dPᵀ operands (unused otherwise).
template <int D, bool kBf16, bool kAtomic, bool kDrop, bool kAlibi, bool kBias, bool kPair>
__global__ void __launch_bounds__(KVCfg<D, kAtomic, kBias>::kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmBias,
                    const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmQ32,
                    const __grid_constant__ CUtensorMap tmDO32) {
  static_assert(!kPair || (D == 128 && !kAtomic && !kBias), "CTA pairs: d = 128, deterministic, no bias tensor");
  using C = KVCfg<D, kAtomic, kBias>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oAbort);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + C::oFlags);
  auto bar = [&](int idx) -> uint32_t { return sb + C::oBar + 8u * idx; };
  const bool ordered = kAtomic && p.dq_flags != nullptr;

  // Work unit: (batch*head or sequence*head, key block), heaviest key blocks
  // first under a causal mask. A key block past the end of its sequence has no
  // work: the whole CTA leaves before any setup. In ordered mode the unit
  // comes from the ticket counter (taken in order by running CTAs), and the
  // tiles are outermost over all units, so that the key blocks of one head
  // that run at the same time are few.
  int idx = blockIdx.x;
  if (ordered) {
    volatile int* slot = reinterpret_cast<volatile int*>(smem + C::oAbort + 4);
    if (threadIdx.x == 0) {
      const unsigned int t = atomicAdd(p.dq_ticket, 1u);
      // A ticket past the grid means the counter was not reset by the
      // preprocess before this launch: do no work and report it.
      if (t >= gridDim.x) atomicOr(p.status, kStatusBadLaunch);
      *slot = t >= gridDim.x ? -1 : (int)t;
    }
    __syncthreads();
    idx = *slot;
    if (idx < 0) return;
  }
  // CTA pairs: a unit is two adjacent key blocks (cluster rank r takes the
  // second-level block 2 * tile + r); both CTAs run the union of the two
  // blocks' query steps, which the leader's MMAs need from both.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  constexpr int kUnitRows = (kPair ? 2 : 1) * kRowsKV;
  Unit u;
  if (!unit_decode(p, kPair ? (int)(blockIdx.x >> 1) : idx, kUnitRows, false, u, ordered ? (1 << 30) : kUnitGroup))
    return;
  const int bh = u.bh, b = u.b, h = u.h;
  const int Nl = u.n;                    // rows of this (batch, head) or sequence
  const int ju = u.tile * kUnitRows;     // first key of the unit
  const int j0 = ju + (int)rank * kRowsKV;  // first key of this CTA
  const int i_first = p.causal ? ju : 0;
  int i_last = Nl - 1;
  if (p.window > 0) i_last = min(i_last, ju + kUnitRows - 2 + p.window);
  const int nsteps = (i_last >= i_first) ? (i_last - i_first) / kStepQ + 1 : 0;
  // First query row of step `it`: ascending from the diagonal in the
  // deterministic kernel, descending from the last step when dQ is accumulated.
  auto step_i0 = [&](int it) { return i_first + (kAtomic ? nsteps - 1 - it : it) * kStepQ; };

  // MMA and commit forms: cta_group::2 (leader of a pair, M = 256; commits
  // arrive on the barrier in both CTAs) or cta_group::1.
  auto mma_ss = [&](uint32_t d, uint64_t a, uint64_t bd, uint32_t id, uint32_t acc) {
    if constexpr (kPair) tc_mma_ss_pair_w(d, a, bd, id, acc); else tc_mma_ss_w(d, a, bd, id, acc);
  };
  auto mma_ts = [&](uint32_t d, uint32_t a, uint64_t bd, uint32_t id, uint32_t acc) {
    if constexpr (kPair) tc_mma_ts_pair_w(d, a, bd, id, acc); else tc_mma_ts_w(d, a, bd, id, acc);
  };
  auto commit = [&](uint32_t br) {
    if constexpr (kPair) tc_commit_pair_w(br); else tc_commit_w(br);
  };
  constexpr int kM = kPair ? 256 : 128;
  // B panels of the S^T / dP^T operands: 64 query rows, or 32 in a pair
  constexpr uint32_t kSPanel = kPair ? 4096u : C::kQPanel;
  // B operands of dV / dK: the whole stage tile, or (pair) this CTA's d half after the two 32-row panels
  constexpr uint32_t kGOff = kPair ? C::kQPanel : 0u;
  // an arrival of this warp on a barrier the leader's MMA issuers wait on
  auto arrive_leader = [&](uint32_t br) {
    if constexpr (kPair) {
      if (leader) {
        warp_arrive(br);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_cnt(mapa_shared(br, 0), 32);
      }
    } else {
      warp_arrive(br);
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bKV), 1);
    for (int s = 0; s < C::kNS; ++s) {
      mbar_init(bar(C::bQFull + s), 1);
      mbar_init(bar(C::bQEmpty + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::bSFull + x), 1);                        // S^T landed
      mbar_init(bar(C::bDPFull + x), 1);                       // dP^T landed
      mbar_init(bar(C::bSEmpty + x), 1);                       // dV done with the P~T image
      mbar_init(bar(C::bDPEmpty + x), kAtomic ? 256 : 1);     // dK done / dQ^T drained
      mbar_init(bar(C::bPFull + x), kPair ? 512 : 256);        // P~T image of two warpgroups (of both CTAs)
      mbar_init(bar(C::bDSFull + x), kPair ? 512 : 256);       // dS^T image of two warpgroups (of both CTAs)
      mbar_init(bar(C::bDQFull + x), 1);
      mbar_init(bar(C::bStaged + x), 2 * D);                   // the warps holding dQ^T rows (d of them per warpgroup)
      mbar_init(bar(C::bStageFree + x), 1);                    // the reducer
    }
    for (int x = 0; x < 3; ++x) mbar_init(bar(C::bDrain + x), 1);
    mbar_init(bar(C::bAcc), 1);
    mbar_init(bar(C::bPeerKV), 1);
    for (int x = 0; x < C::kNS; ++x) mbar_init(bar(C::bPeerQFull + x), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(sb + C::oTmemSlot, 512);  // one warp of each CTA, together
    } else {
      tmem_alloc(sb + C::oTmemSlot, 512);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(kPair ? &tmQ32 : &tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(kPair ? &tmDO32 : &tmDO);
    if constexpr (kAtomic) prefetch_tmap(&tmDQ);
  }
  tc_fence_before();
  __syncthreads();
  // pair: both CTAs' barriers are initialised (and TMEM allocated) before either
  // signals the other
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::oTmemSlot);
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::bKV), 2 * C::kKVTile);
      for (int pn = 0; pn < C::kPanels; ++pn) {
        tma_load_4d(sb + C::oK + pn * C::kKVPanel, &tmK, bar(C::bKV), 64 * pn, u.row0 + j0, h, b);
        tma_load_4d(sb + C::oV + pn * C::kKVPanel, &tmV, bar(C::bKV), 64 * pn, u.row0 + j0, h, b);
      }
      // Q, dO (and bias, L, D) of step `it` into its stage.
      auto issue_stage = [&](int it) {
        const int s = it % C::kNS;
        const int i0 = step_i0(it);
        mbar_arrive_expect_tx(bar(C::bQFull + s), C::kStageBytes);
        if constexpr (kPair) {
          // S^T / dP^T operands: this CTA's 32 queries x all of d (two 32-row
          // panels); dK / dV operands: all 64 queries x this CTA's half of d.
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_4d(sb + C::oQ + s * C::kQTile + pn * 4096, &tmQ32, bar(C::bQFull + s), 64 * pn,
                        u.row0 + i0 + 32 * (int)rank, h, b);
            tma_load_4d(sb + C::oDO + s * C::kQTile + pn * 4096, &tmDO32, bar(C::bQFull + s), 64 * pn,
                        u.row0 + i0 + 32 * (int)rank, h, b);
          }
          tma_load_4d(sb + C::oQ + s * C::kQTile + C::kQPanel, &tmQ, bar(C::bQFull + s), 64 * (int)rank,
                      u.row0 + i0, h, b);
          tma_load_4d(sb + C::oDO + s * C::kQTile + C::kQPanel, &tmDO, bar(C::bQFull + s), 64 * (int)rank,
                      u.row0 + i0, h, b);
        } else {
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_4d(sb + C::oQ + s * C::kQTile + pn * C::kQPanel, &tmQ, bar(C::bQFull + s), 64 * pn,
                        u.row0 + i0, h, b);
            tma_load_4d(sb + C::oDO + s * C::kQTile + pn * C::kQPanel, &tmDO, bar(C::bQFull + s), 64 * pn,
                        u.row0 + i0, h, b);
          }
        }
        if constexpr (kBias)  // 64 query rows x 128 keys of the bias (rows / keys past N read as 0)
          tma_load_4d(sb + C::oB + s * C::kBiasTile, &tmBias, bar(C::bQFull + s), u.row0 + j0, u.row0 + i0,
                      p.bias_sh ? h : 0, p.bias_sb ? b : 0);
        const long long ws = u.ws + i0;
        bulk_load(sb + C::oL + s * kStepQ * 4, p.ws_nL2 + ws, kStepQ * 4, bar(C::bQFull + s));
        bulk_load(sb + C::oD + s * kStepQ * 4, p.ws_nD + ws, kStepQ * 4, bar(C::bQFull + s));
      };
      int issued = 0;
      if (!ordered) {
        for (int it = 0; it < nsteps; ++it) {
          if (!mbar_wait(bar(C::bQEmpty + it % C::kNS), ((it / C::kNS) & 1) ^ 1, abort_flag, p.status)) break;
          issue_stage(it);
          issued = it + 1;
        }
      } else if constexpr (kAtomic) {
        // One loop serves both duties without blocking on either: issue the
        // next stage once its buffer is free; reduce the next staged dQ tile
        // once both warpgroups have staged it (and, ordered, once the key
        // blocks before this one have published their contributions to its
        // chunks). An ordered contribution is published once it has completed:
        // right after the next step's reduction has been issued (waiting for
        // every bulk group but that newest one; the last one after the loop),
        // so the loop never blocks on a reduction that is still in flight and
        // the stage loads it also issues are not held up.
        const bool packed = p.cu_seqlens != nullptr;
        // accumulator map: (d, rows of one head, heads or batch*heads); this unit's rows start at y0
        const int z = packed ? u.h : u.bh;
        const int y0 = (int)(u.acc - (long long)z * p.n_pad);
        const long long fl0 =
            (long long)(packed ? u.seq * p.H + u.h : u.bh) * ((packed ? p.seq_pad : p.n_pad) / 32);
        // Position of this key block among those that visit query step i0
        // (jlo .. the diagonal block, ascending): exactly the key blocks with
        // j0 <= i0 under the causal mask and j0 + 126 + window >= i0 under a window.
        auto chain_pos = [&](int i0) -> unsigned int {
          int jlo = 0;
          if (p.window > 0) {
            const int t = i0 - (kRowsKV - 2) - p.window;
            if (t > 0) jlo = (t + kRowsKV - 1) / kRowsKV;
          }
          return (unsigned int)(u.tile - jlo);
        };
        int reduced = 0, pending = -1;  // pending: a step whose ordered contribution awaits publication
        // Publishes `pending`, whose bulk group has completed (the caller waited):
        // one release fence, then both chunk counters.
        auto publish = [&]() {
          fence_proxy_async_global();
          fence_acq_rel_gpu();
          const int i0 = step_i0(pending);
          const unsigned int pos = chain_pos(i0);
          for (int c = 0; c < 2; ++c) st_relaxed_gpu(p.dq_flags + fl0 + (i0 + 32 * c) / 32, pos + 1);
          pending = -1;
        };
        unsigned long long t_idle = 0;
        uint32_t idle = 0;
        while (issued < nsteps || reduced < nsteps) {
          bool progress = false;
          if (issued < nsteps &&
              mbar_test_wait(bar(C::bQEmpty + issued % C::kNS), ((issued / C::kNS) & 1) ^ 1)) {
            issue_stage(issued);
            ++issued;
            progress = true;
          }
          if (reduced < nsteps && mbar_test_wait(bar(C::bStaged + (reduced & 1)), (reduced >> 1) & 1)) {
            const int i0 = step_i0(reduced);
            // both chunk counters are read before either value is used, with
            // relaxed loads (acquired once they show every predecessor)
            const unsigned int pos = chain_pos(i0);
            const unsigned int f0 = ld_relaxed_gpu(p.dq_flags + fl0 + i0 / 32);
            const unsigned int f1 = ld_relaxed_gpu(p.dq_flags + fl0 + i0 / 32 + 1);
            if (f0 >= pos && f1 >= pos) {
              fence_acq_rel_gpu();
              fence_proxy_async_global();
              const uint32_t img = sb + C::oImg + 2 * (reduced & 1) * C::kPTile;
              for (int c = 0; c < 2; ++c) tma_reduce_add_3d(&tmDQ, img + c * C::kPTile, 0, y0 + i0 + 32 * c, z);
              bulk_commit_group();
              bulk_wait_read_all();
              mbar_arrive(bar(C::bStageFree + (reduced & 1)));
              if (pending >= 0) {
                bulk_wait_all_but_last();  // the previous step's group has landed
                publish();
              }
              pending = reduced;
              ++reduced;
              progress = true;
            }
          }
          if (progress) {
            idle = 0;
            continue;
          }
          // Nothing to do: bounded like every other wait of the kernel.
          if (idle++ == 0) t_idle = globaltimer_ns();
          if ((idle & 63u) == 0) {
            if (*abort_flag) break;
            if (globaltimer_ns() - t_idle > kWaitLimitNs) {
              atomicOr(p.status, kStatusTimeout);
              *abort_flag = 1;
              break;
            }
          }
          __nanosleep(20);
        }
        // every reduction has landed (and, ordered, is published) before the CTA exits
        bulk_wait_all();
        if (pending >= 0 && !*abort_flag) publish();
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        mbar_wait_drain(bar(C::bKV), 0, p.status);
        for (int it = max(0, issued - C::kNS); it < issued; ++it)
          mbar_wait_drain(bar(C::bQFull + it % C::kNS), (it / C::kNS) & 1, p.status);
      }
    }
  } else if (kPair && !leader && warp == 1) {
    // ------------------------ pair: peer's load forwarder -----------------------
    // The leader's MMAs read this CTA's K/V tiles and Q/dO stages: pass each
    // completion on to the leader's barriers.
    if (lane == 0) {
      bool ok = mbar_wait(bar(C::bKV), 0, abort_flag, p.status);
      if (ok) mbar_arrive_remote_cnt(mapa_shared(bar(C::bPeerKV), 0), 1);
      for (int it = 0; ok && it < nsteps; ++it) {
        const int s = it % C::kNS;
        if (!mbar_wait(bar(C::bQFull + s), (it / C::kNS) & 1, abort_flag, p.status)) break;
        mbar_arrive_remote_cnt(mapa_shared(bar(C::bPeerQFull + s), 0), 1);
      }
    }
    __syncwarp();
  } else if (kPair && !leader && (warp == 2 || warp == 3)) {
    // pair: the leader issues every MMA
  } else if (warp == 1) {
    // ------------------------------ S^T MMA issuer -----------------------------
    {
      constexpr uint32_t idS = make_idesc(kM, kStepQ, kBf16, false, false);
      const uint64_t dK0 = make_sdesc(sb + C::oK, 16, 1024), dQ0 = make_sdesc(sb + C::oQ, 16, 1024);
      bool ok = warp_wait<kIssuerPoll>(bar(C::bKV), 0, abort_flag, p.status) &&
                (!kPair || warp_wait<kIssuerPoll, true>(bar(C::bPeerKV), 0, abort_flag, p.status));
      for (int it = 0; ok && it < nsteps; ++it) {
        const int s = it % C::kNS, bb = it & 1;
        if (!warp_wait<kIssuerPoll>(bar(C::bQFull + s), (it / C::kNS) & 1, abort_flag, p.status) ||
            (kPair &&
             !warp_wait<kIssuerPoll, true>(bar(C::bPeerQFull + s), (it / C::kNS) & 1, abort_flag, p.status)) ||
            !warp_wait<kIssuerPoll>(bar(C::bSEmpty + bb), ((it >> 1) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t q = desc_add(dQ0, s * C::kQTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tS + 64 * bb, desc_add(dK0, (k >> 2) * C::kKVPanel + (k & 3) * 32),
                 desc_add(q, (k >> 2) * kSPanel + (k & 3) * 32), idS, k > 0 ? 1u : 0u);
        commit(bar(C::bSFull + bb));
      }
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      commit(bar(C::bDrain));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain), 0, p.status);
      __syncwarp();
    }
  } else if (warp == 3) {
    // ----------------------------- dP^T MMA issuer -----------------------------
    {
      constexpr uint32_t idS = make_idesc(kM, kStepQ, kBf16, false, false);
      const uint64_t dV0 = make_sdesc(sb + C::oV, 16, 1024), dO0 = make_sdesc(sb + C::oDO, 16, 1024);
      bool ok = warp_wait<kIssuerPoll>(bar(C::bKV), 0, abort_flag, p.status) &&
                (!kPair || warp_wait<kIssuerPoll, true>(bar(C::bPeerKV), 0, abort_flag, p.status));
      for (int it = 0; ok && it < nsteps; ++it) {
        const int s = it % C::kNS, bb = it & 1;
        if (!warp_wait<kIssuerPoll>(bar(C::bQFull + s), (it / C::kNS) & 1, abort_flag, p.status) ||
            (kPair &&
             !warp_wait<kIssuerPoll, true>(bar(C::bPeerQFull + s), (it / C::kNS) & 1, abort_flag, p.status)) ||
            !warp_wait<kIssuerPoll>(bar(C::bDPEmpty + bb), ((it >> 1) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t g = desc_add(dO0, s * C::kQTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tdP + 64 * bb, desc_add(dV0, (k >> 2) * C::kKVPanel + (k & 3) * 32),
                 desc_add(g, (k >> 2) * kSPanel + (k & 3) * 32), idS, k > 0 ? 1u : 0u);
        commit(bar(C::bDPFull + bb));
      }
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      commit(bar(C::bDrain + 2));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain + 2), 0, p.status);
      __syncwarp();
    }
  } else if (warp == 2) {
    // ----------------------- dV / dK (/ dQ^T) MMA issuer ----------------------
    {
      constexpr uint32_t idG = make_idesc(kM, D, kBf16, false, true);          // dV, dK
      constexpr uint32_t idQ = make_idesc(128, kStepQ, kBf16, true, true);     // dQ^T
      const uint64_t mQ0 = make_sdesc(sb + C::oQ + kGOff, C::kQPanel, 1024),
                     mO0 = make_sdesc(sb + C::oDO + kGOff, C::kQPanel, 1024);
      const uint64_t mK0 = make_sdesc(sb + C::oK, C::kKVPanel, 1024);
      bool ok = true;
      for (int t = 0; ok && t < nsteps; ++t) {
        const int bt = t & 1, st = t % C::kNS;
        if (!warp_wait<kConsumerPoll, kPair>(bar(C::bPFull + bt), (t >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        bool split = false;
#pragma unroll
        for (int x = 0; x < (kPair ? 16 : 8); ++x) split |= flags[16 * bt + x] != 0;
        const uint32_t first = t > 0 ? 1u : 0u;
        const uint64_t q = desc_add(mQ0, st * C::kQTile), g = desc_add(mO0, st * C::kQTile);
        // dV += P~T dO: K step k reads the 8 rounded columns at 16k of the P~T image
        // and, on split tiles, the 8 residual columns at 16k + 8.
#pragma unroll
        for (int k = 0; k < kStepQ / 16; ++k)
          mma_ts(tdV, tS + 64 * bt + 16 * k, desc_add(g, 2048 * k), idG, k > 0 ? 1u : first);
        if (split) {
#pragma unroll
          for (int k = 0; k < kStepQ / 16; ++k)
            mma_ts(tdV, tS + 64 * bt + 16 * k + 8, desc_add(g, 2048 * k), idG, 1u);
        }
        commit(bar(C::bSEmpty + bt));
        // dK (and dQ^T) once the dS^T image is in place; dV above only needed P~T.
        if (!warp_wait<kConsumerPoll, kPair>(bar(C::bDSFull + bt), (t >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (!kAtomic) {
          // dK += dS^T Q from the dS^T image over the dP^T columns.
#pragma unroll
          for (int k = 0; k < kStepQ / 16; ++k)
            mma_ts(tdK, tdP + 64 * bt + 16 * k, desc_add(q, 2048 * k), idG, k > 0 ? 1u : first);
          if (split) {
#pragma unroll
            for (int k = 0; k < kStepQ / 16; ++k)
              mma_ts(tdK, tdP + 64 * bt + 16 * k + 8, desc_add(q, 2048 * k), idG, 1u);
          }
          commit(bar(C::bDPEmpty + bt));
        } else {
          // dK += dS^T Q and dQ^T = K^T dS^T from the shared dS^T tiles; dQ^T lands in
          // this buffer's dP^T columns, which the row math has consumed. For d = 64
          // the upper 64 rows of the 128-row dQ^T MMA are ignored.
          const uint32_t img = sb + C::oImg + 2 * bt * C::kPTile;
          const uint64_t aK = make_sdesc(img, 16, 1024), bQT = make_sdesc(img, C::kPTile, 1024);
          for (int part = 0; part < (split ? 2 : 1); ++part) {
#pragma unroll
            for (int k = 0; k < kStepQ / 16; ++k)
              tc_mma_ss_w(tdK, desc_add(aK, part * C::kPTile + 32 * k), desc_add(q, 2048 * k), idG,
                          (k > 0 || part > 0) ? 1u : first);
          }
          for (int part = 0; part < (split ? 2 : 1); ++part) {
#pragma unroll
            for (int k = 0; k < kRowsKV / 16; ++k)
              tc_mma_ss_w(tdP + 64 * bt, desc_add(mK0, 2048 * k), desc_add(bQT, part * C::kPTile + 2048 * k), idQ,
                          (k > 0 || part > 0) ? 1u : 0u);
          }
          tc_commit_w(bar(C::bDQFull + bt));
        }
        commit(bar(C::bQEmpty + st));
      }
      commit(bar(C::bAcc));
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      commit(bar(C::bDrain + 1));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain + 1), 0, p.status);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ------------------------- row-math warpgroups --------------------------
    // Four warpgroups: rg = 0, 1 take the even query steps (TMEM buffer 0) and
    // rg = 2, 3 the odd ones (buffer 1); within a pair, warpgroup rg & 1 takes
    // query columns [32 (rg & 1), 32 (rg & 1) + 32) of the step, in halves of 16
    // columns (one MMA K step). Each step runs in two phases: P~T from S^T
    // (released to the dV MMA at once), then dS^T from dP^T and the kept fp32 P.
    const int rg = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int c = rg & 1;
    const int bb = rg >> 1;
    const int jl = wq * 32 + lane;
    const int j = j0 + jl;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tSc = tS + lane_off + 64 * bb + 32 * c, tdPc = tdP + lane_off + 64 * bb + 32 * c;
    const uint32_t imgRow = sb + C::oImg + 2 * bb * C::kPTile + jl * 128;
    const float slope_raw = kAlibi ? alibi_slope_raw(p, u) : 0.f;
    const float inv_scale = kBias ? 1.f / p.scale : 0.f;
    bool ok = true;
    for (int it = bb; it < nsteps; it += 2) {
      const int s = it % C::kNS;
      const int i0 = step_i0(it);
      if (!warp_wait<kRowMathPoll>(bar(C::bQFull + s), (it / C::kNS) & 1, abort_flag, p.status) ||
          !warp_wait<kRowMathPoll>(bar(C::bSFull + bb), (it >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4* L4 = reinterpret_cast<const float4*>(smem + C::oL + s * kStepQ * 4 + 128 * c);
      const float4* D4 = reinterpret_cast<const float4*>(smem + C::oD + s * kStepQ * 4 + 128 * c);
      const int base = i0 + 32 * c;
      // allowed pairs of this chunk (bit x <-> query base + x) and dropout keep bits
      uint32_t allow = 0u;
      if (j < Nl) {
        const int lo = p.causal ? j - base : 0;
        int hi = Nl - base;
        if (p.window > 0) hi = min(hi, j + p.window - base);
        allow = bit_range(lo, hi);
      }
      uint32_t keep = 0xFFFFFFFFu;
      if constexpr (kDrop) {
        __syncwarp();  // warp-collective (shuffles)
        keep = keep_bits_for_key(p.drop, bh, Nl, base, j);
      }
      float P[32];          // P (before dropout) of this thread's 32 pairs, for the dS phase
      bool split_h[2];
      // ---- phase 1: P~T image over the S^T columns ----
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t sr[16];
        __syncwarp();  // per-lane branches above: converge for the TMEM load
        tmem_ld16(tSc + 16 * hh, sr);
        tmem_ld_wait16(sr);
        if constexpr (kAlibi) alibi_fold16<1>(sr, (float)(base + 16 * hh - j), slope_raw);
        if constexpr (kBias)  // bias tile row = query (32c + 16hh + e) of the step, column = this key
          bias_fold16_smem<kBf16>(sr, sb + C::oB + s * C::kBiasTile + (uint32_t)(32 * c + 16 * hh) * (kRowsKV * 2) +
                                          (uint32_t)jl * 2,
                                  kRowsKV * 2, inv_scale);
        float cmax = 0.f;
        float pt[16];
        // P = exp2(S * scale*log2e + (-L*log2e)) on pairs of columns; the unmasked
        // variant skips the per-pair mask test on full tiles.
        auto p_phase = [&](auto masked) {
#pragma unroll
          for (int x = 0; x < 16; x += 4) {
            const float4 l4 = L4[(16 * hh + x) >> 2];
            const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
            float pv[4];
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[x]), __uint_as_float(sr[x + 1])), c2, f2_pack(l4.x, l4.y)),
                      pv[0], pv[1]);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[x + 2]), __uint_as_float(sr[x + 3])), c2, f2_pack(l4.z, l4.w)),
                      pv[2], pv[3]);
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              const int bit = 16 * hh + x + y;
              pv[y] = ex2_approx(pv[y]);
              if constexpr (decltype(masked)::value) pv[y] = ((allow >> bit) & 1u) ? pv[y] : 0.f;
              P[bit] = pv[y];
              if constexpr (kDrop)
                pt[x + y] = ((keep >> bit) & 1u) ? pv[y] * p.drop.rp : 0.f;
              else
                pt[x + y] = pv[y];
            }
            cmax = fmax3(cmax, pv[0], pv[1]);
            cmax = fmax3(cmax, pv[2], pv[3]);
          }
        };
        if (allow == 0xFFFFFFFFu)
          p_phase(std::false_type{});
        else
          p_phase(std::true_type{});
        // The lanes may have split over the two variants: reconverge before the
        // warp-collective vote and TMEM stores below.
        __syncwarp();
        uint32_t hp[8], ep[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) hp[x] = pack2<kBf16>(pt[2 * x], pt[2 * x + 1]);
        // Residuals only where this warp's rows hold a probability above the
        // split threshold; zeros elsewhere keep the residual image well defined.
        split_h[hh] = __any_sync(0xFFFFFFFFu, cmax > kSplitThreshold);
        if (split_h[hh]) {
#pragma unroll
          for (int x = 0; x < 8; ++x) ep[x] = pack2_residual<kBf16>(pt[2 * x], pt[2 * x + 1], hp[x]);
        } else {
#pragma unroll
          for (int x = 0; x < 8; ++x) ep[x] = 0u;
        }
        // This K step's image: 8 rounded columns, then 8 residual columns.
        tmem_st8<0>(tSc + 16 * hh, hp);
        tmem_st8<0>(tSc + 16 * hh + 8, ep);
      }
      tmem_st_wait();
      {
        // split vote of this warp for the MMA issuer (pair: into the leader's
        // votes, second half for the peer)
        const int vote = (split_h[0] || split_h[1]) ? 1 : 0;
        const int vi = 16 * bb + 8 * (int)rank + 4 * c + wq;
        if (lane == 0) {
          if (leader)
            flags[vi] = vote;
          else
            st_shared_cluster_u32(mapa_shared(sb + C::oFlags + 4u * vi, 0), (uint32_t)vote);
        }
      }
      tc_fence_before();
      arrive_leader(bar(C::bPFull + bb));
      // ---- phase 2: dS^T = P o (dP^T (o Z/(1-p)) + (-D)) ----
      // In ordered mode the image of this buffer held the dQ^T staging of step
      // it - 2 until the reducer's TMA read it (a fresh barrier passes the
      // first wait).
      if (!warp_wait<kRowMathPoll>(bar(C::bDPFull + bb), (it >> 1) & 1, abort_flag, p.status) ||
          (ordered &&
           !warp_wait<kRowMathPoll>(bar(C::bStageFree + bb), ((it >> 1) & 1) ^ 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t dr[16];
        tmem_ld16(tdPc + 16 * hh, dr);
        tmem_ld_wait16(dr);
        float ds[16];
#pragma unroll
        for (int x = 0; x < 16; x += 4) {
          const float4 d4 = D4[(16 * hh + x) >> 2];
          if constexpr (!kDrop) {
            const uint64_t d01 =
                f2_add(f2_pack(__uint_as_float(dr[x]), __uint_as_float(dr[x + 1])), f2_pack(d4.x, d4.y));
            const uint64_t d23 =
                f2_add(f2_pack(__uint_as_float(dr[x + 2]), __uint_as_float(dr[x + 3])), f2_pack(d4.z, d4.w));
            f2_unpack(f2_mul(f2_pack(P[16 * hh + x], P[16 * hh + x + 1]), d01), ds[x], ds[x + 1]);
            f2_unpack(f2_mul(f2_pack(P[16 * hh + x + 2], P[16 * hh + x + 3]), d23), ds[x + 2], ds[x + 3]);
          } else {
            const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              const int bit = 16 * hh + x + y;
              const float dpv = ((keep >> bit) & 1u) ? __uint_as_float(dr[x + y]) * p.drop.rp : 0.f;
              ds[x + y] = P[bit] * (dpv + dv[y]);
            }
          }
        }
        uint32_t hd[8], ed[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) hd[x] = pack2<kBf16>(ds[2 * x], ds[2 * x + 1]);
        if (split_h[hh]) {
#pragma unroll
          for (int x = 0; x < 8; ++x) ed[x] = pack2_residual<kBf16>(ds[2 * x], ds[2 * x + 1], hd[x]);
        } else {
#pragma unroll
          for (int x = 0; x < 8; ++x) ed[x] = 0u;
        }
        if constexpr (!kAtomic) {
          tmem_st8<0>(tdPc + 16 * hh, hd);
          tmem_st8<0>(tdPc + 16 * hh + 8, ed);
        } else {
          // dS^T row jl: 16 queries = two 16-byte slots of the 128-byte swizzled rows.
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint32_t slot = (uint32_t)((4 * c + 2 * hh + t) ^ (jl & 7)) << 4;
            st_shared_v4(imgRow + slot, hd[4 * t], hd[4 * t + 1], hd[4 * t + 2], hd[4 * t + 3]);
            st_shared_v4(imgRow + C::kPTile + slot, ed[4 * t], ed[4 * t + 1], ed[4 * t + 2], ed[4 * t + 3]);
          }
        }
      }
      if constexpr (!kAtomic) tmem_st_wait();
      tc_fence_before();
      if constexpr (kAtomic) fence_proxy_async_smem();
      arrive_leader(bar(C::bDSFull + bb));
      if constexpr (kAtomic) {
        // dQ^T (d on lanes, this warpgroup's 32 queries on columns) -> the staging
        // tile [32 queries][d] fp32 over this warpgroup's half of the image; the
        // reducer adds it into the accumulator.
        if (!warp_wait<kRowMathPoll>(bar(C::bDQFull + bb), (it >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r0[32];
        tmem_ld32(tdPc, r0);
        tmem_ld_wait(r0);
        tc_fence_before();
        warp_arrive(bar(C::bDPEmpty + bb));
        if (wq < D / 32) {  // lanes of the warps holding rows d < D of the M = 128 dQ^T
          if (ordered) {
            const uint32_t stg = sb + C::oImg + (2 * bb + c) * C::kPTile + (uint32_t)jl * 4;
#pragma unroll
            for (int x = 0; x < 32; ++x)
              asm volatile("st.shared.b32 [%0], %1;" ::"r"(stg + (uint32_t)x * (D * 4)), "r"(r0[x]) : "memory");
            fence_proxy_async_smem();
            warp_arrive(bar(C::bStaged + bb));
          } else {
            float* dst = p.ws_dq + (u.acc + base) * D + jl;
#pragma unroll
            for (int x = 0; x < 32; ++x) atomicAdd(dst + x * D, __uint_as_float(r0[x]));
          }
        }
      }
    }
    // Epilogue: warpgroups 0, 1 write dV and 2, 3 write scale * dK, each half of the columns.
    if (ok && nsteps > 0) ok = warp_wait<kRowMathPoll>(bar(C::bAcc), 0, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      const bool isK = rg >= 2;
      const long long off = (long long)b * p.sb + (long long)(u.row0 + j) * p.sn + (long long)h * p.sh;
      uint16_t* dst = static_cast<uint16_t*>(isK ? p.dk : p.dv) + off;
      const uint32_t col0 = (isK ? tdK : tdV) + lane_off;
      const float mul = isK ? p.scale : 1.f;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = c * (D / 2) + 32 * cc;
        uint32_t r[32];
        if (nsteps > 0) {
          tmem_ld32(col0 + col, r);
          tmem_ld_wait(r);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          w[x] = pack2<kBf16>(__uint_as_float(r[2 * x]) * mul, __uint_as_float(r[2 * x + 1]) * mul);
        if (j < Nl) {
          uint4* g = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
          for (int t = 0; t < 4; ++t) g[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // pair: the leader's MMAs (drained above) read the peer's shared memory and
  // write its TMEM, so neither CTA frees anything before both get here
  if constexpr (kPair) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem, 512);
    else
      tmem_dealloc(tmem, 512);
  }
}

// One CTA per (unit, key block), or, with kPair, one cluster of two CTAs per
// (unit, pair of adjacent key blocks): the leader issues every MMA with M = 256
// (both CTAs' keys); each CTA holds half of each B operand (32 of the step's 64
// queries for S^T and dP^T, half of d for dV and dK), so a CTA's shared-memory
// operand reads per step fall from 128 KB to 96 KB. A key block past N in the
// last pair of an odd tile count takes part with out-of-range keys, which the
// row math masks and the epilogue does not store.
template <int D, bool kBf16, bool kAtomic, bool kDrop, bool kAlibi, bool kBias, bool kPair>
static cudaError_t launch_dkdv_t(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  using C = KVCfg<D, kAtomic, kBias>;
  auto kern = bwd_dkdv_kernel<D, kBf16, kAtomic, kDrop, kAlibi, kBias, kPair>;
  const int smem = (int)(C::kSmem > kMinSmemOneCtaPerSm ? C::kSmem : kMinSmemOneCtaPerSm);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rows = p.cu_seqlens ? p.max_seqlen : p.N;
  const int units = p.cu_seqlens ? p.nseq * p.H : p.B * p.H;
  if constexpr (!kPair) {
    const int tiles = (rows + kRowsKV - 1) / kRowsKV;
    const unsigned grid = (unsigned)(tiles * units);
    kern<<<grid, C::kThreads, smem, st>>>(p, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6],
                                          maps[7]);
    return cudaGetLastError();
  } else {
    const int pairs = (rows + 2 * kRowsKV - 1) / (2 * kRowsKV);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs * units));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7]);
  }
}

template <int D, bool kBf16, bool kAtomic, bool kBias>
static cudaError_t launch_dkdv_b(const AttnParams& p, bool pair, const CUtensorMap* maps, cudaStream_t st) {
  const bool drop = p.drop.on != 0;
  if constexpr (D == 128 && !kAtomic && !kBias) {
    if (pair) {
      if (p.alibi)
        return drop ? launch_dkdv_t<D, kBf16, false, true, true, false, true>(p, maps, st)
                    : launch_dkdv_t<D, kBf16, false, false, true, false, true>(p, maps, st);
      return drop ? launch_dkdv_t<D, kBf16, false, true, false, false, true>(p, maps, st)
                  : launch_dkdv_t<D, kBf16, false, false, false, false, true>(p, maps, st);
    }
  }
  if (p.alibi)
    return drop ? launch_dkdv_t<D, kBf16, kAtomic, true, true, kBias, false>(p, maps, st)
                : launch_dkdv_t<D, kBf16, kAtomic, false, true, kBias, false>(p, maps, st);
  return drop ? launch_dkdv_t<D, kBf16, kAtomic, true, false, kBias, false>(p, maps, st)
              : launch_dkdv_t<D, kBf16, kAtomic, false, false, kBias, false>(p, maps, st);
}

template <int D, bool kBf16, bool kAtomic>
static cudaError_t launch_dkdv_a(const AttnParams& p, bool pair, const CUtensorMap* maps, cudaStream_t st) {
  return p.bias ? launch_dkdv_b<D, kBf16, kAtomic, true>(p, pair, maps, st)
                : launch_dkdv_b<D, kBf16, kAtomic, false>(p, pair, maps, st);
}

template <int D, bool kBf16>
static cudaError_t launch_dkdv_d(const AttnParams& p, bool atomic, bool pair, const CUtensorMap* maps,
                                 cudaStream_t st) {
  return atomic ? launch_dkdv_a<D, kBf16, true>(p, pair, maps, st) : launch_dkdv_a<D, kBf16, false>(p, pair, maps, st);
}

// Whether the CTA-pair form applies: d = 128, deterministic, no bias tensor, fixed length.
bool dkdv_pair_supported(const AttnParams& p, bool atomic) {
  return p.d == 128 && !atomic && p.bias == nullptr && p.cu_seqlens == nullptr;
}

// maps: Q, K, V, dO (Q/dO boxes of kStepQ rows, K/V boxes of kRowsKV rows), the
// attention bias (boxes of kStepQ rows x kRowsKV keys; any valid map when
// p.bias is null), the fp32 dQ accumulator as (d, rows per head, heads) with
// boxes of d x 32 rows (any valid map in the deterministic kernel), and Q, dO
// with boxes of 32 rows (the pair form's S^T / dP^T operands; any valid map
// otherwise). `pair` asks for the CTA-pair form where dkdv_pair_supported.
cudaError_t launch_bwd_dkdv_tc(const AttnParams& p, bool bf16, bool atomic, bool pair, const CUtensorMap* maps,
                               cudaStream_t st) {
  pair = pair && dkdv_pair_supported(p, atomic);
  if (p.d == 128)
    return bf16 ? launch_dkdv_d<128, true>(p, atomic, pair, maps, st)
                : launch_dkdv_d<128, false>(p, atomic, pair, maps, st);
  return bf16 ? launch_dkdv_d<64, true>(p, atomic, false, maps, st) : launch_dkdv_d<64, false>(p, atomic, false, maps, st);
}

}  // namespace fa
