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
// one MMA per 50 cycles); four row-math warpgroups (warps 4-19) take alternate
// query steps (warpgroups 0, 1 the even ones, in TMEM buffer 0; 2, 3 the odd
// ones); the pair that ran a unit's last step writes its dV and dK epilogue.
//
// Persistent grid (deterministic kernel): one CTA per SM runs unit after unit,
// taking the next unit from a counter in the workspace (the first one is its
// blockIdx), so CTAs that finish early take more units and no CTA waits for a
// launch. (With accumulated dQ the same code runs one unit per CTA.) Steps are numbered across units: stage, TMEM buffer and
// barrier phases continue from one unit to the next, so the next unit's S^T and
// dP^T MMAs and its loads run while the current unit's last steps and its
// epilogue finish. Two hand-offs separate consecutive units: the next unit's
// K and V overwrite this unit's once its last S^T / dP^T (and dQ^T) MMAs have
// completed (KVFree), and its first dV / dK MMAs overwrite the accumulators once
// the epilogue pair has loaded them (AccFree). The producer publishes each
// next unit in a small ring in shared memory, read by every other role. The
// ordered dQ mode takes its one unit from the ticket counter in launch order,
// which its deadlock argument needs.
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
// Warps that read the unit ring (warps 1-3 and the 16 row-math warps).
constexpr int kUnitReaders = 19;
constexpr int kUnitSlots = 4;

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
  static constexpr int bKV = 0;                                // K, V of a unit landed
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
  static constexpr int bAcc = bStageFree + 2;                  // a unit's dV, dK complete in TMEM
  static constexpr int bDrain = bAcc + 1;                      // one per MMA-issuing warp
  static constexpr int bKVFree = bDrain + 3;                   // a unit's last reads of K, V done
  static constexpr int bAccFree = bKVFree + 1;                 // the epilogue has read dV, dK
  static constexpr int bUnit = bAccFree + 1;                   // [kUnitSlots]: next unit published
  static constexpr int bUnitFree = bUnit + kUnitSlots;         // [kUnitSlots]: ring slot read by all
  static constexpr int kBars = bUnitFree + kUnitSlots;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = oAbort + 8;               // [buffer][warp] split votes
  static constexpr uint32_t oUnits = oFlags + 128;             // [kUnitSlots] unit ring
  static constexpr uint32_t kSmem = oUnits + 4 * kUnitSlots + 1024;  // + slack for 1024-byte alignment
  static_assert(kNS >= 2, "shared memory budget leaves fewer than two Q/dO stages");
  static_assert(kBias || kNS >= (kAtomic && D == 128 ? 3 : 4), "Q/dO pipeline shallower than designed");
  static_assert(kSmem <= 227u * 1024u, "shared memory budget exceeded");
};

// Geometry of one key block (unit): its decode, first key, query-step range.
struct KVUnit {
  Unit u;
  int j0, i_first, nsteps;
};

// Decodes unit `idx`; false when the key block lies past its sequence (no work).
// Under the masks every key block that exists sees at least one query step.
__device__ __forceinline__ bool kv_unit(const AttnParams& p, int idx, bool ordered, KVUnit& g) {
  if (!unit_decode(p, idx, kRowsKV, false, g.u, ordered ? (1 << 30) : kUnitGroup)) return false;
  g.j0 = g.u.tile * kRowsKV;
  g.i_first = p.causal ? g.j0 : 0;
  int i_last = g.u.n - 1;
  if (p.window > 0) i_last = min(i_last, g.j0 + kRowsKV - 2 + p.window);
  g.nsteps = (i_last >= g.i_first) ? (i_last - g.i_first) / kStepQ + 1 : 0;
  return true;
}

template <int D, bool kBf16, bool kAtomic, bool kDrop, bool kAlibi, bool kBias>
__global__ void __launch_bounds__(KVCfg<D, kAtomic, kBias>::kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmBias,
                    const __grid_constant__ CUtensorMap tmDQ) {
  using C = KVCfg<D, kAtomic, kBias>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oAbort);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + C::oFlags);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + C::oUnits);
  auto bar = [&](int idx) -> uint32_t { return sb + C::oBar + 8u * idx; };
  const bool ordered = kAtomic && p.dq_flags != nullptr;
  const bool packed = p.cu_seqlens != nullptr;
  const int total_units = ((packed ? p.max_seqlen : p.N) + kRowsKV - 1) / kRowsKV * (packed ? p.nseq * p.H : p.B * p.H);

  // First unit: blockIdx (persistent grid), or, in ordered mode, the ticket
  // counter (taken in order by running CTAs), with the tiles outermost over all
  // units, so that the key blocks of one head that run at the same time are few.
  int first = blockIdx.x;
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
    first = *slot;
    if (first < 0) return;
  }

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
      mbar_init(bar(C::bPFull + x), 256);                      // P~T image of two warpgroups
      mbar_init(bar(C::bDSFull + x), 256);                     // dS^T image of two warpgroups
      mbar_init(bar(C::bDQFull + x), 1);
      mbar_init(bar(C::bStaged + x), 2 * D);                   // the warps holding dQ^T rows (d of them per warpgroup)
      mbar_init(bar(C::bStageFree + x), 1);                    // the reducer
    }
    for (int x = 0; x < 3; ++x) mbar_init(bar(C::bDrain + x), 1);
    mbar_init(bar(C::bAcc), 1);
    mbar_init(bar(C::bKVFree), kAtomic ? 3 : 2);               // S^T, dP^T (and dQ^T) issuers
    mbar_init(bar(C::bAccFree), 8 * 32);                       // the epilogue pair's row-math warps
    for (int x = 0; x < kUnitSlots; ++x) {
      mbar_init(bar(C::bUnit + x), 1);
      mbar_init(bar(C::bUnitFree + x), kUnitReaders * 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + C::oTmemSlot, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
    if constexpr (kAtomic) prefetch_tmap(&tmDQ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::oTmemSlot);
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  // The unit after this CTA's k-th one, from ring slot k % kUnitSlots (every
  // role but the producer; warp-wide). -1: no more units (or the CTA aborted).
  auto next_unit = [&](int k) -> int {
    const int s = k % kUnitSlots;
    if (!warp_wait<kIssuerPoll>(bar(C::bUnit + s), (k / kUnitSlots) & 1, abort_flag, p.status)) return -1;
    const int idx = unit_ring[s];
    __syncwarp();
    warp_arrive(bar(C::bUnitFree + s));
    return idx;
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      int idx = first, k = 0, kl = 0, G = 0, gi = 0;  // units seen / loaded, steps before this unit / issued
      bool ok = true;
      while (ok && idx >= 0) {
        int next_idx = -1;
        // The ticket of the unit after this one is taken first (persistent grid):
        // its latency overlaps this unit's loads. None in ordered mode.
        unsigned int tk = 0;
        if (!ordered && p.unit_ctr != nullptr) tk = atomicAdd(p.unit_ctr, 1u);
        // Publishes the next unit (key blocks past their sequence are skipped).
        auto publish_next = [&]() -> bool {
          int nxt = -1;
          if (!ordered) {
            int cand = p.unit_ctr ? (int)(gridDim.x + tk) : idx + (int)gridDim.x;
            for (;;) {
              if (cand >= total_units) break;
              KVUnit gn;
              if (kv_unit(p, cand, false, gn) && gn.nsteps > 0) {
                nxt = cand;
                break;
              }
              cand = p.unit_ctr ? (int)(gridDim.x + atomicAdd(p.unit_ctr, 1u)) : cand + (int)gridDim.x;
            }
          }
          if (!mbar_wait(bar(C::bUnitFree + k % kUnitSlots), ((k / kUnitSlots) & 1) ^ 1, abort_flag, p.status))
            return false;
          unit_ring[k % kUnitSlots] = nxt;
          mbar_arrive(bar(C::bUnit + k % kUnitSlots));
          next_idx = nxt;
          return true;
        };
        KVUnit g;
        if (!kv_unit(p, idx, ordered, g) || g.nsteps == 0) {
          if (!publish_next()) break;
        } else {
          const Unit& u = g.u;
          const int b = u.b, h = u.h, j0 = g.j0, nsteps = g.nsteps, i_first = g.i_first;
          auto step_i0 = [&](int it) { return i_first + (kAtomic ? nsteps - 1 - it : it) * kStepQ; };
          // K and V of this unit, once the previous unit's last reads of them are done
          if (kl > 0 &&
              !mbar_wait(bar(C::bKVFree), (kl - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::bKV), 2 * C::kKVTile);
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_4d(sb + C::oK + pn * C::kKVPanel, &tmK, bar(C::bKV), 64 * pn, u.row0 + j0, h, b);
            tma_load_4d(sb + C::oV + pn * C::kKVPanel, &tmV, bar(C::bKV), 64 * pn, u.row0 + j0, h, b);
          }
          ++kl;
          // Q, dO (and bias, L, D) of local step `it` into stage s.
          auto issue_stage_at = [&](int it, int s) {
            const int i0 = step_i0(it);
            mbar_arrive_expect_tx(bar(C::bQFull + s), C::kStageBytes);
            for (int pn = 0; pn < C::kPanels; ++pn) {
              tma_load_4d(sb + C::oQ + s * C::kQTile + pn * C::kQPanel, &tmQ, bar(C::bQFull + s), 64 * pn,
                          u.row0 + i0, h, b);
              tma_load_4d(sb + C::oDO + s * C::kQTile + pn * C::kQPanel, &tmDO, bar(C::bQFull + s), 64 * pn,
                          u.row0 + i0, h, b);
            }
            if constexpr (kBias)  // 64 query rows x 128 keys of the bias (rows / keys past N read as 0)
              tma_load_4d(sb + C::oB + s * C::kBiasTile, &tmBias, bar(C::bQFull + s), u.row0 + j0, u.row0 + i0,
                          p.bias_sh ? h : 0, p.bias_sb ? b : 0);
            const long long ws = u.ws + i0;
            bulk_load(sb + C::oL + s * kStepQ * 4, p.ws_nL2 + ws, kStepQ * 4, bar(C::bQFull + s));
            bulk_load(sb + C::oD + s * kStepQ * 4, p.ws_nD + ws, kStepQ * 4, bar(C::bQFull + s));
          };
          if (!ordered) {
            for (int it = 0; it < nsteps; ++it) {
              const int gs = G + it;
              if (!mbar_wait(bar(C::bQEmpty + gs % C::kNS), ((gs / C::kNS) & 1) ^ 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              issue_stage_at(it, gs % C::kNS);
              gi = gs + 1;
            }
          } else if constexpr (kAtomic) {
            // ordered mode: one unit per CTA (G = 0), stage of step it = it % kNS
            auto issue_stage = [&](int it) { issue_stage_at(it, it % C::kNS); };
            int issued = 0;
          // One loop serves both duties without blocking on either: issue the
          // next stage once its buffer is free; reduce the next staged dQ tile
          // once both warpgroups have staged it (and, ordered, once the key
          // blocks before this one have published their contributions to its
          // chunks). An ordered contribution is published once it has completed:
          // right after the next step's reduction has been issued (waiting for
          // every bulk group but that newest one; the last one after the loop),
          // so the loop never blocks on a reduction that is still in flight and
          // the stage loads it also issues are not held up.
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
            gi = issued;
            ok = !*abort_flag;
          }
          G += nsteps;
          // The next unit is published once this unit's loads are issued (the
          // consumers need it only when they finish this unit).
          if (ok && !publish_next()) ok = false;
        }
        idx = next_idx;
        ++k;
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        if (kl > 0) mbar_wait_drain(bar(C::bKV), (kl - 1) & 1, p.status);
        for (int x = max(0, gi - C::kNS); x < gi; ++x)
          mbar_wait_drain(bar(C::bQFull + x % C::kNS), (x / C::kNS) & 1, p.status);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------ S^T (warp 1) / dP^T (warp 3) MMA issuer ----------------
    // S^T = K Q^T or dP~T = V dO^T: M = 128 keys, N = 64 queries, K = d, both
    // operands K-major in shared memory.
    {
      const bool isS = warp == 1;
      constexpr uint32_t idS = make_idesc(128, kStepQ, kBf16, false, false);
      const uint64_t dA0 = make_sdesc(sb + (isS ? C::oK : C::oV), 16, 1024),
                     dB0 = make_sdesc(sb + (isS ? C::oQ : C::oDO), 16, 1024);
      const uint32_t tD = isS ? tS : tdP;
      const int bF = isS ? C::bSFull : C::bDPFull, bE = isS ? C::bSEmpty : C::bDPEmpty;
      int idx = first, k = 0, kl = 0, G = 0;
      bool ok = true;
      while (ok && idx >= 0) {
        KVUnit g;
        if (kv_unit(p, idx, ordered, g) && g.nsteps > 0) {
          ok = warp_wait<kIssuerPoll>(bar(C::bKV), kl & 1, abort_flag, p.status);
          for (int it = 0; ok && it < g.nsteps; ++it) {
            const int gs = G + it, s = gs % C::kNS, bb = gs & 1;
            if (!warp_wait<kIssuerPoll>(bar(C::bQFull + s), (gs / C::kNS) & 1, abort_flag, p.status) ||
                !warp_wait<kIssuerPoll>(bar(bE + bb), ((gs >> 1) & 1) ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bq = desc_add(dB0, s * C::kQTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss_w(tD + 64 * bb, desc_add(dA0, (kk >> 2) * C::kKVPanel + (kk & 3) * 32),
                          desc_add(bq, (kk >> 2) * C::kQPanel + (kk & 3) * 32), idS, kk > 0 ? 1u : 0u);
            tc_commit_w(bar(bF + bb));
          }
          if (!ok) break;
          tc_commit_w(bar(C::bKVFree));  // this unit's last reads of K / V
          G += g.nsteps;
          ++kl;
        }
        idx = next_unit(k++);
      }
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      const int dr = isS ? 0 : 2;
      tc_commit_w(bar(C::bDrain + dr));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain + dr), 0, p.status);
      __syncwarp();
    }
  } else if (warp == 2) {
    // ----------------------- dV / dK (/ dQ^T) MMA issuer ----------------------
    {
      constexpr uint32_t idG = make_idesc(128, D, kBf16, false, true);          // dV, dK
      constexpr uint32_t idQ = make_idesc(128, kStepQ, kBf16, true, true);     // dQ^T
      const uint64_t mQ0 = make_sdesc(sb + C::oQ, C::kQPanel, 1024), mO0 = make_sdesc(sb + C::oDO, C::kQPanel, 1024);
      const uint64_t mK0 = make_sdesc(sb + C::oK, C::kKVPanel, 1024);
      int idx = first, k = 0, kl = 0, G = 0;
      bool ok = true;
      while (ok && idx >= 0) {
        KVUnit g;
        if (kv_unit(p, idx, ordered, g) && g.nsteps > 0) {
          for (int t = 0; ok && t < g.nsteps; ++t) {
            const int gs = G + t, bt = gs & 1, st = gs % C::kNS;
            if (!warp_wait<kConsumerPoll>(bar(C::bPFull + bt), (gs >> 1) & 1, abort_flag, p.status) ||
                // the first dV / dK MMAs of a unit overwrite the accumulators the
                // previous unit's epilogue reads
                (t == 0 && kl > 0 && !warp_wait<kConsumerPoll>(bar(C::bAccFree), (kl - 1) & 1, abort_flag, p.status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            bool split = false;
#pragma unroll
            for (int x = 0; x < 8; ++x) split |= flags[16 * bt + x] != 0;
            const uint32_t first_acc = t > 0 ? 1u : 0u;
            const uint64_t q = desc_add(mQ0, st * C::kQTile), gd = desc_add(mO0, st * C::kQTile);
            // dV += P~T dO: K step kk reads the 8 rounded columns at 16kk of the P~T image
            // and, on split tiles, the 8 residual columns at 16kk + 8.
#pragma unroll
            for (int kk = 0; kk < kStepQ / 16; ++kk)
              tc_mma_ts_w(tdV, tS + 64 * bt + 16 * kk, desc_add(gd, 2048 * kk), idG, kk > 0 ? 1u : first_acc);
            if (split) {
#pragma unroll
              for (int kk = 0; kk < kStepQ / 16; ++kk)
                tc_mma_ts_w(tdV, tS + 64 * bt + 16 * kk + 8, desc_add(gd, 2048 * kk), idG, 1u);
            }
            tc_commit_w(bar(C::bSEmpty + bt));
            // dK (and dQ^T) once the dS^T image is in place; dV above only needed P~T.
            if (!warp_wait<kConsumerPoll>(bar(C::bDSFull + bt), (gs >> 1) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if constexpr (!kAtomic) {
              // dK += dS^T Q from the dS^T image over the dP^T columns.
#pragma unroll
              for (int kk = 0; kk < kStepQ / 16; ++kk)
                tc_mma_ts_w(tdK, tdP + 64 * bt + 16 * kk, desc_add(q, 2048 * kk), idG, kk > 0 ? 1u : first_acc);
              if (split) {
#pragma unroll
                for (int kk = 0; kk < kStepQ / 16; ++kk)
                  tc_mma_ts_w(tdK, tdP + 64 * bt + 16 * kk + 8, desc_add(q, 2048 * kk), idG, 1u);
              }
              tc_commit_w(bar(C::bDPEmpty + bt));
            } else {
              // dK += dS^T Q and dQ^T = K^T dS^T from the shared dS^T tiles; dQ^T lands in
              // this buffer's dP^T columns, which the row math has consumed. For d = 64
              // the upper 64 rows of the 128-row dQ^T MMA are ignored.
              const uint32_t img = sb + C::oImg + 2 * bt * C::kPTile;
              const uint64_t aK = make_sdesc(img, 16, 1024), bQT = make_sdesc(img, C::kPTile, 1024);
              for (int part = 0; part < (split ? 2 : 1); ++part) {
#pragma unroll
                for (int kk = 0; kk < kStepQ / 16; ++kk)
                  tc_mma_ss_w(tdK, desc_add(aK, part * C::kPTile + 32 * kk), desc_add(q, 2048 * kk), idG,
                              (kk > 0 || part > 0) ? 1u : first_acc);
              }
              for (int part = 0; part < (split ? 2 : 1); ++part) {
#pragma unroll
                for (int kk = 0; kk < kRowsKV / 16; ++kk)
                  tc_mma_ss_w(tdP + 64 * bt, desc_add(mK0, 2048 * kk), desc_add(bQT, part * C::kPTile + 2048 * kk), idQ,
                              (kk > 0 || part > 0) ? 1u : 0u);
              }
              tc_commit_w(bar(C::bDQFull + bt));
            }
            tc_commit_w(bar(C::bQEmpty + st));
          }
          if (!ok) break;
          tc_commit_w(bar(C::bAcc));
          if constexpr (kAtomic) tc_commit_w(bar(C::bKVFree));  // the dQ^T MMAs read K
          G += g.nsteps;
          ++kl;
        }
        idx = next_unit(k++);
      }
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      tc_commit_w(bar(C::bDrain + 1));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain + 1), 0, p.status);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ------------------------- row-math warpgroups --------------------------
    // Four warpgroups: rg = 0, 1 take the even query steps (TMEM buffer 0) and
    // rg = 2, 3 the odd ones (buffer 1), counted across units; within a pair,
    // warpgroup rg & 1 takes query columns [32 (rg & 1), 32 (rg & 1) + 32) of
    // the step, in halves of 16 columns (one MMA K step). Each step runs in two
    // phases: P~T from S^T (released to the dV MMA at once), then dS^T from
    // dP^T and the kept fp32 P. After a unit's steps the pair that ran its last
    // step writes the dV / dK epilogue; the other pair goes on to the next unit.
    const int rg = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int c = rg & 1;
    const int bb = rg >> 1;
    const int jl = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tSc = tS + lane_off + 64 * bb + 32 * c, tdPc = tdP + lane_off + 64 * bb + 32 * c;
    const uint32_t imgRow = sb + C::oImg + 2 * bb * C::kPTile + jl * 128;
    const float inv_scale = kBias ? 1.f / p.scale : 0.f;
    int idx = first, k = 0, kl = 0, G = 0;
    bool ok = true;
    while (ok && idx >= 0) {
      KVUnit g;
      if (kv_unit(p, idx, ordered, g)) {
        const Unit& u = g.u;
        const int bh = u.bh, b = u.b, h = u.h, Nl = u.n, nsteps = g.nsteps, i_first = g.i_first;
        const int j = g.j0 + jl;
        const float slope_raw = kAlibi ? alibi_slope_raw(p, u) : 0.f;
        auto step_i0 = [&](int it) { return i_first + (kAtomic ? nsteps - 1 - it : it) * kStepQ; };
        for (int it = (bb ^ G) & 1; it < nsteps; it += 2) {
          const int gs = G + it;
          const int s = gs % C::kNS;
          const int i0 = step_i0(it);
        const int base = i0 + 32 * c;
        // allowed pairs of this chunk (bit x <-> query base + x) and dropout keep
        // bits: both depend on positions only, so they are formed before the waits
        // and the Philox calls overlap the loads and MMAs of this step.
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
          if (!warp_wait<kRowMathPoll>(bar(C::bQFull + s), (gs / C::kNS) & 1, abort_flag, p.status) ||
              !warp_wait<kRowMathPoll>(bar(C::bSFull + bb), (gs >> 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
        const float4* L4 = reinterpret_cast<const float4*>(smem + C::oL + s * kStepQ * 4 + 128 * c);
        const float4* D4 = reinterpret_cast<const float4*>(smem + C::oD + s * kStepQ * 4 + 128 * c);
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
                if constexpr (!kDrop) pt[x + y] = pv[y];
              }
              if constexpr (kDrop) {
                // P~ = P * (kept ? 1/(1-p) : 0), two columns per multiply
                const int bit = 16 * hh + x;
                const float m0 = ((keep >> bit) & 1u) ? p.drop.rp : 0.f, m1 = ((keep >> (bit + 1)) & 1u) ? p.drop.rp : 0.f;
                const float m2 = ((keep >> (bit + 2)) & 1u) ? p.drop.rp : 0.f, m3 = ((keep >> (bit + 3)) & 1u) ? p.drop.rp : 0.f;
                f2_unpack(f2_mul(f2_pack(pv[0], pv[1]), f2_pack(m0, m1)), pt[x], pt[x + 1]);
                f2_unpack(f2_mul(f2_pack(pv[2], pv[3]), f2_pack(m2, m3)), pt[x + 2], pt[x + 3]);
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
        // split vote of this warp for the MMA issuer
        if (lane == 0) flags[16 * bb + 4 * c + wq] = (split_h[0] || split_h[1]) ? 1 : 0;
        tc_fence_before();
        warp_arrive(bar(C::bPFull + bb));
        // ---- phase 2: dS^T = P o (dP^T (o Z/(1-p)) + (-D)) ----
        // In ordered mode the image of this buffer held the dQ^T staging of step
        // it - 2 until the reducer's TMA read it (a fresh barrier passes the
        // first wait).
        if (!warp_wait<kRowMathPoll>(bar(C::bDPFull + bb), (gs >> 1) & 1, abort_flag, p.status) ||
            (ordered &&
             !warp_wait<kRowMathPoll>(bar(C::bStageFree + bb), ((gs >> 1) & 1) ^ 1, abort_flag, p.status))) {
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
              // dS = P * (kept ? dP~ / (1-p) - D : -D): one packed FMA, a select, one packed multiply
              const uint64_t rp2 = f2_pack(p.drop.rp, p.drop.rp);
              float a[4];
              f2_unpack(f2_fma(f2_pack(__uint_as_float(dr[x]), __uint_as_float(dr[x + 1])), rp2, f2_pack(d4.x, d4.y)),
                        a[0], a[1]);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(dr[x + 2]), __uint_as_float(dr[x + 3])), rp2, f2_pack(d4.z, d4.w)),
                        a[2], a[3]);
              const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
  #pragma unroll
              for (int y = 0; y < 4; ++y) a[y] = ((keep >> (16 * hh + x + y)) & 1u) ? a[y] : dv[y];
              f2_unpack(f2_mul(f2_pack(P[16 * hh + x], P[16 * hh + x + 1]), f2_pack(a[0], a[1])), ds[x], ds[x + 1]);
              f2_unpack(f2_mul(f2_pack(P[16 * hh + x + 2], P[16 * hh + x + 3]), f2_pack(a[2], a[3])), ds[x + 2], ds[x + 3]);
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
        warp_arrive(bar(C::bDSFull + bb));
        if constexpr (kAtomic) {
          // dQ^T (d on lanes, this warpgroup's 32 queries on columns) -> the staging
          // tile [32 queries][d] fp32 over this warpgroup's half of the image; the
          // reducer adds it into the accumulator.
          if (!warp_wait<kRowMathPoll>(bar(C::bDQFull + bb), (gs >> 1) & 1, abort_flag, p.status)) {
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
        if (!ok) break;
        // Epilogue, by the warpgroup pair that ran the unit's last query step (the
        // other pair goes on to the next unit's first step meanwhile): dV, then
        // scale * dK, each warpgroup half of the columns. dK is read out after dV's
        // stores are issued; both accumulators are then released (AccFree) before
        // dK's stores, so the next unit's first dV / dK MMAs can start meanwhile.
        const bool epi = nsteps > 0 ? bb == ((G + nsteps - 1) & 1) : bb == 0;
        if (epi) {
          constexpr int kChunks = D / 64;  // 32-column TMEM loads per thread and accumulator
          const long long off = (long long)b * p.sb + (long long)(u.row0 + j) * p.sn + (long long)h * p.sh;
#pragma unroll 1
          for (int which = 0; which < 2; ++which) {
            const bool isK = which == 1;
            uint32_t r[kChunks][32];
            if (nsteps > 0) {
              if (!isK) {
                if (!warp_wait<kRowMathPoll>(bar(C::bAcc), kl & 1, abort_flag, p.status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              __syncwarp();  // the stores above are per-lane: converge for the TMEM loads
              const uint32_t col0 = (isK ? tdK : tdV) + lane_off + c * (D / 2);
              tmem_ld32(col0, r[0]);
              if constexpr (kChunks == 2) {
                tmem_ld32(col0 + 32, r[1]);
                tmem_ld_wait2(r[0], r[1]);
              } else {
                tmem_ld_wait(r[0]);
              }
              if (isK) {
                tc_fence_before();
                warp_arrive(bar(C::bAccFree));
              }
            } else {
#pragma unroll
              for (int cc = 0; cc < kChunks; ++cc)
#pragma unroll
                for (int x = 0; x < 32; ++x) r[cc][x] = 0u;
            }
            if (j < Nl) {
              uint16_t* dst = static_cast<uint16_t*>(isK ? p.dk : p.dv) + off + c * (D / 2);
              const float mul = isK ? p.scale : 1.f;
#pragma unroll
              for (int cc = 0; cc < kChunks; ++cc) {
                uint32_t w[16];
#pragma unroll
                for (int x = 0; x < 16; ++x)
                  w[x] = pack2<kBf16>(__uint_as_float(r[cc][2 * x]) * mul, __uint_as_float(r[cc][2 * x + 1]) * mul);
                uint4* gp = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
                for (int t = 0; t < 4; ++t) gp[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
              }
            }
          }
          if (!ok) break;
        }
        if (nsteps > 0) ++kl;
        (void)bh;
        G += nsteps;
      }
      idx = next_unit(k++);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // Persistent grid: the last CTA to leave resets the unit counter pair (next
  // ticket, CTAs done), so a later launch on the same workspace starts afresh
  // even without the preprocess in between. Each CTA's final ticket was taken
  // by this thread (the producer) before its fence.
  if (!ordered && p.unit_ctr != nullptr && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.unit_ctr + 1, 1u) == gridDim.x - 1) {
      p.unit_ctr[0] = 0u;
      p.unit_ctr[1] = 0u;
    }
  }
}

// Persistent grid of at most one CTA per SM (deterministic kernel); one CTA per
// unit with accumulated dQ (atomic and ordered modes).
template <int D, bool kBf16, bool kAtomic, bool kDrop, bool kAlibi, bool kBias>
static cudaError_t launch_dkdv_t(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  using C = KVCfg<D, kAtomic, kBias>;
  auto kern = bwd_dkdv_kernel<D, kBf16, kAtomic, kDrop, kAlibi, kBias>;
  const int smem = (int)(C::kSmem > kMinSmemOneCtaPerSm ? C::kSmem : kMinSmemOneCtaPerSm);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rows = p.cu_seqlens ? p.max_seqlen : p.N;
  const int units = p.cu_seqlens ? p.nseq * p.H : p.B * p.H;
  const long long total = (long long)((rows + kRowsKV - 1) / kRowsKV) * units;
  // Persistent in the deterministic kernel only: with accumulated dQ the next
  // unit's K / V would also wait for the last dQ^T MMAs (measured slower:
  // N = 2048 0.302 -> 0.329 ms, headline 1.58 -> 1.60 ms).
  long long grid = total;
  if (!kAtomic) {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    grid = total < sms ? total : sms;
  }
  kern<<<(unsigned)grid, C::kThreads, smem, st>>>(p, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5]);
  return cudaGetLastError();
}

template <int D, bool kBf16, bool kAtomic, bool kBias>
static cudaError_t launch_dkdv_b(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  const bool drop = p.drop.on != 0;
  if (p.alibi)
    return drop ? launch_dkdv_t<D, kBf16, kAtomic, true, true, kBias>(p, maps, st)
                : launch_dkdv_t<D, kBf16, kAtomic, false, true, kBias>(p, maps, st);
  return drop ? launch_dkdv_t<D, kBf16, kAtomic, true, false, kBias>(p, maps, st)
              : launch_dkdv_t<D, kBf16, kAtomic, false, false, kBias>(p, maps, st);
}

template <int D, bool kBf16, bool kAtomic>
static cudaError_t launch_dkdv_a(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  return p.bias ? launch_dkdv_b<D, kBf16, kAtomic, true>(p, maps, st) : launch_dkdv_b<D, kBf16, kAtomic, false>(p, maps, st);
}

template <int D, bool kBf16>
static cudaError_t launch_dkdv_d(const AttnParams& p, bool atomic, const CUtensorMap* maps, cudaStream_t st) {
  return atomic ? launch_dkdv_a<D, kBf16, true>(p, maps, st) : launch_dkdv_a<D, kBf16, false>(p, maps, st);
}

// maps: Q, K, V, dO (Q/dO boxes of kStepQ rows, K/V boxes of kRowsKV rows), the
// attention bias (boxes of kStepQ rows x kRowsKV keys; any valid map when
// p.bias is null), and the fp32 dQ accumulator as (d, rows per head, heads)
// with boxes of d x 32 rows (any valid map in the deterministic kernel).
cudaError_t launch_bwd_dkdv_tc(const AttnParams& p, bool bf16, bool atomic, const CUtensorMap* maps,
                               cudaStream_t st) {
  if (p.d == 128)
    return bf16 ? launch_dkdv_d<128, true>(p, atomic, maps, st) : launch_dkdv_d<128, false>(p, atomic, maps, st);
  return bf16 ? launch_dkdv_d<64, true>(p, atomic, maps, st) : launch_dkdv_d<64, false>(p, atomic, maps, st);
}

}  // namespace fa
