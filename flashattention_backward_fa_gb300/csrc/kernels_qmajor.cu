// Query-major kernels on the sm_103a tensor cores: the deterministic dQ kernel
// of the backward and the forward that produces O and L.
//
// dQ ("FlashAttention backward", §The loop structure, choice (b)): a separate
// kernel loops the other way — outer over query blocks, inner over key blocks —
// recomputing S and dP so that dQ accumulates in TMEM without atomics:
//   S = Q_i K_j^T, dP~ = dO_i V_j^T, P = exp2(S*scale*log2e - L_i*log2e),
//   dP = dP~ o Z/(1-p), dS = P o (dP - D_i), dQ_i += dS K_j; dQ = scale * dQ.
// The reduction order over key blocks is fixed, so dQ is bit-reproducible.
//
// Forward ("FlashAttention backward", §What the forward left behind): the
// output O and the per-row log-sum-exp L = m + log(l) (natural log), in one
// pass with an online softmax. Per key block the four row-math warpgroups
// exchange their chunk maxima of each row through shared memory; a row's
// reference maximum moves only when the maximum grows by more than 2^8 (so the
// probabilities relative to it stay below 2^8), and then the O accumulator's
// row is rescaled in TMEM once the previous O MMA has finished. Each warpgroup
// keeps its columns' partial sum l relative to the reference; at the end
// O = acc / l and L = (reference + log2 l) * ln 2. Dropout: O += (P o Z/(1-p)) V,
// with l taken before dropout.
//
// Queries sit on the 128 TMEM lanes: one thread owns one query row, so L_i and
// D_i are per-thread scalars. Row-math warps wait warp-wide (warp_wait) and
// reconverge after per-lane branches: TMEM loads and stores are warp-collective
// (.aligned) and must not run on a split warp. A step covers 128 keys, so every S, dP and
// accumulating MMA has N = 128 (N = 64 MMAs are limited by shared-memory
// operand reads to about two thirds of the tensor rate). The row math writes
// dS (or P~) back over the S columns it has read, rounded to 16 bits with the
// rounding residual beside it (see interleave_split), and the accumulating MMA
// reads it from TMEM. In the dQ kernel S alternates between two TMEM buffers
// and dP has one, which the row math releases as soon as it has read it; the
// forward, with no dP, rotates S over three buffers.
//
// Shared memory holds Q (and dO) for the whole kernel and two rings of key
// tiles: ring E for the tile only the first MMAs read (V for dP; K in the
// forward) and ring L for the tile the accumulating MMA reads (K, which S
// also reads; V in the forward), so that E tiles are recycled early.
//
// Warp 0 issues TMA loads, warp 1 owns TMEM and issues the S MMAs, warp 3 the
// dP MMAs and warp 2 the accumulating MMAs, so the three streams go out in
// parallel. Four row-math warpgroups (warps 4-19) each take 32 of the step's
// 128 key columns and a quarter of the epilogue columns.
//
// Persistent grid (dQ kernel): one CTA per SM runs unit after unit (query
// blocks), taking the next from a counter in the workspace (the first is its
// blockIdx). Steps, ring stages, TMEM buffers and barrier phases continue from
// one unit to the next, so the next unit's loads and first S / dP MMAs overlap
// the current unit's last steps and epilogue; the next unit's Q and dO
// overwrite this unit's once its last S / dP MMAs have completed (ResFree), and
// its first accumulating MMA overwrites the accumulator once every row-math
// warp has loaded it (AccFree). The producer publishes each next unit in a
// small ring in shared memory. The forward runs the same code with one unit
// per CTA (it has no workspace for a counter).
//
// TMEM columns: dQ kernel [0,256) two S buffers, [256,384) the dP buffer;
// forward [0,384) three S buffers; then [384,384+d) the dQ or O accumulator.
#include "fa_internal.h"

namespace fa {

constexpr int kModeFwd = 0;
constexpr int kModeDq = 1;
constexpr int kQThreads = 640;  // 4 role warps + 4 row-math warpgroups
constexpr int kQUnitSlots = 4;   // ring of published units

template <int D, int kMode, bool kBias = false>
struct QCfg {
  static constexpr bool kDq = kMode == kModeDq;
  static constexpr int kPanels = D / 64;
  static constexpr uint32_t kPanel = 128 * 128;                // 16 KB: 128 rows x 64 elements
  static constexpr uint32_t kTile = kPanels * kPanel;          // one 128-row tile of Q, dO, K or V
  static constexpr uint32_t kResident = (kDq ? 2 : 1) * kTile;
  // forward: per-step chunk maxima [2 steps][4 warpgroups][rows], then the
  // final partial sums [4 warpgroups][rows]
  static constexpr uint32_t kStats = kDq ? 0 : (2 * 4 + 4) * kRowsQ * 4;
  // ring depths; with an attention bias the deeper ring gives up a stage (d = 128)
  // to make room for the bias tile
  static constexpr int kNE = kDq ? 2 : (D == 64 ? 4 : (kBias ? 2 : 3));  // ring E stages
  static constexpr int kNL = kDq ? (D == 64 ? 4 : (kBias ? 2 : 3)) : 2;  // ring L stages
  // attention bias of a step: 128 query rows x 128 keys, 16-bit, as two
  // 128-byte-swizzled panels of 64 keys (one buffer, refilled once the row
  // math has copied its segments to registers)
  static constexpr uint32_t kBiasPanel = 128 * 128;
  static constexpr uint32_t kBiasTile = kBias ? 2 * kBiasPanel : 0;
  // S buffers in TMEM: two beside the dP buffer in the dQ kernel; three in the
  // forward, which has no dP.
  static constexpr int kSBuf = kDq ? 2 : 3;
  static constexpr uint32_t oQ = 0;
  static constexpr uint32_t oDO = oQ + kTile;
  static constexpr uint32_t oE = kResident;
  static constexpr uint32_t oL = oE + kNE * kTile;
  static constexpr uint32_t oBias = oL + kNL * kTile;
  static constexpr uint32_t oStats = oBias + kBiasTile;         // forward: row-statistics exchange
  static constexpr uint32_t oBar = oStats + kStats;
  static constexpr int bRes = 0;
  static constexpr int bEFull = 1;
  static constexpr int bEEmpty = bEFull + kNE;
  static constexpr int bLFull = bEEmpty + kNE;
  static constexpr int bLEmpty = bLFull + kNL;
  static constexpr int bSFull = bLEmpty + kNL;                 // [kSBuf]: S (and dP) landed
  static constexpr int bSEmpty = bSFull + kSBuf;               // [kSBuf]: accumulating MMA done with the image
  static constexpr int bDPEmpty = bSEmpty + kSBuf;             // row math has read dP
  static constexpr int bPFull = bDPEmpty + 1;                  // [kSBuf]: image written
  static constexpr int bAcc = bPFull + kSBuf;
  static constexpr int bDrain = bAcc + 1;                      // one per MMA-issuing warp
  static constexpr int bStats = bDrain + 3;                    // forward: final sums exchanged
  static constexpr int bXchg = bStats + 1;                     // [2][4] forward: chunk maxima of step it exchanged (per row quarter)
  static constexpr int bODone = bXchg + 8;                     // forward: O MMA of a step done
  static constexpr int bBFull = bODone + 1;                    // bias tile landed
  static constexpr int bBEmpty = bBFull + 1;                   // row math has copied the bias tile
  static constexpr int bResFree = bBEmpty + 1;                 // a unit's last reads of Q (and dO) done
  static constexpr int bAccFree = bResFree + 1;                // the epilogue has read the accumulator
  static constexpr int bUnit = bAccFree + 1;                   // [kQUnitSlots]: next unit published
  static constexpr int bUnitFree = bUnit + kQUnitSlots;        // [kQUnitSlots]: ring slot read by all
  static constexpr int kBars = bUnitFree + kQUnitSlots;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = (oAbort + 8 + 15) & ~15u;  // [buffer][16 warps] split votes
  static constexpr uint32_t oUnits = oFlags + kSBuf * 16 * 4;  // [kQUnitSlots] unit ring
  static constexpr uint32_t kSmem = oUnits + 4 * kQUnitSlots + 1024;  // + slack for 1024-byte alignment
  static_assert(kSmem <= 227u * 1024u, "shared memory budget exceeded");
};

// Forward: the reference maximum of a row moves only when the row maximum grows by
// more than this (log2 units), bounding relative probabilities by 2^8.
constexpr float kRescaleLog2 = 8.f;

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr));
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool kBf16, int kMode, bool kDrop, bool kAlibi, bool kBias>
__global__ void __launch_bounds__(kQThreads, 1)
    qmajor_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmBias) {
  using C = QCfg<D, kMode, kBias>;
  constexpr bool kDq = kMode == kModeDq;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oAbort);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + C::oFlags);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + C::oUnits);
  auto bar = [&](int idx) -> uint32_t { return sb + C::oBar + 8u * idx; };
  const bool packed = p.cu_seqlens != nullptr;
  const int total_units = ((packed ? p.max_seqlen : p.N) + kRowsQ - 1) / kRowsQ * (packed ? p.nseq * p.H : p.B * p.H);
  // the dQ kernel's pair of the workspace unit counters (null: a fixed stride)
  unsigned int* const ctr = (kDq && p.unit_ctr != nullptr) ? p.unit_ctr + 2 : nullptr;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bRes), 1);
    for (int s = 0; s < C::kNE; ++s) {
      mbar_init(bar(C::bEFull + s), 1);
      mbar_init(bar(C::bEEmpty + s), 1);
    }
    for (int s = 0; s < C::kNL; ++s) {
      mbar_init(bar(C::bLFull + s), 1);
      mbar_init(bar(C::bLEmpty + s), 1);
    }
    for (int x = 0; x < C::kSBuf; ++x) {
      mbar_init(bar(C::bSFull + x), kDq ? 2 : 1);
      mbar_init(bar(C::bSEmpty + x), 1);
      mbar_init(bar(C::bPFull + x), 512);
    }
    mbar_init(bar(C::bDPEmpty), 512);
    mbar_init(bar(C::bAcc), 1);
    for (int x = 0; x < 3; ++x) mbar_init(bar(C::bDrain + x), 1);
    mbar_init(bar(C::bStats), 512);
    for (int x = 0; x < 8; ++x) mbar_init(bar(C::bXchg + x), 128);
    mbar_init(bar(C::bODone), 1);
    mbar_init(bar(C::bBFull), 1);
    mbar_init(bar(C::bBEmpty), 512);
    mbar_init(bar(C::bResFree), kDq ? 2 : 1);                  // S (and dP) issuers
    mbar_init(bar(C::bAccFree), 512);                          // every row-math warp
    for (int x = 0; x < kQUnitSlots; ++x) {
      mbar_init(bar(C::bUnit + x), 1);
      mbar_init(bar(C::bUnitFree + x), 19 * 32);               // warps 1-3 and the row-math warps
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
    if (kDq) prefetch_tmap(&tmDO);
    if (kBias) prefetch_tmap(&tmBias);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::oTmemSlot);
  const uint32_t tS = tmem, tdP = tmem + 256, tAcc = tmem + 384;

  // Work unit: (batch*head or sequence*head, query block), heaviest query
  // blocks first under a causal mask; a block past the end of its sequence has
  // no work. Every role decodes the units the producer publishes.
  struct QUnit {
    Unit u;
    int i0, j_first, nsteps;
  };
  auto q_unit = [&](int idx, QUnit& g) -> bool {
    if (!unit_decode(p, idx, kRowsQ, true, g.u)) return false;
    g.i0 = g.u.tile * kRowsQ;
    const int j_last = p.causal ? min(g.u.n - 1, g.i0 + kRowsQ - 1) : g.u.n - 1;
    g.j_first = p.window > 0 ? (max(0, g.i0 - p.window + 1) / kStepKV) * kStepKV : 0;
    g.nsteps = (j_last >= g.j_first) ? (j_last - g.j_first) / kStepKV + 1 : 0;  // one pass over the key blocks
    return true;
  };
  // Key block of step it. Ascending, except in the ALiBi forward: there the
  // blocks go outward from the one holding this tile's diagonal (nearest first,
  // alternating below and above), so that every row meets its largest biased
  // scores early and the online softmax's reference rarely has to move.
  auto key_block = [&](const QUnit& g, int it) -> int {
    if constexpr (kAlibi && !kDq) {
      const int nkv = g.nsteps;
      const int gd = min(max((g.i0 - g.j_first) / kStepKV, 0), nkv - 1);
      const int below = gd, above = nkv - 1 - gd, m = min(below, above);
      int t;
      if (it == 0) t = gd;
      else if (it <= 2 * m) t = (it & 1) ? gd - (it + 1) / 2 : gd + it / 2;
      else t = below > above ? gd - (it - m) : gd + (it - m);
      return g.j_first + t * kStepKV;
    } else {
      return g.j_first + it * kStepKV;
    }
  };
  // The unit after this CTA's k-th one, from ring slot k % kQUnitSlots (every
  // role but the producer; warp-wide). -1: no more units (or the CTA aborted).
  auto next_unit = [&](int k) -> int {
    const int s = k % kQUnitSlots;
    if (!warp_wait<kIssuerPoll>(bar(C::bUnit + s), (k / kQUnitSlots) & 1, abort_flag, p.status)) return -1;
    const int idx = unit_ring[s];
    __syncwarp();
    warp_arrive(bar(C::bUnitFree + s));
    return idx;
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    // Step it: ring E gets V (dQ) or K (forward); ring L gets K (dQ) or V
    // (forward). Stages are counted across units.
    if (lane == 0) {
      const CUtensorMap* mE = kDq ? &tmV : &tmK;
      const CUtensorMap* mL = kDq ? &tmK : &tmV;
      int idx = blockIdx.x, k = 0, kl = 0, G = 0;  // units seen / loaded, steps before this unit
      int issuedE = 0, issuedL = 0, issuedB = 0;    // (global) stages issued
      bool ok = true;
      while (ok && idx >= 0) {
        int next_idx = -1;
        // The ticket of the unit after this one is taken first (its latency
        // overlaps this unit's loads); the unit is published once they are issued.
        const unsigned int tk = ctr ? atomicAdd(ctr, 1u) : 0u;
        auto publish_next = [&]() -> bool {
          int nxt = -1;
          int cand = ctr ? (int)(gridDim.x + tk) : idx + (int)gridDim.x;
          for (;;) {  // query blocks past their sequence are skipped
            if (cand >= total_units) break;
            QUnit gn;
            if (q_unit(cand, gn)) {
              nxt = cand;
              break;
            }
            cand = ctr ? (int)(gridDim.x + atomicAdd(ctr, 1u)) : cand + (int)gridDim.x;
          }
          if (!mbar_wait(bar(C::bUnitFree + k % kQUnitSlots), ((k / kQUnitSlots) & 1) ^ 1, abort_flag, p.status))
            return false;
          unit_ring[k % kQUnitSlots] = nxt;
          mbar_arrive(bar(C::bUnit + k % kQUnitSlots));
          next_idx = nxt;
          return true;
        };
        QUnit g;
        if (q_unit(idx, g)) {
          const Unit& u = g.u;
          const int b = u.b, h = u.h, i0 = g.i0;
          // Q (and dO) of this unit, once the previous unit's last reads of them are done
          if (kl > 0 && !mbar_wait(bar(C::bResFree), (kl - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::bRes), C::kResident);
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_4d(sb + C::oQ + pn * C::kPanel, &tmQ, bar(C::bRes), 64 * pn, u.row0 + i0, h, b);
            if (kDq) tma_load_4d(sb + C::oDO + pn * C::kPanel, &tmDO, bar(C::bRes), 64 * pn, u.row0 + i0, h, b);
          }
          ++kl;
          for (int it = 0; ok && it < g.nsteps; ++it) {
            const int gs = G + it;
            const int jj = key_block(g, it);
            const int se = gs % C::kNE;
            if (!mbar_wait(bar(C::bEEmpty + se), ((gs / C::kNE) & 1) ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(C::bEFull + se), C::kTile);
            for (int pn = 0; pn < C::kPanels; ++pn)
              tma_load_4d(sb + C::oE + se * C::kTile + pn * C::kPanel, mE, bar(C::bEFull + se), 64 * pn,
                          u.row0 + jj, h, b);
            issuedE = gs + 1;
            const int sl = gs % C::kNL;
            if (!mbar_wait(bar(C::bLEmpty + sl), ((gs / C::kNL) & 1) ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(C::bLFull + sl), C::kTile);
            for (int pn = 0; pn < C::kPanels; ++pn)
              tma_load_4d(sb + C::oL + sl * C::kTile + pn * C::kPanel, mL, bar(C::bLFull + sl), 64 * pn,
                          u.row0 + jj, h, b);
            issuedL = gs + 1;
            if constexpr (kBias) {
              // the step's bias tile, once the row math has copied the previous one
              if (!mbar_wait(bar(C::bBEmpty), (gs & 1) ^ 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(bar(C::bBFull), C::kBiasTile);
              for (int pn = 0; pn < 2; ++pn)
                tma_load_4d(sb + C::oBias + pn * C::kBiasPanel, &tmBias, bar(C::bBFull), jj + 64 * pn,
                            u.row0 + i0, p.bias_sh ? h : 0, p.bias_sb ? b : 0);
              issuedB = gs + 1;
            }
          }
          G += g.nsteps;
        }
        if (ok && !publish_next()) ok = false;
        idx = next_idx;
        ++k;
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        if (kl > 0) mbar_wait_drain(bar(C::bRes), (kl - 1) & 1, p.status);
        for (int x = max(0, issuedE - C::kNE); x < issuedE; ++x)
          mbar_wait_drain(bar(C::bEFull + x % C::kNE), (x / C::kNE) & 1, p.status);
        for (int x = max(0, issuedL - C::kNL); x < issuedL; ++x)
          mbar_wait_drain(bar(C::bLFull + x % C::kNL), (x / C::kNL) & 1, p.status);
        if (issuedB > 0) mbar_wait_drain(bar(C::bBFull), (issuedB - 1) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ S MMA issuer ------------------------------
    {
      constexpr uint32_t idS = make_idesc(128, kStepKV, kBf16, false, false);
      const uint64_t dQ0 = make_sdesc(sb + C::oQ, 16, 1024);
      const uint64_t dK0 = make_sdesc(sb + (kDq ? C::oL : C::oE), 16, 1024);
      int idx = blockIdx.x, k = 0, kl = 0, G = 0;
      bool ok = true;
      while (ok && idx >= 0) {
        QUnit g;
        if (q_unit(idx, g)) {
          ok = warp_wait<kIssuerPoll>(bar(C::bRes), kl & 1, abort_flag, p.status);
          for (int it = 0; ok && it < g.nsteps; ++it) {
            const int gs = G + it;
            const int bb = gs % C::kSBuf;
            // K lives in ring L (dQ; one tile per step) or ring E (forward)
            const int ks = kDq ? gs % C::kNL : gs % C::kNE;
            const uint32_t kpar = kDq ? (gs / C::kNL) & 1 : (gs / C::kNE) & 1;
            if (!warp_wait<kIssuerPoll>(bar((kDq ? C::bLFull : C::bEFull) + ks), kpar, abort_flag, p.status) ||
                !warp_wait<kIssuerPoll>(bar(C::bSEmpty + bb), ((gs / C::kSBuf) & 1) ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t kd = desc_add(dK0, ks * C::kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss_w(tS + 128 * bb, desc_add(dQ0, (kk >> 2) * C::kPanel + (kk & 3) * 32),
                          desc_add(kd, (kk >> 2) * C::kPanel + (kk & 3) * 32), idS, kk > 0 ? 1u : 0u);
            tc_commit_w(bar(C::bSFull + bb));
            if (!kDq) tc_commit_w(bar(C::bEEmpty + ks));   // forward: K is done once S is
          }
          if (!ok) break;
          tc_commit_w(bar(C::bResFree));  // this unit's last reads of Q
          G += g.nsteps;
          ++kl;
        }
        idx = next_unit(k++);
      }
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      tc_commit_w(bar(C::bDrain));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain), 0, p.status);
      __syncwarp();
    }
  } else if (warp == 3) {
    // ---------------------- dP MMA issuer (dQ mode only) ----------------------
    if (kDq) {
      constexpr uint32_t idS = make_idesc(128, kStepKV, kBf16, false, false);
      const uint64_t dO0 = make_sdesc(sb + C::oDO, 16, 1024), dV0 = make_sdesc(sb + C::oE, 16, 1024);
      int idx = blockIdx.x, k = 0, kl = 0, G = 0;
      bool ok = true;
      while (ok && idx >= 0) {
        QUnit g;
        if (q_unit(idx, g)) {
          ok = warp_wait<kIssuerPoll>(bar(C::bRes), kl & 1, abort_flag, p.status);
          for (int it = 0; ok && it < g.nsteps; ++it) {
            const int gs = G + it;
            const int se = gs % C::kNE;
            if (!warp_wait<kIssuerPoll>(bar(C::bEFull + se), (gs / C::kNE) & 1, abort_flag, p.status) ||
                (gs > 0 && !warp_wait<kIssuerPoll>(bar(C::bDPEmpty), (gs - 1) & 1, abort_flag, p.status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vd = desc_add(dV0, se * C::kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss_w(tdP, desc_add(dO0, (kk >> 2) * C::kPanel + (kk & 3) * 32),
                          desc_add(vd, (kk >> 2) * C::kPanel + (kk & 3) * 32), idS, kk > 0 ? 1u : 0u);
            tc_commit_w(bar(C::bSFull + gs % C::kSBuf));
            tc_commit_w(bar(C::bEEmpty + se));
          }
          if (!ok) break;
          tc_commit_w(bar(C::bResFree));  // this unit's last reads of dO
          G += g.nsteps;
          ++kl;
        }
        idx = next_unit(k++);
      }
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      tc_commit_w(bar(C::bDrain + 2));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain + 2), 0, p.status);
      __syncwarp();
    } else {
      // forward: no dP; this warp still reads the unit ring
      int idx = blockIdx.x, k = 0;
      while (idx >= 0) idx = next_unit(k++);
    }
  } else if (warp == 2) {
    // ------------------ accumulating MMA issuer (O or dQ) ---------------------
    // After the row math of step t: acc += (P~ or dS) . (V_j or K_j), then
    // release the S buffer and the ring-L tile.
    {
      constexpr uint32_t idO = make_idesc(128, D, kBf16, false, true);
      const uint64_t b0 = make_sdesc(sb + C::oL, C::kPanel, 1024);
      int idx = blockIdx.x, k = 0, kl = 0, G = 0;
      bool ok = true;
      while (ok && idx >= 0) {
        QUnit g;
        if (q_unit(idx, g) && g.nsteps > 0) {
          for (int t = 0; ok && t < g.nsteps; ++t) {
            const int gs = G + t;
            const int bt = gs % C::kSBuf;
            if (!warp_wait<kConsumerPoll>(bar(C::bPFull + bt), (gs / C::kSBuf) & 1, abort_flag, p.status) ||
                // the first MMA of a unit overwrites the accumulator the previous
                // unit's epilogue reads
                (t == 0 && kl > 0 && !warp_wait<kConsumerPoll>(bar(C::bAccFree), (kl - 1) & 1, abort_flag, p.status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int sl = gs % C::kNL;
            // Forward: V (ring L) must have landed before the MMA reads it. In the dQ
            // kernel ring L holds K, whose arrival the S issuer waited for before S.
            if (!kDq && !warp_wait<kIssuerPoll>(bar(C::bLFull + sl), (gs / C::kNL) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            const uint32_t first = t > 0 ? 1u : 0u;  // the first step overwrites the accumulator
            const int4* f4 = reinterpret_cast<const int4*>(const_cast<const int*>(flags) + 16 * bt);
            int any = 0;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const int4 v = f4[x];
              any |= v.x | v.y | v.z | v.w;
            }
            const uint64_t bop = desc_add(b0, sl * C::kTile);
#pragma unroll
            for (int kk = 0; kk < kStepKV / 16; ++kk)
              tc_mma_ts_w(tAcc, tS + 128 * bt + 16 * kk, desc_add(bop, 2048 * kk), idO, kk > 0 ? 1u : first);
            if (any) {
#pragma unroll
              for (int kk = 0; kk < kStepKV / 16; ++kk)
                tc_mma_ts_w(tAcc, tS + 128 * bt + 16 * kk + 8, desc_add(bop, 2048 * kk), idO, 1u);
            }
            tc_commit_w(bar(C::bSEmpty + bt));
            tc_commit_w(bar(C::bLEmpty + sl));
            if (!kDq) tc_commit_w(bar(C::bODone));
          }
          if (!ok) break;
          tc_commit_w(bar(C::bAcc));
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
    // ---------------- row-math warpgroups + epilogue ----------------------
    // Warpgroup c takes key columns [32c, 32c + 32) of every step, in halves of
    // 16 columns (one MMA K step), and a quarter of the epilogue columns.
    const int c = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int il = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tdPc = tdP + lane_off + 32 * c;
    const float inv_scale = kBias ? 1.f / p.scale : 0.f;
    float* xchg = reinterpret_cast<float*>(smem + C::oStats);
    int idx = blockIdx.x, k = 0, kl = 0, G = 0;
    bool ok = true;
    while (ok && idx >= 0) {
      QUnit g;
      if (q_unit(idx, g)) {
        const Unit& u = g.u;
        const int bh = u.bh, b = u.b, h = u.h;
        const int Nl = u.n;                    // rows of this (batch, head) or sequence
        const int i = g.i0 + il;
        const int nsteps = g.nsteps;
        const long long ws = u.ws + i;  // i < the padded row count always
        // dQ: -L*log2(e) (-inf for a row with no allowed key) and -D, read; the
        // negated forms are addends of one FMA / add (packed two-wide below).
        // Forward: mref, the running reference maximum of S*scale*log2e over the
        // keys seen so far (log2 domain), shared by the four warpgroups, and lsum,
        // this warpgroup's sum of exp2(S*scale*log2e - mref) over its columns.
        float nL2 = -INFINITY, nD = 0.f;
        if (kDq) {
          nL2 = p.ws_nL2[ws];
          nD = p.ws_nD[ws];
        }
        const float slope_raw = kAlibi ? alibi_slope_raw(p, u) : 0.f;
        float mref = -INFINITY, lsum = 0.f;
        auto key_block_u = [&](int it) { return key_block(g, it); };
        for (int it = 0; it < nsteps; ++it) {
          const int gs = G + it;  // step counted across units
          const int bb = gs % C::kSBuf, xb = gs & 1;
          const int base = key_block_u(it) + 32 * c;
          const uint32_t tSc = tS + lane_off + 128 * bb + 32 * c;
          // This row's bias over the chunk's 32 keys (four 16-byte pieces of the
          // swizzled tile; zeros past N), copied to registers so that the buffer is
          // released, and the next step's tile loads, before this step's row math.
          uint32_t bw[16];
          if constexpr (kBias) {
            if (!warp_wait<kRowMathPoll>(bar(C::bBFull), gs & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            const uint32_t rowa = sb + C::oBias + (uint32_t)(c >> 1) * C::kBiasPanel + (uint32_t)il * 128;
    #pragma unroll
            for (int t = 0; t < 4; ++t)
              ld_shared_v4(rowa + ((uint32_t)((4 * (c & 1) + t) ^ (il & 7)) << 4), bw[4 * t], bw[4 * t + 1],
                           bw[4 * t + 2], bw[4 * t + 3]);
            warp_arrive(bar(C::bBEmpty));
          }
          // allowed keys of this warpgroup's 32 columns (bit x <-> key base + x) and
          // their dropout keep bits: both depend on positions only, so the Philox
          // calls run while the S MMAs of this step are still in flight.
          const uint32_t allow =
              bit_range(p.window > 0 ? i - p.window + 1 - base : 0, min(Nl - base, p.causal ? i + 1 - base : 32));
          uint32_t keep = 0xFFFFFFFFu;
          if constexpr (kDrop) keep = keep_bits_for_query(p.drop, bh, Nl, i, base);
          if (!warp_wait<kRowMathPoll>(bar(C::bSFull + bb), (gs / C::kSBuf) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dQ: both halves of this warpgroup's dP columns come in with S, so the dP
          // buffer is released (and the next dP MMAs may run) before any arithmetic.
          // Forward: all of S comes in, for the row maximum.
          // (dQ: the second S half comes in after the first half's arithmetic,
          // which keeps fewer registers live.)
          uint32_t sr2[2][16], dr2[2][16];
          __syncwarp();
          tmem_ld16(tSc, sr2[0]);
          if constexpr (kDq) {
            tmem_ld16(tdPc, dr2[0]);
            tmem_ld16(tdPc + 16, dr2[1]);
            tmem_ld_wait16x3(sr2[0], dr2[0], dr2[1]);
            tc_fence_before();
            warp_arrive(bar(C::bDPEmpty));
          } else {
            tmem_ld16(tSc + 16, sr2[1]);
            tmem_ld_wait16x2(sr2[0], sr2[1]);
          }
          // attention bias, in score units (the dQ kernel's second half follows its load)
          if constexpr (kBias) {
            bias_fold16_regs<kBf16>(sr2[0], bw, inv_scale);
            if constexpr (!kDq) bias_fold16_regs<kBf16>(sr2[1], bw + 8, inv_scale);
          }
          // ALiBi: where every allowed key of this chunk lies on one side of the
          // diagonal (always under a causal mask), the bias -m|i - j| is a row
          // constant plus a ramp over the chunk's columns: the ramp goes into the
          // raw scores (one FMA a score) and the constant, rc2 (log2 domain), into
          // the exp2 addend. A chunk that straddles the diagonal folds |i - j| in.
          float rc2 = 0.f, ramp = 0.f;
          bool straddle = false;
          if constexpr (kAlibi) {
            const int dd = i - base;  // i - j of the chunk's column 0
            if (p.causal || dd >= 31) {
              ramp = slope_raw;
              rc2 = -slope_raw * (float)dd * p.scale_log2;
            } else if (dd <= 0) {
              ramp = -slope_raw;
              rc2 = slope_raw * (float)dd * p.scale_log2;
            } else {
              straddle = true;
            }
            auto fold = [&](auto half) {
              constexpr int hx = decltype(half)::value;
              if (straddle)
                alibi_fold16<-1>(sr2[hx], (float)(dd - 16 * hx), slope_raw);
              else
                alibi_ramp16<16 * hx>(sr2[hx], ramp);
            };
            fold(std::integral_constant<int, 0>{});
            if constexpr (!kDq) fold(std::integral_constant<int, 1>{});
          }
          bool resc = false;
          float alpha = 1.f;
          if constexpr (!kDq) {
            // Online softmax: the maximum of this step's 128 columns of the row,
            // from the four warpgroups' chunk maxima exchanged through shared memory.
            // (Full tiles with a positive scale take the maximum on S and scale it
            // once, without the per-column mask.)
            float cm = -INFINITY;
            if (allow == 0xFFFFFFFFu && p.scale_log2 > 0.f) {
    #pragma unroll
              for (int hh = 0; hh < 2; ++hh)
    #pragma unroll
                for (int e = 0; e < 16; e += 2)
                  cm = fmax3(cm, __uint_as_float(sr2[hh][e]), __uint_as_float(sr2[hh][e + 1]));
              cm = cm * p.scale_log2;
            } else {
    #pragma unroll
              for (int hh = 0; hh < 2; ++hh)
    #pragma unroll
                for (int e = 0; e < 16; ++e)
                  cm = ((allow >> (16 * hh + e)) & 1u) ? fmaxf(cm, __uint_as_float(sr2[hh][e]) * p.scale_log2) : cm;
            }
            if constexpr (kAlibi) cm += rc2;  // -inf stays -inf
            xchg[(xb * 4 + c) * kRowsQ + il] = cm;
            // Rows 32 wq .. 32 wq + 31 are shared by the four warps with this wq (one
            // per warpgroup, all on one scheduler): only they exchange.
            warp_arrive(bar(C::bXchg + 4 * xb + wq));
            // A blocking wait: the warps still computing their maxima share the
            // schedulers with the ones waiting here, and a spinning wait would take
            // their issue slots.
            if (!warp_wait<false>(bar(C::bXchg + 4 * xb + wq), (gs >> 1) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            float mstep = -INFINITY;
    #pragma unroll
            for (int g = 0; g < 4; ++g) mstep = fmaxf(mstep, xchg[(xb * 4 + g) * kRowsQ + il]);
            // The reference moves only when the maximum grows by more than 2^8 (or
            // the row sees its first allowed key): probabilities relative to a stale
            // reference stay below 2^8, and the O accumulator is rescaled rarely.
            if (mstep > mref + kRescaleLog2) {
              resc = mref != -INFINITY;
              alpha = resc ? ex2_approx(mref - mstep) : 1.f;
              lsum *= alpha;
              mref = mstep;
            }
            nL2 = -mref;  // P = exp2(S*scale*log2e + (-mref)); +inf only where every key so far is masked
            // With a bias, an allowed score may be -inf: while a row has no finite
            // score its addend must stay finite (-inf + inf is NaN).
            if constexpr (kBias) nL2 = mref == -INFINITY ? 0.f : nL2;
          }
          const float nL2c = kAlibi ? nL2 + rc2 : nL2;  // the exp2 addend of this chunk
          bool lo_any = false;
    #pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (kDq && hh == 1) {
              __syncwarp();
              tmem_ld16(tSc + 16, sr2[1]);
              tmem_ld_wait16(sr2[1]);
              if constexpr (kBias) bias_fold16_regs<kBf16>(sr2[1], bw + 8, inv_scale);
              if constexpr (kAlibi) {
                if (straddle)
                  alibi_fold16<-1>(sr2[1], (float)(i - base - 16), slope_raw);
                else
                  alibi_ramp16<16>(sr2[1], ramp);
              }
            }
            const uint32_t (&sr)[16] = sr2[hh];
            const uint32_t (&dr)[16] = dr2[hh];
            float outv[16];
            float cmax = 0.f, psum = 0.f;
            uint64_t psum2 = f2_pack(0.f, 0.f);
            auto elementwise = [&](auto masked) {
              if constexpr (!kDrop) {
                // pairs of columns through the packed FMA / add / multiply
                const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2), l2 = f2_pack(nL2c, nL2c);
    #pragma unroll
                for (int e = 0; e < 16; e += 2) {
                  float p0, p1;
                  f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, l2), p0, p1);
                  p0 = ex2_approx(p0);
                  p1 = ex2_approx(p1);
                  if constexpr (decltype(masked)::value) {
                    p0 = ((allow >> (16 * hh + e)) & 1u) ? p0 : 0.f;
                    p1 = ((allow >> (16 * hh + e + 1)) & 1u) ? p1 : 0.f;
                  }
                  cmax = fmax3(cmax, p0, p1);
                  if constexpr (kDq) {
                    const uint64_t dd = f2_add(f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), f2_pack(nD, nD));
                    f2_unpack(f2_mul(f2_pack(p0, p1), dd), outv[e], outv[e + 1]);
                  } else {
                    psum2 = f2_add(psum2, f2_pack(p0, p1));
                    outv[e] = p0;
                    outv[e + 1] = p1;
                  }
                }
              } else {
                // dropout: the same pairs of columns, with the keep decisions as selects
                const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2), l2 = f2_pack(nL2c, nL2c);
                const uint64_t rp2 = f2_pack(p.drop.rp, p.drop.rp), nD2 = f2_pack(nD, nD);
    #pragma unroll
                for (int e = 0; e < 16; e += 2) {
                  const int bit = 16 * hh + e;
                  float p0, p1;
                  f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, l2), p0, p1);
                  p0 = ex2_approx(p0);
                  p1 = ex2_approx(p1);
                  if constexpr (decltype(masked)::value) {
                    p0 = ((allow >> bit) & 1u) ? p0 : 0.f;
                    p1 = ((allow >> (bit + 1)) & 1u) ? p1 : 0.f;
                  }
                  cmax = fmax3(cmax, p0, p1);
                  const bool k0 = (keep >> bit) & 1u, k1 = (keep >> (bit + 1)) & 1u;
                  if constexpr (kDq) {
                    // dS = P * (kept ? dP~ / (1-p) - D : -D)
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), rp2, nD2), a0, a1);
                    f2_unpack(f2_mul(f2_pack(p0, p1), f2_pack(k0 ? a0 : nD, k1 ? a1 : nD)), outv[e], outv[e + 1]);
                  } else {
                    psum2 = f2_add(psum2, f2_pack(p0, p1));
                    f2_unpack(f2_mul(f2_pack(p0, p1), f2_pack(k0 ? p.drop.rp : 0.f, k1 ? p.drop.rp : 0.f)), outv[e],
                              outv[e + 1]);
                  }
                }
              }
            };
            // nL2 = -inf (a row with no allowed key) gives exp2(-inf) = 0 on the fast path too.
            if (allow == 0xFFFFFFFFu)
              elementwise(std::false_type{});
            else
              elementwise(std::true_type{});
            // The lanes may have split over the two variants: reconverge before the
            // warp-collective vote and TMEM stores below.
            __syncwarp();
            if constexpr (!kDq) {
              float s0, s1;
              f2_unpack(psum2, s0, s1);
              lsum += psum + (s0 + s1);
            }
            uint32_t hv[8], ev[8];
    #pragma unroll
            for (int x = 0; x < 8; ++x) hv[x] = pack2<kBf16>(outv[2 * x], outv[2 * x + 1]);
            // Residuals where a probability can exceed the split threshold. In the
            // forward the values are relative to the reference (exp(s - m)) and
            // lsum, this warpgroup's sum over the keys seen so far including these
            // columns, is a part of the final row sum: P = exp(s - m) / (full sum)
            // <= cmax / lsum, whatever keys and reference moves come later.
            const bool split_h = __any_sync(0xFFFFFFFFu, kDq ? cmax > kSplitThreshold : cmax > kSplitThreshold * lsum);
            lo_any |= split_h;
            if (split_h) {
    #pragma unroll
              for (int x = 0; x < 8; ++x) ev[x] = pack2_residual<kBf16>(outv[2 * x], outv[2 * x + 1], hv[x]);
            } else {
    #pragma unroll
              for (int x = 0; x < 8; ++x) ev[x] = 0u;
            }
            // this K step's image: 8 rounded columns, then 8 residual columns
            tmem_st8<0>(tSc + 16 * hh, hv);
            tmem_st8<0>(tSc + 16 * hh + 8, ev);
          }
          if constexpr (!kDq) {
            // Rescale this warpgroup's quarter of the O columns of rows whose
            // reference moved, once the O MMA of the previous step has finished.
            if (__any_sync(0xFFFFFFFFu, resc)) {
              if (it > 0 && !warp_wait<kRowMathPoll>(bar(C::bODone), (gs - 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
    #pragma unroll
              for (int cc = 0; cc < D / 64; ++cc) {
                const uint32_t ta = tAcc + lane_off + c * (D / 4) + 16 * cc;
                uint32_t r[16];
                tmem_ld16(ta, r);
                tmem_ld_wait16(r);
    #pragma unroll
                for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
                tmem_st16(ta, r);
              }
            }
          }
          tmem_st_wait();
          // Step it - kSBuf used these vote slots; its accumulating MMAs were issued
          // (the votes read) before S(it) could land in this buffer.
          if (lane == 0) flags[16 * bb + 4 * c + wq] = lo_any ? 1 : 0;
          tc_fence_before();
          warp_arrive(bar(C::bPFull + bb));
        }
        if (!ok) break;
        float scale_out = kDq ? p.scale : 1.f;  // forward: 1 / (row sum), below
        float lse_row = -INFINITY;
        if constexpr (!kDq) {
          // The row sum over the four warpgroups' columns.
          float* xl = xchg + 8 * kRowsQ;
          xl[c * kRowsQ + il] = lsum;
          warp_arrive(bar(C::bStats));
          if (!warp_wait<false>(bar(C::bStats), kl & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          float ltot = 0.f;
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) ltot += xl[gg * kRowsQ + il];
          scale_out = ltot > 0.f ? 1.f / ltot : 0.f;
          lse_row = ltot > 0.f ? (mref + lg2_approx(ltot)) * 0.6931471805599453f : -INFINITY;
        }
        // Epilogue: O (forward) or scale * dQ; warpgroup c writes columns
        // [c*d/4, (c+1)*d/4). The accumulator is loaded and released (AccFree)
        // before the stores, so the next unit's first MMA can start meanwhile.
        constexpr int kChunks = D / 64;  // 16-column TMEM loads per thread
        uint32_t r[kChunks][16];
        if (nsteps > 0) {
          if (!warp_wait<kRowMathPoll>(bar(C::bAcc), kl & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t col0 = tAcc + lane_off + c * (D / 4);
          tmem_ld16(col0, r[0]);
          if constexpr (kChunks == 2) {
            tmem_ld16(col0 + 16, r[1]);
            tmem_ld_wait16x2(r[0], r[1]);
          } else {
            tmem_ld_wait16(r[0]);
          }
          tc_fence_before();
          warp_arrive(bar(C::bAccFree));
          ++kl;
        } else {
#pragma unroll
          for (int cc = 0; cc < kChunks; ++cc)
#pragma unroll
            for (int x = 0; x < 16; ++x) r[cc][x] = 0u;
        }
        if (i < Nl) {
          const long long off = (long long)b * p.sb + (long long)(u.row0 + i) * p.sn + (long long)h * p.sh;
          uint16_t* dst = static_cast<uint16_t*>(p.out) + off + c * (D / 4);
#pragma unroll
          for (int cc = 0; cc < kChunks; ++cc) {
            uint32_t w[8];
#pragma unroll
            for (int x = 0; x < 8; ++x)
              w[x] = pack2<kBf16>(__uint_as_float(r[cc][2 * x]) * scale_out, __uint_as_float(r[cc][2 * x + 1]) * scale_out);
            uint4* gp = reinterpret_cast<uint4*>(dst + 16 * cc);
            gp[0] = make_uint4(w[0], w[1], w[2], w[3]);
            gp[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
          if (!kDq && c == 0) p.lse_out[u.lse + i] = lse_row;
        }
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
  // Persistent dQ kernel: the last CTA to leave resets its counter pair (next
  // ticket, CTAs done), so a later launch on the same workspace starts afresh
  // even without the preprocess in between. Each CTA's final ticket was taken
  // by this thread (the producer) before its fence.
  if (ctr != nullptr && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
      ctr[0] = 0u;
      ctr[1] = 0u;
    }
  }
}

template <int D, bool kBf16, int kMode, bool kDrop, bool kAlibi, bool kBias>
static cudaError_t launch_q_t(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  using C = QCfg<D, kMode, kBias>;
  auto kern = qmajor_kernel<D, kBf16, kMode, kDrop, kAlibi, kBias>;
  const int smem = (int)(C::kSmem > kMinSmemOneCtaPerSm ? C::kSmem : kMinSmemOneCtaPerSm);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rows = p.cu_seqlens ? p.max_seqlen : p.N;
  const long long total = (long long)((rows + kRowsQ - 1) / kRowsQ) * (p.cu_seqlens ? p.nseq * p.H : p.B * p.H);
  long long grid = total;  // the forward: one CTA per unit
  if (kMode == kModeDq && p.unit_ctr != nullptr) {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    grid = total < sms ? total : sms;
  }
  kern<<<(unsigned)grid, kQThreads, smem, st>>>(p, maps[0], maps[1], maps[2], maps[3], maps[4]);
  return cudaGetLastError();
}

template <int D, bool kBf16, int kMode, bool kBias>
static cudaError_t launch_q_b(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  const bool drop = p.drop.on != 0;
  if (p.alibi)
    return drop ? launch_q_t<D, kBf16, kMode, true, true, kBias>(p, maps, st)
                : launch_q_t<D, kBf16, kMode, false, true, kBias>(p, maps, st);
  return drop ? launch_q_t<D, kBf16, kMode, true, false, kBias>(p, maps, st)
              : launch_q_t<D, kBf16, kMode, false, false, kBias>(p, maps, st);
}

template <int D, bool kBf16, int kMode>
static cudaError_t launch_q_m(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  return p.bias ? launch_q_b<D, kBf16, kMode, true>(p, maps, st) : launch_q_b<D, kBf16, kMode, false>(p, maps, st);
}

template <int D, bool kBf16>
static cudaError_t launch_q_d(const AttnParams& p, bool dq_mode, const CUtensorMap* maps, cudaStream_t st) {
  return dq_mode ? launch_q_m<D, kBf16, kModeDq>(p, maps, st) : launch_q_m<D, kBf16, kModeFwd>(p, maps, st);
}

// maps: Q, K, V, dO (Q/dO boxes of kRowsQ rows, K/V boxes of kStepKV rows), and
// the attention bias (boxes of 128 rows x 64 keys, 128-byte swizzle; any valid
// map when p.bias is null).
cudaError_t launch_qmajor_tc(const AttnParams& p, bool bf16, bool dq_mode, const CUtensorMap* maps,
                             cudaStream_t st) {
  if (p.d == 128)
    return bf16 ? launch_q_d<128, true>(p, dq_mode, maps, st) : launch_q_d<128, false>(p, dq_mode, maps, st);
  return bf16 ? launch_q_d<64, true>(p, dq_mode, maps, st) : launch_q_d<64, false>(p, dq_mode, maps, st);
}

}  // namespace fa
