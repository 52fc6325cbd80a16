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
// TMEM columns: dQ kernel [0,256) two S buffers, [256,384) the dP buffer;
// forward [0,384) three S buffers; then [384,384+d) the dQ or O accumulator.
#include "fa_internal.h"

namespace fa {

constexpr int kModeFwd = 0;
constexpr int kModeDq = 1;
constexpr int kQThreads = 640;  // 4 role warps + 4 row-math warpgroups

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
  static constexpr int kBars = bBEmpty + 1;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = (oAbort + 8 + 15) & ~15u;  // [buffer][16 warps] split votes
  static constexpr uint32_t kSmem = oFlags + kSBuf * 16 * 4 + 1024;  // + slack for 1024-byte alignment
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
  auto bar = [&](int idx) -> uint32_t { return sb + C::oBar + 8u * idx; };

  // Work unit: (batch*head or sequence*head, query block), heaviest query
  // blocks first under a causal mask. A query block past the end of its
  // sequence has no work: the whole CTA leaves before any setup.
  Unit u;
  if (!unit_decode(p, blockIdx.x, kRowsQ, true, u)) return;
  const int bh = u.bh, b = u.b, h = u.h;
  const int Nl = u.n;                    // rows of this (batch, head) or sequence
  const int i0 = u.tile * kRowsQ;
  const int j_last = p.causal ? min(Nl - 1, i0 + kRowsQ - 1) : Nl - 1;
  const int j_first = p.window > 0 ? (max(0, i0 - p.window + 1) / kStepKV) * kStepKV : 0;
  const int nkv = (j_last >= j_first) ? (j_last - j_first) / kStepKV + 1 : 0;
  // One pass over the key blocks in both modes.
  const int nsteps = nkv;
  // Key block of step it. Ascending, except in the ALiBi forward: there the
  // blocks go outward from the one holding this tile's diagonal (nearest first,
  // alternating below and above), so that every row meets its largest biased
  // scores early and the online softmax's reference rarely has to move.
  auto key_block = [&](int it) -> int {
    if constexpr (kAlibi && !kDq) {
      const int g = min(max((i0 - j_first) / kStepKV, 0), nkv - 1);
      const int below = g, above = nkv - 1 - g, m = min(below, above);
      int t;
      if (it == 0) t = g;
      else if (it <= 2 * m) t = (it & 1) ? g - (it + 1) / 2 : g + it / 2;
      else t = below > above ? g - (it - m) : g + (it - m);
      return j_first + t * kStepKV;
    } else {
      return j_first + it * kStepKV;
    }
  };

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

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    // Step it: ring E gets V (dQ) or K (forward); ring L gets K (dQ) or, on
    // forward output steps, V. L tiles are counted from the first output step.
    if (lane == 0) {
      const CUtensorMap* mE = kDq ? &tmV : &tmK;
      const CUtensorMap* mL = kDq ? &tmK : &tmV;
      mbar_arrive_expect_tx(bar(C::bRes), C::kResident);
      for (int pn = 0; pn < C::kPanels; ++pn) {
        tma_load_4d(sb + C::oQ + pn * C::kPanel, &tmQ, bar(C::bRes), 64 * pn, u.row0 + i0, h, b);
        if (kDq) tma_load_4d(sb + C::oDO + pn * C::kPanel, &tmDO, bar(C::bRes), 64 * pn, u.row0 + i0, h, b);
      }
      int issuedE = 0, issuedL = 0, issuedB = 0;
      bool ok = true;
      for (int it = 0; ok && it < nsteps; ++it) {
        const int jj = key_block(it);
        const int se = it % C::kNE;
        if (!mbar_wait(bar(C::bEEmpty + se), ((it / C::kNE) & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(bar(C::bEFull + se), C::kTile);
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_4d(sb + C::oE + se * C::kTile + pn * C::kPanel, mE, bar(C::bEFull + se), 64 * pn, u.row0 + jj,
                      h, b);
        issuedE = it + 1;
        const int sl = it % C::kNL;
        if (!mbar_wait(bar(C::bLEmpty + sl), ((it / C::kNL) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(C::bLFull + sl), C::kTile);
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_4d(sb + C::oL + sl * C::kTile + pn * C::kPanel, mL, bar(C::bLFull + sl), 64 * pn, u.row0 + jj,
                      h, b);
        issuedL = it + 1;
        if constexpr (kBias) {
          // the step's bias tile, once the row math has copied the previous one
          if (!mbar_wait(bar(C::bBEmpty), (it & 1) ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::bBFull), C::kBiasTile);
          for (int pn = 0; pn < 2; ++pn)
            tma_load_4d(sb + C::oBias + pn * C::kBiasPanel, &tmBias, bar(C::bBFull), jj + 64 * pn, u.row0 + i0,
                        p.bias_sh ? h : 0, p.bias_sb ? b : 0);
          issuedB = it + 1;
        }
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        mbar_wait_drain(bar(C::bRes), 0, p.status);
        for (int it = max(0, issuedE - C::kNE); it < issuedE; ++it)
          mbar_wait_drain(bar(C::bEFull + it % C::kNE), (it / C::kNE) & 1, p.status);
        for (int li = max(0, issuedL - C::kNL); li < issuedL; ++li)
          mbar_wait_drain(bar(C::bLFull + li % C::kNL), (li / C::kNL) & 1, p.status);
        if (issuedB > 0) mbar_wait_drain(bar(C::bBFull), (issuedB - 1) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ S MMA issuer ------------------------------
    {
      constexpr uint32_t idS = make_idesc(128, kStepKV, kBf16, false, false);
      const uint64_t dQ0 = make_sdesc(sb + C::oQ, 16, 1024);
      const uint64_t dK0 = make_sdesc(sb + (kDq ? C::oL : C::oE), 16, 1024);
      bool ok = warp_wait<kIssuerPoll>(bar(C::bRes), 0, abort_flag, p.status);
      for (int it = 0; ok && it < nsteps; ++it) {
        const int bb = it % C::kSBuf;
        // K lives in ring L (dQ; one tile per step) or ring E (forward)
        const int ks = kDq ? it % C::kNL : it % C::kNE;
        const uint32_t kpar = kDq ? (it / C::kNL) & 1 : (it / C::kNE) & 1;
        if (!warp_wait<kIssuerPoll>(bar((kDq ? C::bLFull : C::bEFull) + ks), kpar, abort_flag, p.status) ||
            !warp_wait<kIssuerPoll>(bar(C::bSEmpty + bb), ((it / C::kSBuf) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kd = desc_add(dK0, ks * C::kTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc_mma_ss_w(tS + 128 * bb, desc_add(dQ0, (k >> 2) * C::kPanel + (k & 3) * 32),
                      desc_add(kd, (k >> 2) * C::kPanel + (k & 3) * 32), idS, k > 0 ? 1u : 0u);
        tc_commit_w(bar(C::bSFull + bb));
        if (!kDq) tc_commit_w(bar(C::bEEmpty + ks));   // forward: K is done once S is
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
      bool ok = warp_wait<kIssuerPoll>(bar(C::bRes), 0, abort_flag, p.status);
      for (int it = 0; ok && it < nsteps; ++it) {
        const int se = it % C::kNE;
        if (!warp_wait<kIssuerPoll>(bar(C::bEFull + se), (it / C::kNE) & 1, abort_flag, p.status) ||
            (it > 0 && !warp_wait<kIssuerPoll>(bar(C::bDPEmpty), (it - 1) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t vd = desc_add(dV0, se * C::kTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc_mma_ss_w(tdP, desc_add(dO0, (k >> 2) * C::kPanel + (k & 3) * 32),
                      desc_add(vd, (k >> 2) * C::kPanel + (k & 3) * 32), idS, k > 0 ? 1u : 0u);
        tc_commit_w(bar(C::bSFull + it % C::kSBuf));
        tc_commit_w(bar(C::bEEmpty + se));
      }
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      tc_commit_w(bar(C::bDrain + 2));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain + 2), 0, p.status);
      __syncwarp();
    }
  } else if (warp == 2) {
    // ------------------ accumulating MMA issuer (O or dQ) ---------------------
    // After the row math of step t: acc += (P~ or dS) . (V_j or K_j), then
    // release the S buffer and the ring-L tile.
    {
      constexpr uint32_t idO = make_idesc(128, D, kBf16, false, true);
      const uint64_t b0 = make_sdesc(sb + C::oL, C::kPanel, 1024);
      bool ok = true;
      for (int t = 0; ok && t < nsteps; ++t) {
        const int bt = t % C::kSBuf;
        if (!warp_wait<kConsumerPoll>(bar(C::bPFull + bt), (t / C::kSBuf) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int sl = t % C::kNL;
        // Forward: V (ring L) must have landed before the MMA reads it. In the dQ
        // kernel ring L holds K, whose arrival the S issuer waited for before S.
        if (!kDq && !warp_wait<kIssuerPoll>(bar(C::bLFull + sl), (t / C::kNL) & 1, abort_flag, p.status)) {
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
        for (int k = 0; k < kStepKV / 16; ++k)
          tc_mma_ts_w(tAcc, tS + 128 * bt + 16 * k, desc_add(bop, 2048 * k), idO, k > 0 ? 1u : first);
        if (any) {
#pragma unroll
          for (int k = 0; k < kStepKV / 16; ++k)
            tc_mma_ts_w(tAcc, tS + 128 * bt + 16 * k + 8, desc_add(bop, 2048 * k), idO, 1u);
        }
        tc_commit_w(bar(C::bSEmpty + bt));
        tc_commit_w(bar(C::bLEmpty + sl));
        if (!kDq) tc_commit_w(bar(C::bODone));
      }
      tc_commit_w(bar(C::bAcc));
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
    const int i = i0 + il;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tdPc = tdP + lane_off + 32 * c;
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
    const float inv_scale = kBias ? 1.f / p.scale : 0.f;
    float mref = -INFINITY, lsum = 0.f;
    float* xchg = reinterpret_cast<float*>(smem + C::oStats);
    bool ok = true;
    for (int it = 0; it < nsteps; ++it) {
      const int bb = it % C::kSBuf, xb = it & 1;
      const int base = key_block(it) + 32 * c;
      const uint32_t tSc = tS + lane_off + 128 * bb + 32 * c;
      // This row's bias over the chunk's 32 keys (four 16-byte pieces of the
      // swizzled tile; zeros past N), copied to registers so that the buffer is
      // released, and the next step's tile loads, before this step's row math.
      uint32_t bw[16];
      if constexpr (kBias) {
        if (!warp_wait<kRowMathPoll>(bar(C::bBFull), it & 1, abort_flag, p.status)) {
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
      if (!warp_wait<kRowMathPoll>(bar(C::bSFull + bb), (it / C::kSBuf) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // allowed keys of this warpgroup's 32 columns (bit x <-> key base + x)
      const uint32_t allow =
          bit_range(p.window > 0 ? i - p.window + 1 - base : 0, min(Nl - base, p.causal ? i + 1 - base : 32));
      uint32_t keep = 0xFFFFFFFFu;
      if constexpr (kDrop) keep = keep_bits_for_query(p.drop, bh, Nl, i, base);
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
        if (!warp_wait<false>(bar(C::bXchg + 4 * xb + wq), (it >> 1) & 1, abort_flag, p.status)) {
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
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int bit = 16 * hh + e;
              float pv = ex2_approx(fmaf(__uint_as_float(sr[e]), p.scale_log2, nL2c));
              if constexpr (decltype(masked)::value) pv = ((allow >> bit) & 1u) ? pv : 0.f;
              cmax = fmaxf(cmax, pv);
              const bool kept = (keep >> bit) & 1u;
              if constexpr (kDq) {
                const float dpv = kept ? __uint_as_float(dr[e]) * p.drop.rp : 0.f;
                outv[e] = pv * (dpv + nD);
              } else {
                psum += pv;
                outv[e] = kept ? pv * p.drop.rp : 0.f;
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
          if (it > 0 && !warp_wait<kRowMathPoll>(bar(C::bODone), (it - 1) & 1, abort_flag, p.status)) {
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
    float scale_out = kDq ? p.scale : 1.f;  // forward: 1 / (row sum), below
    float lse_row = -INFINITY;
    if constexpr (!kDq) {
      if (ok) {
        // The row sum over the four warpgroups' columns.
        float* xl = xchg + 8 * kRowsQ;
        xl[c * kRowsQ + il] = lsum;
        warp_arrive(bar(C::bStats));
        ok = warp_wait<false>(bar(C::bStats), 0, abort_flag, p.status);
        float ltot = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) ltot += xl[g * kRowsQ + il];
        scale_out = ltot > 0.f ? 1.f / ltot : 0.f;
        lse_row = ltot > 0.f ? (mref + lg2_approx(ltot)) * 0.6931471805599453f : -INFINITY;
      }
    }
    // Epilogue: O (forward) or scale * dQ; warpgroup c writes columns [c*d/4, (c+1)*d/4).
    const bool have_acc = nsteps > 0;
    if (ok && have_acc) ok = warp_wait<kRowMathPoll>(bar(C::bAcc), 0, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      const long long off = (long long)b * p.sb + (long long)(u.row0 + i) * p.sn + (long long)h * p.sh;
      uint16_t* dst = static_cast<uint16_t*>(p.out) + off;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = c * (D / 4) + 16 * cc;
        uint32_t r[16];
        if (have_acc) {
          tmem_ld16(tAcc + lane_off + col, r);
          tmem_ld_wait16(r);
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) r[x] = 0u;
        }
        uint32_t w[8];
#pragma unroll
        for (int x = 0; x < 8; ++x)
          w[x] = pack2<kBf16>(__uint_as_float(r[2 * x]) * scale_out, __uint_as_float(r[2 * x + 1]) * scale_out);
        if (i < Nl) {
          uint4* g = reinterpret_cast<uint4*>(dst + col);
          g[0] = make_uint4(w[0], w[1], w[2], w[3]);
          g[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      if (!kDq && c == 0 && i < Nl) p.lse_out[u.lse + i] = lse_row;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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
  const int tiles = (rows + kRowsQ - 1) / kRowsQ;
  const unsigned grid = (unsigned)(tiles * (p.cu_seqlens ? p.nseq * p.H : p.B * p.H));
  kern<<<grid, kQThreads, smem, st>>>(p, maps[0], maps[1], maps[2], maps[3], maps[4]);
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
