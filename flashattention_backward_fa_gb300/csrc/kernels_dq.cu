// Query-major dQ kernel with Q and dO resident in TMEM (sm_103a tcgen05).
//
// "FlashAttention backward", §The loop structure, choice (b): outer loop over
// query blocks, inner loop over key blocks, recomputing S and dP so that dQ
// accumulates on chip without atomics (the reduction order over key blocks is
// fixed, so dQ is bit-reproducible):
//   S = Q_i K_j^T, dP~ = dO_i V_j^T, P = exp2(S*scale*log2e - L_i*log2e),
//   dP = dP~ o Z/(1-p), dS = P o (dP - D_i), dQ_i += dS K_j; dQ = scale * dQ.
//
// Layout. One CTA owns 128 queries (the TMEM lanes). Q and dO are loaded once
// and copied into TMEM, where they are the A operands of S = Q K^T and
// dP = dO V^T (TS MMAs): shared memory then carries only the B operands (K, V)
// and their TMA writes, about 80 KB per 64-key step, against the 128 B/clk a
// shared-memory port delivers; the MMAs (768 cycles of tensor work a step) are
// the bound. A step covers 64 keys; S and dP have two TMEM buffers each, so the
// MMAs of one step run under the row math of the other.
//
// TMEM columns (d = 128): Q [0, 64), dO [64, 128) (two 16-bit values a
// column), S buffers [128, 192) [192, 256), dP buffers [256, 320) [320, 384),
// dQ accumulator [384, 512). (d = 64: the same with Q and dO 32 columns each
// and a 64-column accumulator.)
//
// Warp roles: warp 0 issues TMA loads (Q, dO once; K and V per step into a ring
// of stages); warp 1 owns TMEM and issues the S MMAs, warp 3 the dP MMAs,
// warp 2 the dQ MMAs (A = the dS image in TMEM, over the S columns it
// replaces). Four row-math warpgroups (warps 4-19): warpgroups 0, 1 take the
// even steps (buffer 0), 2, 3 the odd ones, each 32 of the step's 64 key
// columns; each thread owns one query row. They also copy Q and dO into TMEM
// at the start and write the dQ epilogue, a quarter of the columns each.
#include "fa_internal.h"

namespace fa {

constexpr int kDqThreads = 640;
constexpr int kDqStepKV = 64;  // keys per step

__device__ __forceinline__ void ld_shared_v4_dq(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr));
}

template <int D>
struct DqCfg {
  static constexpr int kPanels = D / 64;
  static constexpr uint32_t kQPanel = kRowsQ * 128;             // 16 KB: 128 rows x 64 elements
  static constexpr uint32_t kQTile = kPanels * kQPanel;         // Q or dO of the CTA's 128 rows
  static constexpr uint32_t kKVPanel = kDqStepKV * 128;         // 8 KB: 64 keys x 64 elements
  static constexpr uint32_t kKVTile = kPanels * kKVPanel;       // K or V of a step
  static constexpr uint32_t kStage = 2 * kKVTile;               // K then V
  static constexpr uint32_t kFixed = 2 * kQTile + 1024 + 1024;
  static constexpr int kNSraw = (int)((227u * 1024u - kFixed) / kStage);
  static constexpr int kNS = kNSraw > 6 ? 6 : kNSraw;           // ring stages
  static constexpr uint32_t oQ = 0;
  static constexpr uint32_t oDO = oQ + kQTile;
  static constexpr uint32_t oRing = oDO + kQTile;
  static constexpr uint32_t oBar = oRing + kNS * kStage;
  static constexpr int bRes = 0;                                // Q, dO landed
  static constexpr int bQReady = 1;                             // Q, dO copied into TMEM
  static constexpr int bFull = 2;                               // [kNS] K, V of a step landed
  static constexpr int bEmpty = bFull + kNS;                    // [kNS] stage released (after dQ)
  static constexpr int bSFull = bEmpty + kNS;                   // [2] S and dP of a step landed (two commits)
  static constexpr int bSEmpty = bSFull + 2;                    // [2] dQ MMAs done with the image
  static constexpr int bDPEmpty = bSEmpty + 2;                  // [2] row math has read dP
  static constexpr int bPFull = bDPEmpty + 2;                   // [2] dS image written
  static constexpr int bAcc = bPFull + 2;
  static constexpr int bDrain = bAcc + 1;                       // [3] one per MMA-issuing warp
  static constexpr int kBars = bDrain + 3;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = (oAbort + 8 + 15) & ~15u;  // [buffer][8 warps] split votes
  static constexpr uint32_t kSmem = oFlags + 2 * 16 * 4 + 1024;  // + slack for 1024-byte alignment
  static_assert(kNS >= 3, "shared memory budget leaves fewer than three K/V stages");
  static_assert(kSmem <= 227u * 1024u, "shared memory budget exceeded");
  // TMEM columns
  static constexpr uint32_t cQ = 0, cDO = D / 2, cS = D, cDP = D + 128, cAcc = D + 256;
  static_assert(cAcc + D <= 512, "TMEM columns");
};

template <int D, bool kBf16, bool kDrop, bool kAlibi>
__global__ void __launch_bounds__(kDqThreads, 1)
    dq_tmem_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmDO) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oAbort);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + C::oFlags);
  auto bar = [&](int idx) -> uint32_t { return sb + C::oBar + 8u * idx; };

  // Work unit: (batch*head or sequence*head, query block), heaviest query
  // blocks first under a causal mask; a block past the end of its sequence
  // leaves before any setup.
  Unit u;
  if (!unit_decode(p, blockIdx.x, kRowsQ, true, u)) return;
  const int bh = u.bh, b = u.b, h = u.h;
  const int Nl = u.n;
  const int i0 = u.tile * kRowsQ;
  const int j_last = p.causal ? min(Nl - 1, i0 + kRowsQ - 1) : Nl - 1;
  const int j_first = p.window > 0 ? (max(0, i0 - p.window + 1) / kDqStepKV) * kDqStepKV : 0;
  const int nsteps = (j_last >= j_first) ? (j_last - j_first) / kDqStepKV + 1 : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bRes), 1);
    mbar_init(bar(C::bQReady), 512);
    for (int s = 0; s < C::kNS; ++s) {
      mbar_init(bar(C::bFull + s), 1);
      mbar_init(bar(C::bEmpty + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::bSFull + x), 2);
      mbar_init(bar(C::bSEmpty + x), 1);
      mbar_init(bar(C::bDPEmpty + x), 256);
      mbar_init(bar(C::bPFull + x), 256);
    }
    mbar_init(bar(C::bAcc), 1);
    for (int x = 0; x < 3; ++x) mbar_init(bar(C::bDrain + x), 1);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::oTmemSlot);
  const uint32_t tQ = tmem + C::cQ, tDO = tmem + C::cDO, tS = tmem + C::cS, tdP = tmem + C::cDP,
                 tAcc = tmem + C::cAcc;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::bRes), 2 * C::kQTile);
      for (int pn = 0; pn < C::kPanels; ++pn) {
        tma_load_4d(sb + C::oQ + pn * C::kQPanel, &tmQ, bar(C::bRes), 64 * pn, u.row0 + i0, h, b);
        tma_load_4d(sb + C::oDO + pn * C::kQPanel, &tmDO, bar(C::bRes), 64 * pn, u.row0 + i0, h, b);
      }
      int issued = 0;
      for (int it = 0; it < nsteps; ++it) {
        const int s = it % C::kNS;
        if (!mbar_wait(bar(C::bEmpty + s), ((it / C::kNS) & 1) ^ 1, abort_flag, p.status)) break;
        const int jj = j_first + it * kDqStepKV;
        const uint32_t st = sb + C::oRing + s * C::kStage;
        mbar_arrive_expect_tx(bar(C::bFull + s), C::kStage);
        for (int pn = 0; pn < C::kPanels; ++pn) {
          tma_load_4d(st + pn * C::kKVPanel, &tmK, bar(C::bFull + s), 64 * pn, u.row0 + jj, h, b);
          tma_load_4d(st + C::kKVTile + pn * C::kKVPanel, &tmV, bar(C::bFull + s), 64 * pn, u.row0 + jj, h, b);
        }
        issued = it + 1;
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        mbar_wait_drain(bar(C::bRes), 0, p.status);
        for (int it = max(0, issued - C::kNS); it < issued; ++it)
          mbar_wait_drain(bar(C::bFull + it % C::kNS), (it / C::kNS) & 1, p.status);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // --------------------- S (warp 1) / dP (warp 3) MMA issuer -----------------
    // S = Q K^T or dP~ = dO V^T: M = 128 queries, N = 64 keys, K = d; A from
    // TMEM, B the K-major K or V tile of the step.
    {
      const bool isS = warp == 1;
      constexpr uint32_t idS = make_idesc(128, kDqStepKV, kBf16, false, false);
      const uint32_t tA = isS ? tQ : tDO;
      const uint32_t tD = isS ? tS : tdP;
      const int bE = isS ? C::bSEmpty : C::bDPEmpty;
      const uint64_t b0 = make_sdesc(sb + C::oRing + (isS ? 0u : C::kKVTile), 16, 1024);
      bool ok = warp_wait<kIssuerPoll>(bar(C::bQReady), 0, abort_flag, p.status);
      for (int it = 0; ok && it < nsteps; ++it) {
        const int s = it % C::kNS, bb = it & 1;
        if (!warp_wait<kIssuerPoll>(bar(C::bFull + s), (it / C::kNS) & 1, abort_flag, p.status) ||
            !warp_wait<kIssuerPoll>(bar(bE + bb), ((it >> 1) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t bd = desc_add(b0, s * C::kStage);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc_mma_ts_w(tD + 64 * bb, tA + 8 * k, desc_add(bd, (k >> 2) * C::kKVPanel + (k & 3) * 32), idS,
                      k > 0 ? 1u : 0u);
        tc_commit_w(bar(C::bSFull + bb));  // S and dP both arrive here
      }
      // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
      const int dr = isS ? 0 : 2;
      tc_commit_w(bar(C::bDrain + dr));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain + dr), 0, p.status);
      __syncwarp();
    }
  } else if (warp == 2) {
    // ---------------------------- dQ MMA issuer -------------------------------
    // dQ += dS K: M = 128 queries, N = d, K = the step's 64 keys; A = the dS
    // image over the S columns (per 16-key K step: 8 rounded columns, then 8
    // residual columns, added only when a warp voted for them), B = the K tile
    // read MN-major. Then release the S buffer and the ring stage.
    {
      constexpr uint32_t idQ = make_idesc(128, D, kBf16, false, true);
      const uint64_t b0 = make_sdesc(sb + C::oRing, C::kKVPanel, 1024);
      bool ok = true;
      for (int t = 0; ok && t < nsteps; ++t) {
        const int bt = t & 1, s = t % C::kNS;
        if (!warp_wait<kConsumerPoll>(bar(C::bPFull + bt), (t >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int4* f4 = reinterpret_cast<const int4*>(const_cast<const int*>(flags) + 16 * bt);
        const int4 v0 = f4[0], v1 = f4[1];
        const int any = v0.x | v0.y | v0.z | v0.w | v1.x | v1.y | v1.z | v1.w;
        const uint32_t first = t > 0 ? 1u : 0u;
        const uint64_t bd = desc_add(b0, s * C::kStage);
#pragma unroll
        for (int k = 0; k < kDqStepKV / 16; ++k)
          tc_mma_ts_w(tAcc, tS + 64 * bt + 16 * k, desc_add(bd, 2048 * k), idQ, k > 0 ? 1u : first);
        if (any) {
#pragma unroll
          for (int k = 0; k < kDqStepKV / 16; ++k)
            tc_mma_ts_w(tAcc, tS + 64 * bt + 16 * k + 8, desc_add(bd, 2048 * k), idQ, 1u);
        }
        tc_commit_w(bar(C::bSEmpty + bt));
        tc_commit_w(bar(C::bEmpty + s));
      }
      tc_commit_w(bar(C::bAcc));
      tc_commit_w(bar(C::bDrain + 1));
      if (lane == 0) mbar_wait_drain(bar(C::bDrain + 1), 0, p.status);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ---------------- row-math warpgroups + Q/dO copy + epilogue ----------------
    const int rg = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int c = rg & 1;        // key columns [32c, 32c + 32) of a step
    const int bb = rg >> 1;      // steps it with it % 2 == bb (TMEM buffer bb)
    const int il = wq * 32 + lane;
    const int i = i0 + il;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    bool ok = warp_wait<kRowMathPoll>(bar(C::bRes), 0, abort_flag, p.status);
    if (ok) {
      // Copy this warpgroup's share into TMEM: warpgroups 0, 1 take the two
      // halves of Q's head dimension, 2, 3 those of dO. Row il of the
      // 128-byte-swizzled tile: element e of panel pn sits in 16-byte chunk
      // (e / 8) ^ (il & 7) of the row.
      const int half = rg & 1;
      const uint32_t src = sb + ((rg >> 1) ? C::oDO : C::oQ) + (uint32_t)il * 128;
      const uint32_t dstc = ((rg >> 1) ? tDO : tQ) + lane_off + (uint32_t)(half * (D / 4));
#pragma unroll
      for (int g = 0; g < D / 64; ++g) {  // 32 elements (16 columns) at a time
        const int e0 = half * (D / 2) + 32 * g;  // first element of the group
        const uint32_t pan = src + (uint32_t)(e0 / 64) * C::kQPanel;
        uint32_t w[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t chunk = (uint32_t)(((e0 % 64) / 8 + t) ^ (il & 7));
          ld_shared_v4_dq(pan + (chunk << 4), w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
        tmem_st16(dstc + 16 * g, w);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    warp_arrive(bar(C::bQReady));
    // -L*log2(e) (-inf for a row with no allowed key) and -D of this row; the
    // negated forms are addends of one FMA / add.
    const long long ws = u.ws + i;  // i < the padded row count always
    const float nL2 = p.ws_nL2[ws];
    const float nD = p.ws_nD[ws];
    const float slope_raw = kAlibi ? alibi_slope_raw(p, u) : 0.f;
    for (int it = bb; ok && it < nsteps; it += 2) {
      const int base = j_first + it * kDqStepKV + 32 * c;
      const uint32_t tSc = tS + lane_off + 64 * bb + 32 * c, tdPc = tdP + lane_off + 64 * bb + 32 * c;
      if (!warp_wait<kRowMathPoll>(bar(C::bSFull + bb), (it >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t allow =
          bit_range(p.window > 0 ? i - p.window + 1 - base : 0, min(Nl - base, p.causal ? i + 1 - base : 32));
      uint32_t keep = 0xFFFFFFFFu;
      if constexpr (kDrop) keep = keep_bits_for_query(p.drop, bh, Nl, i, base);
      // this warpgroup's S and dP columns in one go (no wait between a TMEM load
      // and its completion wait), then the dP buffer is released
      uint32_t sr2[2][16], dr2[2][16];
      __syncwarp();
      tmem_ld16(tSc, sr2[0]);
      tmem_ld16(tSc + 16, sr2[1]);
      tmem_ld16(tdPc, dr2[0]);
      tmem_ld16(tdPc + 16, dr2[1]);
      tmem_ld_wait16x4(sr2[0], sr2[1], dr2[0], dr2[1]);
      tc_fence_before();
      warp_arrive(bar(C::bDPEmpty + bb));
      // ALiBi: a chunk whose allowed keys all lie on one side of the diagonal
      // (always under a causal mask) takes the bias as a ramp over the columns
      // plus a row constant folded into the exp2 addend; a chunk straddling the
      // diagonal folds |i - j| per score.
      float rc2 = 0.f;
      if constexpr (kAlibi) {
        const int dd = i - base;  // i - j of column 0
        if (p.causal || dd >= 31) {
          rc2 = -slope_raw * (float)dd * p.scale_log2;
          alibi_ramp16<0>(sr2[0], slope_raw);
          alibi_ramp16<16>(sr2[1], slope_raw);
        } else if (dd <= 0) {
          rc2 = slope_raw * (float)dd * p.scale_log2;
          alibi_ramp16<0>(sr2[0], -slope_raw);
          alibi_ramp16<16>(sr2[1], -slope_raw);
        } else {
          alibi_fold16<-1>(sr2[0], (float)dd, slope_raw);
          alibi_fold16<-1>(sr2[1], (float)(dd - 16), slope_raw);
        }
      }
      const float nL2c = kAlibi ? nL2 + rc2 : nL2;
      bool lo_any = false;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t (&sr)[16] = sr2[hh];
        const uint32_t (&dr)[16] = dr2[hh];
        float outv[16];
        float cmax = 0.f;
        auto elementwise = [&](auto masked) {
          if constexpr (!kDrop) {
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
              const uint64_t dd2 = f2_add(f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), f2_pack(nD, nD));
              f2_unpack(f2_mul(f2_pack(p0, p1), dd2), outv[e], outv[e + 1]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int bit = 16 * hh + e;
              float pv = ex2_approx(fmaf(__uint_as_float(sr[e]), p.scale_log2, nL2c));
              if constexpr (decltype(masked)::value) pv = ((allow >> bit) & 1u) ? pv : 0.f;
              cmax = fmaxf(cmax, pv);
              const float dpv = ((keep >> bit) & 1u) ? __uint_as_float(dr[e]) * p.drop.rp : 0.f;
              outv[e] = pv * (dpv + nD);
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
        uint32_t hv[8], ev[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) hv[x] = pack2<kBf16>(outv[2 * x], outv[2 * x + 1]);
        // Residuals where a probability exceeds the split threshold (zeros
        // elsewhere keep the residual image well defined).
        const bool split_h = __any_sync(0xFFFFFFFFu, cmax > kSplitThreshold);
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
      tmem_st_wait();
      // Step it - 2 used these vote slots; its dQ MMAs were issued (the votes
      // read) before S(it) could land in this buffer.
      if (lane == 0) flags[16 * bb + 4 * c + wq] = lo_any ? 1 : 0;
      tc_fence_before();
      warp_arrive(bar(C::bPFull + bb));
    }
    // Epilogue: scale * dQ; warpgroup rg writes columns [rg*d/4, (rg+1)*d/4).
    const bool have_acc = nsteps > 0;
    if (ok && have_acc) ok = warp_wait<kRowMathPoll>(bar(C::bAcc), 0, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      const long long off = (long long)b * p.sb + (long long)(u.row0 + i) * p.sn + (long long)h * p.sh;
      uint16_t* dst = static_cast<uint16_t*>(p.out) + off;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = rg * (D / 4) + 16 * cc;
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
          w[x] = pack2<kBf16>(__uint_as_float(r[2 * x]) * p.scale, __uint_as_float(r[2 * x + 1]) * p.scale);
        if (i < Nl) {
          uint4* g = reinterpret_cast<uint4*>(dst + col);
          g[0] = make_uint4(w[0], w[1], w[2], w[3]);
          g[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
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

template <int D, bool kBf16, bool kDrop, bool kAlibi>
static cudaError_t launch_dq_tmem_t(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  using C = DqCfg<D>;
  auto kern = dq_tmem_kernel<D, kBf16, kDrop, kAlibi>;
  const int smem = (int)(C::kSmem > kMinSmemOneCtaPerSm ? C::kSmem : kMinSmemOneCtaPerSm);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rows = p.cu_seqlens ? p.max_seqlen : p.N;
  const int tiles = (rows + kRowsQ - 1) / kRowsQ;
  const unsigned grid = (unsigned)(tiles * (p.cu_seqlens ? p.nseq * p.H : p.B * p.H));
  kern<<<grid, kDqThreads, smem, st>>>(p, maps[0], maps[1], maps[2], maps[3]);
  return cudaGetLastError();
}

template <int D, bool kBf16>
static cudaError_t launch_dq_tmem_d(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  const bool drop = p.drop.on != 0;
  if (p.alibi)
    return drop ? launch_dq_tmem_t<D, kBf16, true, true>(p, maps, st)
                : launch_dq_tmem_t<D, kBf16, false, true>(p, maps, st);
  return drop ? launch_dq_tmem_t<D, kBf16, true, false>(p, maps, st)
              : launch_dq_tmem_t<D, kBf16, false, false>(p, maps, st);
}

// Whether this kernel serves the deterministic dQ step: 16-bit inputs with
// d in {64, 128} and no attention bias tensor (the bias path stays on the
// query-major kernel of kernels_qmajor.cu).
bool dq_tmem_supported(const AttnParams& p) { return (p.d == 64 || p.d == 128) && p.bias == nullptr; }

// maps: Q, dO (boxes of kRowsQ rows), K, V (boxes of 64 rows), all 64-element
// 128-byte-swizzled panels of the head dimension.
cudaError_t launch_dq_tmem(const AttnParams& p, bool bf16, const CUtensorMap* maps, cudaStream_t st) {
  if (p.d == 128) return bf16 ? launch_dq_tmem_d<128, true>(p, maps, st) : launch_dq_tmem_d<128, false>(p, maps, st);
  return bf16 ? launch_dq_tmem_d<64, true>(p, maps, st) : launch_dq_tmem_d<64, false>(p, maps, st);
}

}  // namespace fa
