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
// output O and the per-row log-sum-exp L = m + log(l) (natural log). It runs
// two passes over the key blocks: the first keeps the running row maximum and
// sum of exponentials, the second forms P = exp(S - L) with L already known —
// so O never needs rescaling — and accumulates O += (P o Z/(1-p)) V.
//
// Queries sit on the 128 TMEM lanes: one thread owns one query row, so L_i and
// D_i are per-thread scalars. The row math writes dS (or P~) back over the S
// columns it has read, rounded to 16 bits with the rounding residual beside
// it (see interleave_split), and the accumulating MMA reads it from TMEM. S
// rotates over three TMEM buffers, so the S MMA of step it + 3 waits only for
// the accumulating MMA of step it; dP rotates over two buffers that the row
// math releases as soon as it has read them.
// Warp 0 issues TMA loads, warp 1 owns TMEM and issues the S (and dP) MMAs,
// warp 2 issues the accumulating MMAs, two row-math warpgroups (warps 4-7,
// 8-11) take alternate key steps and split the epilogue columns.
//
// TMEM columns: [0,192) three S buffers, [192,320) two dP buffers (dQ mode),
// [320,320+d) the O or dQ accumulator.
#include "fa_internal.h"

namespace fa {

constexpr int kModeFwd = 0;
constexpr int kModeDq = 1;

template <int D, int kMode>
struct QCfg {
  static constexpr int kPanels = D / 64;
  static constexpr uint32_t kRowPanel = kRowsQ * 128;          // 16 KB
  static constexpr uint32_t kRowTile = kPanels * kRowPanel;
  static constexpr uint32_t kKVPanel = kStepKV * 128;          // 8 KB
  static constexpr uint32_t kKVTile = kPanels * kKVPanel;
  static constexpr uint32_t kResident = (kMode == kModeDq ? 2 : 1) * kRowTile;
  static constexpr uint32_t kStats = kMode == kModeFwd ? 2 * 2 * kRowsQ * 4 : 0;
  static constexpr uint32_t kBudget = 225u * 1024u;
  static constexpr int kNSraw = (int)((kBudget - kResident - kStats - 2048) / (2 * kKVTile));
  static constexpr int kNS = kNSraw > 6 ? 6 : kNSraw;          // K/V pipeline stages
  static constexpr uint32_t oQ = 0;
  static constexpr uint32_t oDO = oQ + kRowTile;
  static constexpr uint32_t oK = kResident;
  static constexpr uint32_t oV = oK + kNS * kKVTile;
  static constexpr uint32_t oStats = oV + kNS * kKVTile;       // forward: [wg][m | l][row]
  static constexpr uint32_t oBar = oStats + kStats;
  static constexpr int bRes = 0;
  static constexpr int bKVFull = 1;
  static constexpr int bKVEmpty = bKVFull + kNS;
  static constexpr int bSFull = bKVEmpty + kNS;
  static constexpr int bSEmpty = bSFull + 3;
  static constexpr int bDPEmpty = bSEmpty + 3;
  static constexpr int bPFull = bDPEmpty + 2;
  static constexpr int bAcc = bPFull + 2;
  static constexpr int bDrain = bAcc + 1;                      // one per MMA-issuing warp
  static constexpr int bStats = bDrain + 2;
  static constexpr int kBars = bStats + 1;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = oAbort + 8;               // [buffer][warp] split votes
  static constexpr uint32_t kSmem = oFlags + 32 + 1024;
  static_assert(kNS >= 2, "shared memory budget leaves fewer than two K/V stages");
  static_assert(kSmem <= 227u * 1024u, "shared memory budget exceeded");
};

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool kBf16, int kMode, bool kDrop>
__global__ void __launch_bounds__(384, 1)
    qmajor_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmDO) {
  using C = QCfg<D, kMode>;
  constexpr bool kDq = kMode == kModeDq;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oAbort);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + C::oFlags);
  auto bar = [&](int idx) -> uint32_t { return sb + C::oBar + 8u * idx; };

  // Work unit: (batch*head, query block), heaviest query blocks first under a causal mask.
  const int BH = p.B * p.H;
  const int ntiles = (p.N + kRowsQ - 1) / kRowsQ;
  const int q_tile = ntiles - 1 - (int)(blockIdx.x / BH);
  const int bh = blockIdx.x % BH;
  const int b = bh / p.H, h = bh % p.H;
  const int i0 = q_tile * kRowsQ;
  const int j_last = p.causal ? min(p.N - 1, i0 + kRowsQ - 1) : p.N - 1;
  const int j_first = p.window > 0 ? (max(0, i0 - p.window + 1) / kStepKV) * kStepKV : 0;
  const int nkv = (j_last >= j_first) ? (j_last - j_first) / kStepKV + 1 : 0;
  // Forward: nkv statistics steps, then nkv output steps. dQ: nkv steps.
  const int nsteps = kDq ? nkv : 2 * nkv;
  const int first_out = kDq ? 0 : nkv;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bRes), 1);
    for (int s = 0; s < C::kNS; ++s) {
      mbar_init(bar(C::bKVFull + s), 1);
      mbar_init(bar(C::bKVEmpty + s), 1);
    }
    for (int x = 0; x < 3; ++x) {
      mbar_init(bar(C::bSFull + x), 1);
      mbar_init(bar(C::bSEmpty + x), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::bDPEmpty + x), 128);
      mbar_init(bar(C::bPFull + x), 128);
    }
    mbar_init(bar(C::bAcc), 1);
    mbar_init(bar(C::bDrain), 1);
    mbar_init(bar(C::bDrain + 1), 1);
    mbar_init(bar(C::bStats), 256);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::oTmemSlot);
  const uint32_t tS = tmem, tdP = tmem + 192, tAcc = tmem + 320;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::bRes), C::kResident);
      for (int pn = 0; pn < C::kPanels; ++pn) {
        tma_load_4d(sb + C::oQ + pn * C::kRowPanel, &tmQ, bar(C::bRes), 64 * pn, i0, h, b);
        if (kDq) tma_load_4d(sb + C::oDO + pn * C::kRowPanel, &tmDO, bar(C::bRes), 64 * pn, i0, h, b);
      }
      int issued = 0;
      for (int it = 0; it < nsteps; ++it) {
        const int s = it % C::kNS;
        if (!mbar_wait(bar(C::bKVEmpty + s), ((it / C::kNS) & 1) ^ 1, abort_flag, p.status)) break;
        const int jt = it >= nkv ? it - nkv : it;
        const int jj = j_first + jt * kStepKV;
        const bool need_v = kDq || it >= first_out;
        mbar_arrive_expect_tx(bar(C::bKVFull + s), (need_v ? 2 : 1) * C::kKVTile);
        for (int pn = 0; pn < C::kPanels; ++pn) {
          tma_load_4d(sb + C::oK + s * C::kKVTile + pn * C::kKVPanel, &tmK, bar(C::bKVFull + s), 64 * pn, jj,
                      h, b);
          if (need_v)
            tma_load_4d(sb + C::oV + s * C::kKVTile + pn * C::kKVPanel, &tmV, bar(C::bKVFull + s), 64 * pn,
                        jj, h, b);
        }
        issued = it + 1;
      }
      if (*abort_flag) {
        mbar_wait_drain(bar(C::bRes), 0, p.status);
        for (int it = max(0, issued - C::kNS); it < issued; ++it)
          mbar_wait_drain(bar(C::bKVFull + it % C::kNS), (it / C::kNS) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------- S / dP MMA issuer ---------------------------
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc(128, kStepKV, kBf16, false, false);
      const uint64_t dQ0 = make_sdesc(sb + C::oQ, 16, 1024), dO0 = make_sdesc(sb + C::oDO, 16, 1024);
      const uint64_t dK0 = make_sdesc(sb + C::oK, 16, 1024), dV0 = make_sdesc(sb + C::oV, 16, 1024);
      bool ok = mbar_wait(bar(C::bRes), 0, abort_flag, p.status);
      for (int it = 0; ok && it < nsteps; ++it) {
        const int s = it % C::kNS, bb = it & 1, bs = it % 3;
        if (!mbar_wait(bar(C::bKVFull + s), (it / C::kNS) & 1, abort_flag, p.status) ||
            !mbar_wait(bar(C::bSEmpty + bs), ((it / 3) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kd = desc_add(dK0, s * C::kKVTile), vd = desc_add(dV0, s * C::kKVTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc_mma_ss(tS + 64 * bs, desc_add(dQ0, (k >> 2) * C::kRowPanel + (k & 3) * 32),
                    desc_add(kd, (k >> 2) * C::kKVPanel + (k & 3) * 32), idS, k > 0 ? 1u : 0u);
        if constexpr (kDq) {
          if (!mbar_wait(bar(C::bDPEmpty + bb), ((it >> 1) & 1) ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            tc_mma_ss(tdP + 64 * bb, desc_add(dO0, (k >> 2) * C::kRowPanel + (k & 3) * 32),
                      desc_add(vd, (k >> 2) * C::kKVPanel + (k & 3) * 32), idS, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::bSFull + bs));
      }
      if (!ok) {
        tc_commit(bar(C::bDrain));
        mbar_wait_drain(bar(C::bDrain), 0, p.status);
      }
    }
  } else if (warp == 2) {
    // ------------------ accumulating MMA issuer (O or dQ) ---------------------
    // After the row math of step t: acc += (P~ or dS) . (V_j or K_j) on output
    // steps, then release the S buffer and the K/V stage.
    if (lane == 0) {
      constexpr uint32_t idO = make_idesc(128, D, kBf16, false, true);
      const uint64_t b0 = make_sdesc(sb + (kDq ? C::oK : C::oV), C::kKVPanel, 1024);
      bool ok = true;
      for (int t = 0; ok && t < nsteps; ++t) {
        const int bt = t & 1, bs = t % 3, st = t % C::kNS;
        if (!mbar_wait(bar(C::bPFull + bt), (t >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (t >= first_out) {
          const uint32_t first = t > first_out ? 1u : 0u;
          const bool split = (flags[4 * bt] | flags[4 * bt + 1] | flags[4 * bt + 2] | flags[4 * bt + 3]) != 0;
          const uint64_t bop = desc_add(b0, st * C::kKVTile);
#pragma unroll
          for (int k = 0; k < kStepKV / 16; ++k)
            tc_mma_ts(tAcc, tS + 64 * bs + 16 * k, desc_add(bop, 2048 * k), idO, k > 0 ? 1u : first);
          if (split) {
#pragma unroll
            for (int k = 0; k < kStepKV / 16; ++k)
              tc_mma_ts(tAcc, tS + 64 * bs + 16 * k + 8, desc_add(bop, 2048 * k), idO, 1u);
          }
        }
        tc_commit(bar(C::bSEmpty + bs));
        tc_commit(bar(C::bKVEmpty + st));
      }
      tc_commit(bar(C::bAcc));
      if (!ok) {
        tc_commit(bar(C::bDrain + 1));
        mbar_wait_drain(bar(C::bDrain + 1), 0, p.status);
      }
    }
  } else if (warp >= 4) {
    // ------------- row-math warpgroups (alternate key steps) + epilogue -------
    const int wg = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int il = wq * 32 + lane;
    const int i = i0 + il;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tdPb = tdP + lane_off + 64 * wg;
    const long long ws = (long long)bh * p.n_pad + i;  // i < n_pad always
    float L2 = INFINITY, Dv = 0.f;
    if (kDq) {
      L2 = p.ws_L2[ws];
      Dv = p.ws_D[ws];
    }
    float m = -INFINITY, l = 0.f;  // forward statistics of this warpgroup's steps, log2 domain
    bool merged = kDq;
    bool ok = true;
    for (int it = wg; it < nsteps; it += 2) {
      const int jt = it >= nkv ? it - nkv : it;
      const int jj0 = j_first + jt * kStepKV;
      if (!kDq && it >= first_out && !merged) {
        // Combine the two warpgroups' partial row statistics into L.
        float* st = reinterpret_cast<float*>(smem + C::oStats);
        st[(2 * wg) * kRowsQ + il] = m;
        st[(2 * wg + 1) * kRowsQ + il] = l;
        mbar_arrive(bar(C::bStats));
        if (!mbar_wait(bar(C::bStats), 0, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const float mo = st[(2 * (1 - wg)) * kRowsQ + il], lo = st[(2 * (1 - wg) + 1) * kRowsQ + il];
        const float mm = fmaxf(m, mo);
        const float ll = (mm == -INFINITY) ? 0.f
                                           : l * ex2_approx(m - mm) + lo * ex2_approx(mo - mm);
        L2 = (ll > 0.f) ? mm + lg2_approx(ll) : INFINITY;
        merged = true;
      }
      const uint32_t tSb = tS + lane_off + 64 * (it % 3);
      if (!mbar_wait(bar(C::bSFull + it % 3), (it / 3) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (!kDq && it < first_out) {
        // statistics step
#pragma unroll
        for (int c = 0; c < kStepKV / 32; ++c) {
          const int base = jj0 + 32 * c;
          const uint32_t allow =
              bit_range(p.window > 0 ? i - p.window + 1 - base : 0, min(p.N - base, p.causal ? i + 1 - base : 32));
          uint32_t sr[32];
          tmem_ld32(tSb + 32 * c, sr);
          tmem_ld_wait(sr);
          float x[32];
          float mx = m;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = ((allow >> e) & 1u) ? __uint_as_float(sr[e]) * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, x[e]);
          }
          if (mx != -INFINITY) {
            float acc = l * ex2_approx(m - mx);
#pragma unroll
            for (int e = 0; e < 32; ++e) acc += ex2_approx(x[e] - mx);
            l = acc;
            m = mx;
          }
        }
        tc_fence_before();
        mbar_arrive(bar(C::bPFull + wg));
        continue;
      }
      bool lo_any = false;
#pragma unroll
      for (int c = 0; c < kStepKV / 32; ++c) {
        const int base = jj0 + 32 * c;
        const uint32_t allow =
            bit_range(p.window > 0 ? i - p.window + 1 - base : 0, min(p.N - base, p.causal ? i + 1 - base : 32));
        uint32_t keep = 0xFFFFFFFFu;
        if constexpr (kDrop) keep = keep_bits_for_query(p.drop, bh, p.N, i, base);
        uint32_t sr[32], dr[32];
        tmem_ld32(tSb + 32 * c, sr);
        if constexpr (kDq) {
          tmem_ld32(tdPb + 32 * c, dr);
          tmem_ld_wait2(sr, dr);
          if (c == kStepKV / 32 - 1) {
            // every dP column of this buffer is in registers: the next dP may land
            tc_fence_before();
            mbar_arrive(bar(C::bDPEmpty + wg));
          }
        } else {
          tmem_ld_wait(sr);
        }
        float outv[32];
        float cmax = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const bool on = (allow >> e) & 1u;
          const float pv = on ? ex2_approx(fmaf(__uint_as_float(sr[e]), p.scale_log2, -L2)) : 0.f;
          cmax = fmaxf(cmax, pv);
          const bool kept = !kDrop || ((keep >> e) & 1u);
          const float rp = kDrop ? p.drop.rp : 1.f;
          if constexpr (kDq) {
            const float dpv = kept ? __uint_as_float(dr[e]) * rp : 0.f;
            outv[e] = pv * (dpv - Dv);
          } else {
            outv[e] = kept ? pv * rp : 0.f;
          }
        }
        uint32_t hv[16], ev[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) hv[x] = pack2<kBf16>(outv[2 * x], outv[2 * x + 1]);
        const bool split_c = __any_sync(0xFFFFFFFFu, cmax > kSplitThreshold);
        lo_any |= split_c;
        if (split_c) {
#pragma unroll
          for (int x = 0; x < 16; ++x) ev[x] = pack2_residual<kBf16>(outv[2 * x], outv[2 * x + 1], hv[x]);
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) ev[x] = 0u;
        }
        uint32_t img[32];
        interleave_split(hv, ev, img);
        tmem_st32(tSb + 32 * c, img);
      }
      tmem_st_wait();
      if (lane == 0) flags[4 * wg + wq] = lo_any ? 1 : 0;
      tc_fence_before();
      mbar_arrive(bar(C::bPFull + wg));
    }
    if (!kDq && ok && !merged) {
      // This warpgroup saw no output step (tiny key ranges): still publish its statistics.
      float* st = reinterpret_cast<float*>(smem + C::oStats);
      st[(2 * wg) * kRowsQ + il] = m;
      st[(2 * wg + 1) * kRowsQ + il] = l;
      mbar_arrive(bar(C::bStats));
      if (!mbar_wait(bar(C::bStats), 0, abort_flag, p.status)) ok = false;
      const float mo = st[(2 * (1 - wg)) * kRowsQ + il], lo = st[(2 * (1 - wg) + 1) * kRowsQ + il];
      const float mm = fmaxf(m, mo);
      const float ll = (mm == -INFINITY) ? 0.f : l * ex2_approx(m - mm) + lo * ex2_approx(mo - mm);
      L2 = (ll > 0.f) ? mm + lg2_approx(ll) : INFINITY;
    }
    // Epilogue: O (forward) or scale * dQ; warpgroup w writes columns [w*d/2, (w+1)*d/2).
    const bool have_acc = nsteps > first_out;
    if (ok && have_acc) ok = mbar_wait(bar(C::bAcc), 0, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      const long long off = (long long)b * p.sb + (long long)i * p.sn + (long long)h * p.sh;
      uint16_t* dst = static_cast<uint16_t*>(p.out) + off;
      const float mul = kDq ? p.scale : 1.f;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = wg * (D / 2) + 32 * c;
        uint32_t r[32];
        if (have_acc) {
          tmem_ld32(tAcc + lane_off + col, r);
          tmem_ld_wait(r);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          w[x] = pack2<kBf16>(__uint_as_float(r[2 * x]) * mul, __uint_as_float(r[2 * x + 1]) * mul);
        if (i < p.N) {
          uint4* g = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
          for (int t = 0; t < 4; ++t) g[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
      }
      if (!kDq && wg == 0 && i < p.N)
        p.lse_out[(long long)bh * p.N + i] = (L2 == INFINITY) ? -INFINITY : L2 * 0.6931471805599453f;
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

template <int D, bool kBf16, int kMode, bool kDrop>
static cudaError_t launch_q_t(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  using C = QCfg<D, kMode>;
  auto kern = qmajor_kernel<D, kBf16, kMode, kDrop>;
  const int smem = (int)(C::kSmem > kMinSmemOneCtaPerSm ? C::kSmem : kMinSmemOneCtaPerSm);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int tiles = (p.N + kRowsQ - 1) / kRowsQ;
  const unsigned grid = (unsigned)(tiles * p.B * p.H);
  kern<<<grid, 384, smem, st>>>(p, maps[0], maps[1], maps[2], maps[3]);
  return cudaGetLastError();
}

template <int D, bool kBf16>
static cudaError_t launch_q_d(const AttnParams& p, bool dq_mode, const CUtensorMap* maps, cudaStream_t st) {
  const bool drop = p.drop.threshold != 0;
  if (dq_mode)
    return drop ? launch_q_t<D, kBf16, kModeDq, true>(p, maps, st) : launch_q_t<D, kBf16, kModeDq, false>(p, maps, st);
  return drop ? launch_q_t<D, kBf16, kModeFwd, true>(p, maps, st) : launch_q_t<D, kBf16, kModeFwd, false>(p, maps, st);
}

// maps: Q, K, V, dO (Q/dO boxes of kRowsQ rows, K/V boxes of kStepKV rows).
cudaError_t launch_qmajor_tc(const AttnParams& p, bool bf16, bool dq_mode, const CUtensorMap* maps,
                             cudaStream_t st) {
  if (p.d == 128)
    return bf16 ? launch_q_d<128, true>(p, dq_mode, maps, st) : launch_q_d<128, false>(p, dq_mode, maps, st);
  return bf16 ? launch_q_d<64, true>(p, dq_mode, maps, st) : launch_q_d<64, false>(p, dq_mode, maps, st);
}

}  // namespace fa
