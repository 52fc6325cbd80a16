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
// D_i are per-thread scalars. Warp 0 issues TMA loads, warp 1 owns TMEM and
// issues MMAs, warps 4-7 run the row math and the epilogue.
//
// TMEM columns: [0,128) S double buffer, [128,256) dP double buffer (dQ mode),
// [256,256+d) the O or dQ accumulator.
#include "fa_internal.h"

namespace fa {

constexpr int kModeFwd = 0;
constexpr int kModeDq = 1;

template <int D, int kMode>
struct QCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kNS = (D == 128) ? 3 : 4;               // K/V pipeline stages
  static constexpr uint32_t kRowPanel = kRowsQ * 128;          // 16 KB
  static constexpr uint32_t kRowTile = kPanels * kRowPanel;
  static constexpr uint32_t kKVPanel = kStepKV * 128;          // 8 KB
  static constexpr uint32_t kKVTile = kPanels * kKVPanel;
  static constexpr uint32_t kPTile = kRowsQ * kStepKV * 2;     // 16 KB
  static constexpr uint32_t oQ = 0;
  static constexpr uint32_t oDO = oQ + kRowTile;
  static constexpr uint32_t oK = oDO + (kMode == kModeDq ? kRowTile : 0);
  static constexpr uint32_t oV = oK + kNS * kKVTile;
  static constexpr uint32_t oP = oV + kNS * kKVTile;   // P~ or dS rounded to 16 bits
  static constexpr uint32_t oPlo = oP + kPTile;         // rounding residuals (split tiles only)
  static constexpr uint32_t oBar = oPlo + kPTile;
  static constexpr int bRes = 0;
  static constexpr int bKVFull = 1;
  static constexpr int bKVEmpty = bKVFull + kNS;
  static constexpr int bSFull = bKVEmpty + kNS;
  static constexpr int bSEmpty = bSFull + 2;
  static constexpr int bPFull = bSEmpty + 2;
  static constexpr int bPEmpty = bPFull + 1;
  static constexpr int bAcc = bPEmpty + 1;
  static constexpr int bDrain = bAcc + 1;
  static constexpr int bVote = bDrain + 1;
  static constexpr int kBars = bVote + 1;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = oAbort + 8;        // per-warp "split this tile" votes
  static constexpr uint32_t kSmem = oFlags + 16 + 1024;
};

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool kBf16, int kMode>
__global__ void __launch_bounds__(256, 1)
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
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::bSFull + x), 1);
      mbar_init(bar(C::bSEmpty + x), 128);
    }
    mbar_init(bar(C::bPFull), 128);
    mbar_init(bar(C::bPEmpty), 1);
    mbar_init(bar(C::bAcc), 1);
    mbar_init(bar(C::bDrain), 1);
    mbar_init(bar(C::bVote), 128);
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

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::bRes), (kDq ? 2 : 1) * C::kRowTile);
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
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc(128, kStepKV, kBf16, false, false);
      constexpr uint32_t idO = make_idesc(128, D, kBf16, false, true);
      const uint32_t tS = tmem, tdP = tmem + 128, tAcc = tmem + 256;
      bool ok = mbar_wait(bar(C::bRes), 0, abort_flag, p.status);
      tc_fence_after();
      // Second MMA of an output step: acc += (P~ or dS) . (V_j or K_j).
      auto second = [&](int t) -> bool {
        const int u = t - first_out;
        const int sp = t % C::kNS;
        if (!mbar_wait(bar(C::bPFull), u & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const volatile int* flags = reinterpret_cast<const volatile int*>(smem + C::oFlags);
        const bool split = (flags[0] | flags[1] | flags[2] | flags[3]) != 0;
        const uint32_t bOp = sb + (kDq ? C::oK : C::oV) + sp * C::kKVTile;
        // From the rounded tile and, on split tiles, again from the residuals.
        for (int part = 0; part < (split ? 2 : 1); ++part) {
          const uint32_t aP = sb + (part ? C::oPlo : C::oP);
#pragma unroll
          for (int k = 0; k < kStepKV / 16; ++k)
            tc_mma_ss(tAcc, make_sdesc(aP + 32 * k, 16, 1024), make_sdesc(bOp + 2048 * k, C::kKVPanel, 1024),
                      idO, (u > 0 || k > 0 || part > 0) ? 1u : 0u);
        }
        tc_commit(bar(C::bPEmpty));
        tc_commit(bar(C::bKVEmpty + sp));
        return true;
      };
      for (int it = 0; ok && it < nsteps; ++it) {
        const int s = it % C::kNS, bb = it & 1;
        if (!mbar_wait(bar(C::bKVFull + s), (it / C::kNS) & 1, abort_flag, p.status) ||
            !mbar_wait(bar(C::bSEmpty + bb), ((it >> 1) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kB = sb + C::oK + s * C::kKVTile, vB = sb + C::oV + s * C::kKVTile;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t qo = (k >> 2) * C::kRowPanel + (k & 3) * 32, ko = (k >> 2) * C::kKVPanel + (k & 3) * 32;
          tc_mma_ss(tS + 64 * bb, make_sdesc(sb + C::oQ + qo, 16, 1024), make_sdesc(kB + ko, 16, 1024), idS,
                    k > 0 ? 1u : 0u);
        }
        if constexpr (kDq) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t qo = (k >> 2) * C::kRowPanel + (k & 3) * 32, ko = (k >> 2) * C::kKVPanel + (k & 3) * 32;
            tc_mma_ss(tdP + 64 * bb, make_sdesc(sb + C::oDO + qo, 16, 1024), make_sdesc(vB + ko, 16, 1024), idS,
                      k > 0 ? 1u : 0u);
          }
        }
        tc_commit(bar(C::bSFull + bb));
        if (it < first_out) tc_commit(bar(C::bKVEmpty + s));  // statistics step: K no longer needed
        if (it > first_out && !second(it - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && nsteps > first_out) ok = second(nsteps - 1);
      tc_commit(bar(C::bAcc));
      if (!ok) {
        tc_commit(bar(C::bDrain));
        mbar_wait_drain(bar(C::bDrain), 0, p.status);
      }
    }
  } else if (warp >= 4) {
    // ----------------------- row math + epilogue warpgroup -------------------
    const int wq = warp & 3;
    const int il = wq * 32 + lane;
    const int i = i0 + il;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool drop = p.drop.threshold != 0;
    const long long ws = (long long)bh * p.n_pad + i;  // i < n_pad always
    float L2 = 0.f, Dv = 0.f;
    if (kDq) {
      L2 = p.ws_L2[ws];
      Dv = p.ws_D[ws];
    }
    float m = -INFINITY, l = 0.f;  // forward statistics, log2 domain
    if (!kDq) L2 = INFINITY;
    volatile int* flags = reinterpret_cast<volatile int*>(smem + C::oFlags);
    bool ok = true;
    for (int it = 0; it < nsteps; ++it) {
      const int bb = it & 1;
      const int jt = it >= nkv ? it - nkv : it;
      const int jj0 = j_first + jt * kStepKV;
      if (!mbar_wait(bar(C::bSFull + bb), (it >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const bool need_mask = (p.causal && jj0 + kStepKV - 1 > i0) ||
                             (p.window > 0 && jj0 <= i0 + kRowsQ - 1 - p.window) || (jj0 + kStepKV > p.N);
      if (!kDq && it < first_out) {
        // statistics step
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kStepKV / 32; ++c) {
          uint32_t sr[32];
          tmem_ld32(tmem + lane_off + 64 * bb + 32 * c, sr);
          tmem_ld_wait(sr);
          float x[32];
          float mx = m;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(sr[e]) * p.scale_log2;
            if (need_mask && !pair_allowed(p, i, jj0 + 32 * c + e)) x[e] = -INFINITY;
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
        mbar_arrive(bar(C::bSEmpty + bb));
        if (it == first_out - 1) L2 = (l > 0.f) ? m + lg2_approx(l) : INFINITY;
        continue;
      }
      const int u = it - first_out;
      if (!mbar_wait(bar(C::bPEmpty), (u & 1) ^ 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Pass 0 writes the tile (P~ or dS) rounded to 16 bits; pass 1 (only when
      // some P of the tile exceeds kSplitThreshold) recomputes it from TMEM and
      // writes the rounding residuals.
      float pmax = 0.f;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        if (pass == 1) {
          const bool mine = __any_sync(0xffffffffu, pmax > kSplitThreshold);
          if (lane == 0) flags[wq] = mine ? 1 : 0;
          mbar_arrive(bar(C::bVote));
          if (!mbar_wait(bar(C::bVote), u & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if ((flags[0] | flags[1] | flags[2] | flags[3]) == 0) break;
        }
        const uint32_t pRow = sb + (pass ? C::oPlo : C::oP) + il * 128;
#pragma unroll
        for (int c = 0; c < kStepKV / 32; ++c) {
          uint32_t sr[32], dr[32];
          tmem_ld32(tmem + lane_off + 64 * bb + 32 * c, sr);
          if (kDq) {
            tmem_ld32(tmem + lane_off + 128 + 64 * bb + 32 * c, dr);
            tmem_ld_wait2(sr, dr);
          } else {
            tmem_ld_wait(sr);
          }
          uint32_t pk[16];
          const uint32_t keep = drop ? keep_bits_for_query(p.drop, bh, p.N, i, jj0 + 32 * c) : 0xFFFFFFFFu;
          const float rp = drop ? p.drop.rp : 1.f;
#pragma unroll
          for (int x = 0; x < 32; x += 4) {
            const int jb = jj0 + 32 * c + x;
            float outv[4];
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              float pv = ex2_approx(fmaf(__uint_as_float(sr[x + y]), p.scale_log2, -L2));
              if (need_mask && !pair_allowed(p, i, jb + y)) pv = 0.f;
              pmax = fmaxf(pmax, pv);
              const bool kept = (keep >> (x + y)) & 1u;
              if constexpr (kDq) {
                const float dpv = kept ? __uint_as_float(dr[x + y]) * rp : 0.f;
                outv[y] = pv * (dpv - Dv);
              } else {
                outv[y] = kept ? pv * rp : 0.f;
              }
            }
            const uint32_t h0 = pack2<kBf16>(outv[0], outv[1]), h1 = pack2<kBf16>(outv[2], outv[3]);
            pk[x >> 1] = pass ? pack2_residual<kBf16>(outv[0], outv[1], h0) : h0;
            pk[(x >> 1) + 1] = pass ? pack2_residual<kBf16>(outv[2], outv[3], h1) : h1;
          }
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t chunk = (uint32_t)((4 * c + t) ^ (il & 7)) << 4;
            st_shared_v4(pRow + chunk, pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(bar(C::bSEmpty + bb));
      fence_proxy_async_smem();
      mbar_arrive(bar(C::bPFull));
    }
    // Epilogue: O (forward) or scale * dQ, one query row per thread.
    const bool have_acc = nsteps > first_out;
    if (ok && have_acc) ok = mbar_wait(bar(C::bAcc), 0, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      const long long off = (long long)b * p.sb + (long long)i * p.sn + (long long)h * p.sh;
      uint16_t* dst = static_cast<uint16_t*>(p.out) + off;
      const float mul = kDq ? p.scale : 1.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        if (have_acc) {
          tmem_ld32(tmem + lane_off + 256 + 32 * c, r);
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
          uint4* g = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int t = 0; t < 4; ++t) g[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
      }
      if (!kDq && i < p.N)
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

template <int D, bool kBf16, int kMode>
static cudaError_t launch_q_t(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  using C = QCfg<D, kMode>;
  auto kern = qmajor_kernel<D, kBf16, kMode>;
  const int smem = (int)(C::kSmem > kMinSmemOneCtaPerSm ? C::kSmem : kMinSmemOneCtaPerSm);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int tiles = (p.N + kRowsQ - 1) / kRowsQ;
  const unsigned grid = (unsigned)(tiles * p.B * p.H);
  kern<<<grid, 256, smem, st>>>(p, maps[0], maps[1], maps[2], maps[3]);
  return cudaGetLastError();
}

// maps: Q, K, V, dO (Q/dO boxes of kRowsQ rows, K/V boxes of kStepKV rows).
cudaError_t launch_qmajor_tc(const AttnParams& p, bool bf16, bool dq_mode, const CUtensorMap* maps,
                             cudaStream_t st) {
  if (p.d == 128) {
    if (bf16) return dq_mode ? launch_q_t<128, true, kModeDq>(p, maps, st) : launch_q_t<128, true, kModeFwd>(p, maps, st);
    return dq_mode ? launch_q_t<128, false, kModeDq>(p, maps, st) : launch_q_t<128, false, kModeFwd>(p, maps, st);
  }
  if (bf16) return dq_mode ? launch_q_t<64, true, kModeDq>(p, maps, st) : launch_q_t<64, true, kModeFwd>(p, maps, st);
  return dq_mode ? launch_q_t<64, false, kModeDq>(p, maps, st) : launch_q_t<64, false, kModeFwd>(p, maps, st);
}

size_t smem_qmajor_tc(int d, bool dq_mode) {
  if (d == 128) return dq_mode ? QCfg<128, kModeDq>::kSmem : QCfg<128, kModeFwd>::kSmem;
  return dq_mode ? QCfg<64, kModeDq>::kSmem : QCfg<64, kModeFwd>::kSmem;
}

}  // namespace fa
