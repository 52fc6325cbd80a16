// Key/value-major backward kernel on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// "FlashAttention backward", §The loop structure: the outer loop runs over
// key/value blocks and the inner loop over query blocks, so that dK_j and dV_j
// accumulate on chip and are written once. Per (query step, key block) pair:
//
//   S^T  = K_j Q_i^T            (recomputed, "Lecture 7" §The recomputation trick)
//   dP~T = V_j dO_i^T
//   P^T  = exp2(S^T * scale*log2e - L_i*log2e)    masked pairs -> 0
//   P~T  = P^T o Z/(1-p),  dP^T = dP~T o Z/(1-p)  (dropout, "Lecture 7" §Dropout)
//   dS^T = P^T o (dP^T - D_i)                     ("FlashAttention backward" §The gradients)
//   dV  += P~T dO_i,   dK += dS^T Q_i             (fp32 in TMEM, scaled by `scale` on store)
//   atomic mode only: dQ_i^T = K_j^T dS^T, added into an fp32 HBM accumulator
//   with red.add ("FlashAttention backward" §The loop structure, choice (a)).
//
// Keys sit on the 128 TMEM lanes, so one thread owns one key row of S^T and
// dP^T, and its row of P~T / dS^T goes to shared memory in the 128-byte
// swizzled layout the MMA reads as a K-major A operand. The same dS^T tile is
// read as an MN-major B operand for dQ^T.
//
// Warp roles: warp 0 issues TMA loads, warp 1 owns TMEM and issues MMAs,
// warps 4-7 turn S/dP into P/dS and write the dK/dV epilogue, warps 8-11
// (atomic mode) drain dQ^T from TMEM into the HBM accumulator.
//
// TMEM columns (512 allocated): [0,128) S^T double buffer (reused for dQ^T in
// atomic mode once S^T has been consumed), [128,256) dP^T double buffer,
// [256,256+d) dV, [256+d,256+2d) dK.
#include "fa_internal.h"

namespace fa {

template <int D>
struct KVCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kNS = (D == 128) ? 2 : 4;               // Q/dO pipeline stages
  static constexpr uint32_t kKVPanel = kRowsKV * 128;          // 16 KB: 128 rows x 64 elements
  static constexpr uint32_t kKVTile = kPanels * kKVPanel;
  static constexpr uint32_t kQPanel = kStepQ * 128;            // 8 KB: 64 rows x 64 elements
  static constexpr uint32_t kQTile = kPanels * kQPanel;
  static constexpr uint32_t kPTile = kRowsKV * kStepQ * 2;     // 16 KB: 128 keys x 64 queries
  static constexpr uint32_t oK = 0;
  static constexpr uint32_t oV = oK + kKVTile;
  static constexpr uint32_t oQ = oV + kKVTile;
  static constexpr uint32_t oDO = oQ + kNS * kQTile;
  static constexpr uint32_t oP = oDO + kNS * kQTile;    // P~T, rounded to 16 bits
  static constexpr uint32_t oDS = oP + kPTile;           // dS^T, rounded
  static constexpr uint32_t oPlo = oDS + kPTile;         // rounding residuals (split tiles only)
  static constexpr uint32_t oDSlo = oPlo + kPTile;
  static constexpr uint32_t oL = oDSlo + kPTile;
  static constexpr uint32_t oD = oL + kNS * kStepQ * 4;
  static constexpr uint32_t oBar = oD + kNS * kStepQ * 4;
  // barrier indices
  static constexpr int bKV = 0;
  static constexpr int bQFull = 1;
  static constexpr int bQEmpty = bQFull + kNS;
  static constexpr int bSFull = bQEmpty + kNS;
  static constexpr int bSEmpty = bSFull + 2;
  static constexpr int bPFull = bSEmpty + 2;
  static constexpr int bPEmpty = bPFull + 1;
  static constexpr int bDQFull = bPEmpty + 1;
  static constexpr int bAcc = bDQFull + 2;
  static constexpr int bDrain = bAcc + 1;
  static constexpr int bVote = bDrain + 1;
  static constexpr int kBars = bVote + 1;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = oAbort + 8;         // per-warp "split this tile" votes
  static constexpr uint32_t kSmem = oFlags + 16 + 1024;  // + slack for 1024-byte alignment
};

template <int D, bool kBf16, bool kAtomic>
__global__ void __launch_bounds__(kAtomic ? 384 : 256, 1)
    bwd_dkdv_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmDO) {
  using C = KVCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oAbort);
  auto bar = [&](int idx) -> uint32_t { return sb + C::oBar + 8u * idx; };

  // Work unit: (batch*head, key block), heaviest key blocks first under a causal mask.
  const int BH = p.B * p.H;
  const int kv_tile = blockIdx.x / BH;
  const int bh = blockIdx.x % BH;
  const int b = bh / p.H, h = bh % p.H;
  const int j0 = kv_tile * kRowsKV;
  const int i_first = p.causal ? j0 : 0;
  int i_last = p.N - 1;
  if (p.window > 0) i_last = min(i_last, j0 + kRowsKV - 2 + p.window);
  const int nsteps = (i_last >= i_first) ? (i_last - i_first) / kStepQ + 1 : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bKV), 1);
    for (int s = 0; s < C::kNS; ++s) {
      mbar_init(bar(C::bQFull + s), 1);
      mbar_init(bar(C::bQEmpty + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::bSFull + x), 1);
      mbar_init(bar(C::bSEmpty + x), kAtomic ? 256 : 128);
      mbar_init(bar(C::bDQFull + x), 1);
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
    prefetch_tmap(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::oTmemSlot);

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::bKV), 2 * C::kKVTile);
      for (int pn = 0; pn < C::kPanels; ++pn) {
        tma_load_4d(sb + C::oK + pn * C::kKVPanel, &tmK, bar(C::bKV), 64 * pn, j0, h, b);
        tma_load_4d(sb + C::oV + pn * C::kKVPanel, &tmV, bar(C::bKV), 64 * pn, j0, h, b);
      }
      int issued = 0;
      for (int it = 0; it < nsteps; ++it) {
        const int s = it % C::kNS;
        if (!mbar_wait(bar(C::bQEmpty + s), ((it / C::kNS) & 1) ^ 1, abort_flag, p.status)) break;
        const int i0 = i_first + it * kStepQ;
        mbar_arrive_expect_tx(bar(C::bQFull + s), 2 * C::kQTile + 2 * kStepQ * 4);
        for (int pn = 0; pn < C::kPanels; ++pn) {
          tma_load_4d(sb + C::oQ + s * C::kQTile + pn * C::kQPanel, &tmQ, bar(C::bQFull + s), 64 * pn, i0,
                      h, b);
          tma_load_4d(sb + C::oDO + s * C::kQTile + pn * C::kQPanel, &tmDO, bar(C::bQFull + s), 64 * pn,
                      i0, h, b);
        }
        const long long ws = (long long)bh * p.n_pad + i0;
        bulk_load(sb + C::oL + s * kStepQ * 4, p.ws_L2 + ws, kStepQ * 4, bar(C::bQFull + s));
        bulk_load(sb + C::oD + s * kStepQ * 4, p.ws_D + ws, kStepQ * 4, bar(C::bQFull + s));
        issued = it + 1;
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        mbar_wait_drain(bar(C::bKV), 0, p.status);
        for (int it = max(0, issued - C::kNS); it < issued; ++it)
          mbar_wait_drain(bar(C::bQFull + it % C::kNS), (it / C::kNS) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc(128, kStepQ, kBf16, false, false);
      constexpr uint32_t idG = make_idesc(128, D, kBf16, false, true);
      constexpr uint32_t idQ = make_idesc(128, kStepQ, kBf16, true, true);
      const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
      bool ok = mbar_wait(bar(C::bKV), 0, abort_flag, p.status);
      tc_fence_after();
      auto grads = [&](int t) -> bool {
        const int bp = t & 1, sp = t % C::kNS;
        if (!mbar_wait(bar(C::bPFull), t & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const volatile int* flags = reinterpret_cast<const volatile int*>(smem + C::oFlags);
        const bool split = (flags[0] | flags[1] | flags[2] | flags[3]) != 0;
        const uint32_t doB = sb + C::oDO + sp * C::kQTile, qB = sb + C::oQ + sp * C::kQTile;
        // dV += P~T dO and dK += dS^T Q, from the rounded tiles and, on split
        // tiles, again from the rounding residuals.
        for (int part = 0; part < (split ? 2 : 1); ++part) {
          const uint32_t pA = sb + (part ? C::oPlo : C::oP), dsA = sb + (part ? C::oDSlo : C::oDS);
#pragma unroll
          for (int k = 0; k < kStepQ / 16; ++k)
            tc_mma_ss(tdV, make_sdesc(pA + 32 * k, 16, 1024), make_sdesc(doB + 2048 * k, C::kQPanel, 1024), idG,
                      (t > 0 || k > 0 || part > 0) ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < kStepQ / 16; ++k)
            tc_mma_ss(tdK, make_sdesc(dsA + 32 * k, 16, 1024), make_sdesc(qB + 2048 * k, C::kQPanel, 1024), idG,
                      (t > 0 || k > 0 || part > 0) ? 1u : 0u);
        }
        if constexpr (kAtomic) {
          // dQ^T (d x 64) = K_j^T (d x 128 keys) . dS^T (128 keys x 64); for d = 64 the
          // upper 64 rows of the 128-row MMA are ignored.
          for (int part = 0; part < (split ? 2 : 1); ++part) {
            const uint32_t dsA = sb + (part ? C::oDSlo : C::oDS);
#pragma unroll
            for (int k = 0; k < kRowsKV / 16; ++k)
              tc_mma_ss(tS + 64 * bp, make_sdesc(sb + C::oK + 2048 * k, C::kKVPanel, 1024),
                        make_sdesc(dsA + 2048 * k, C::kPTile, 1024), idQ, (k > 0 || part > 0) ? 1u : 0u);
          }
          tc_commit(bar(C::bDQFull + bp));
        }
        tc_commit(bar(C::bPEmpty));
        tc_commit(bar(C::bQEmpty + sp));
        return true;
      };
      for (int it = 0; ok && it < nsteps; ++it) {
        const int s = it % C::kNS, bb = it & 1;
        if (!mbar_wait(bar(C::bQFull + s), (it / C::kNS) & 1, abort_flag, p.status)) { ok = false; break; }
        if (!mbar_wait(bar(C::bSEmpty + bb), ((it >> 1) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qB = sb + C::oQ + s * C::kQTile, doB = sb + C::oDO + s * C::kQTile;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (k >> 2) * C::kKVPanel + (k & 3) * 32, qo = (k >> 2) * C::kQPanel + (k & 3) * 32;
          tc_mma_ss(tS + 64 * bb, make_sdesc(sb + C::oK + ko, 16, 1024), make_sdesc(qB + qo, 16, 1024), idS,
                    k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ko = (k >> 2) * C::kKVPanel + (k & 3) * 32, qo = (k >> 2) * C::kQPanel + (k & 3) * 32;
          tc_mma_ss(tdP + 64 * bb, make_sdesc(sb + C::oV + ko, 16, 1024), make_sdesc(doB + qo, 16, 1024), idS,
                    k > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::bSFull + bb));
        if (it > 0 && !grads(it - 1)) { ok = false; break; }
      }
      if (ok && nsteps > 0) ok = grads(nsteps - 1);
      tc_commit(bar(C::bAcc));
      if (!ok) {
        // Drain MMAs already issued before TMEM is released.
        tc_commit(bar(C::bDrain));
        mbar_wait_drain(bar(C::bDrain), 0, p.status);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // --------------------- softmax-gradient warpgroup + epilogue -------------
    const int wq = warp & 3;
    const int jl = wq * 32 + lane;
    const int j = j0 + jl;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool drop = p.drop.threshold != 0;
    bool ok = true;
    volatile int* flags = reinterpret_cast<volatile int*>(smem + C::oFlags);
    const uint32_t pRow = sb + C::oP + jl * 128, dsRow = sb + C::oDS + jl * 128;
    const uint32_t pRowLo = sb + C::oPlo + jl * 128, dsRowLo = sb + C::oDSlo + jl * 128;
    for (int it = 0; it < nsteps; ++it) {
      const int bb = it & 1, s = it % C::kNS;
      const int i0 = i_first + it * kStepQ;
      if (!mbar_wait(bar(C::bQFull + s), (it / C::kNS) & 1, abort_flag, p.status) ||
          !mbar_wait(bar(C::bSFull + bb), (it >> 1) & 1, abort_flag, p.status) ||
          !mbar_wait(bar(C::bPEmpty), (it & 1) ^ 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* Ls = reinterpret_cast<const float*>(smem + C::oL + s * kStepQ * 4);
      const float* Ds = reinterpret_cast<const float*>(smem + C::oD + s * kStepQ * 4);
      const bool need_mask = (p.causal && i0 < j0 + kRowsKV - 1) ||
                             (p.window > 0 && i0 + kStepQ - 1 - p.window >= j0) || (j0 + kRowsKV > p.N);
      // Pass 0 writes P~T and dS^T rounded to 16 bits; pass 1 (only when some
      // P of the tile exceeds kSplitThreshold) recomputes them from TMEM and
      // writes the rounding residuals.
      float pmax = 0.f;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        if (pass == 1) {
          const bool mine = __any_sync(0xffffffffu, pmax > kSplitThreshold);
          if (lane == 0) flags[wq] = mine ? 1 : 0;
          mbar_arrive(bar(C::bVote));
          if (!mbar_wait(bar(C::bVote), it & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const bool split = (flags[0] | flags[1] | flags[2] | flags[3]) != 0;
          if (!split) break;
        }
#pragma unroll
        for (int c = 0; c < kStepQ / 32; ++c) {
          uint32_t sr[32], dr[32];
          tmem_ld32(tmem + lane_off + 64 * bb + 32 * c, sr);
          tmem_ld32(tmem + lane_off + 128 + 64 * bb + 32 * c, dr);
          tmem_ld_wait2(sr, dr);
          const uint32_t keep = drop ? keep_bits_for_key(p.drop, bh, p.N, i0 + 32 * c, j) : 0xFFFFFFFFu;
          const float rp = drop ? p.drop.rp : 1.f;
          uint32_t pp[16], dd[16];
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            float pt[2], ds[2];
#pragma unroll
            for (int y = 0; y < 2; ++y) {
              const int col = 32 * c + x + y;
              const int i = i0 + col;
              float pv = ex2_approx(fmaf(__uint_as_float(sr[x + y]), p.scale_log2, -Ls[col]));
              if (need_mask && !pair_allowed(p, i, j)) pv = 0.f;
              pmax = fmaxf(pmax, pv);
              const bool kept = (keep >> (x + y)) & 1u;
              const float dpv = kept ? __uint_as_float(dr[x + y]) * rp : 0.f;
              const float ptv = kept ? pv * rp : 0.f;
              pt[y] = ptv;
              ds[y] = pv * (dpv - Ds[col]);
            }
            const uint32_t ph = pack2<kBf16>(pt[0], pt[1]), dh = pack2<kBf16>(ds[0], ds[1]);
            pp[x >> 1] = pass ? pack2_residual<kBf16>(pt[0], pt[1], ph) : ph;
            dd[x >> 1] = pass ? pack2_residual<kBf16>(ds[0], ds[1], dh) : dh;
          }
          const uint32_t pr = pass ? pRowLo : pRow, dr2 = pass ? dsRowLo : dsRow;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t chunk = (uint32_t)((4 * c + t) ^ (jl & 7)) << 4;
            st_shared_v4(pr + chunk, pp[4 * t], pp[4 * t + 1], pp[4 * t + 2], pp[4 * t + 3]);
            st_shared_v4(dr2 + chunk, dd[4 * t], dd[4 * t + 1], dd[4 * t + 2], dd[4 * t + 3]);
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(bar(C::bSEmpty + bb));
      fence_proxy_async_smem();
      mbar_arrive(bar(C::bPFull));
    }
    // Epilogue: dV and scale * dK, rounded to the tensor dtype, one key row per thread.
    if (ok && nsteps > 0) ok = mbar_wait(bar(C::bAcc), 0, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      const long long off = (long long)b * p.sb + (long long)j * p.sn + (long long)h * p.sh;
      uint16_t* dv = static_cast<uint16_t*>(p.dv) + off;
      uint16_t* dk = static_cast<uint16_t*>(p.dk) + off;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col0 = 256 + which * D;
        const float mul = which ? p.scale : 1.f;
        uint16_t* dst = which ? dk : dv;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (nsteps > 0) {
            tmem_ld32(tmem + lane_off + col0 + 32 * c, r);
            tmem_ld_wait(r);
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) r[x] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            w[x] = pack2<kBf16>(__uint_as_float(r[2 * x]) * mul, __uint_as_float(r[2 * x + 1]) * mul);
          if (j < p.N) {
            uint4* g = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
            for (int t = 0; t < 4; ++t) g[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
          }
        }
      }
    }
  } else if (kAtomic && warp >= 8) {
    // ------------------ dQ drain: TMEM dQ^T -> fp32 HBM accumulator ----------
    const int wq = warp & 3;
    const int dd = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    for (int it = 0; it < nsteps; ++it) {
      const int bb = it & 1;
      if (!mbar_wait(bar(C::bDQFull + bb), (it >> 1) & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const int i0 = i_first + it * kStepQ;
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem + lane_off + 64 * bb, r0);
      tmem_ld32(tmem + lane_off + 64 * bb + 32, r1);
      tmem_ld_wait2(r0, r1);
      tc_fence_before();
      mbar_arrive(bar(C::bSEmpty + bb));
      if (dd < D) {
        float* dst = p.ws_dq + ((long long)bh * p.n_pad + i0) * D + dd;
#pragma unroll
        for (int x = 0; x < 32; ++x) atomicAdd(dst + x * D, __uint_as_float(r0[x]));
#pragma unroll
        for (int x = 0; x < 32; ++x) atomicAdd(dst + (32 + x) * D, __uint_as_float(r1[x]));
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

template <int D, bool kBf16, bool kAtomic>
static cudaError_t launch_dkdv_t(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  using C = KVCfg<D>;
  auto kern = bwd_dkdv_kernel<D, kBf16, kAtomic>;
  const int smem = (int)(C::kSmem > kMinSmemOneCtaPerSm ? C::kSmem : kMinSmemOneCtaPerSm);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int tiles = (p.N + kRowsKV - 1) / kRowsKV;
  const unsigned grid = (unsigned)(tiles * p.B * p.H);
  kern<<<grid, kAtomic ? 384 : 256, smem, st>>>(p, maps[0], maps[1], maps[2], maps[3]);
  return cudaGetLastError();
}

// maps: Q, K, V, dO (Q/dO boxes of kStepQ rows, K/V boxes of kRowsKV rows).
cudaError_t launch_bwd_dkdv_tc(const AttnParams& p, bool bf16, bool atomic, const CUtensorMap* maps,
                               cudaStream_t st) {
  if (p.d == 128) {
    if (bf16) return atomic ? launch_dkdv_t<128, true, true>(p, maps, st) : launch_dkdv_t<128, true, false>(p, maps, st);
    return atomic ? launch_dkdv_t<128, false, true>(p, maps, st) : launch_dkdv_t<128, false, false>(p, maps, st);
  }
  if (bf16) return atomic ? launch_dkdv_t<64, true, true>(p, maps, st) : launch_dkdv_t<64, true, false>(p, maps, st);
  return atomic ? launch_dkdv_t<64, false, true>(p, maps, st) : launch_dkdv_t<64, false, false>(p, maps, st);
}

size_t smem_bwd_dkdv_tc(int d) { return d == 128 ? KVCfg<128>::kSmem : KVCfg<64>::kSmem; }

}  // namespace fa
