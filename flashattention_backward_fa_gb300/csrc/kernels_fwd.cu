// Forward (O and the row log-sum-exp L) on the sm_103a tensor cores, with two
// query tiles per CTA in ping-pong and one thread per query row.
//
// "FlashAttention backward", §What the forward left behind: the backward needs
// the output O and L = m + log(l) (natural log) per query row. One pass over
// the key blocks with an online softmax ("Lecture 7", §The recomputation
// trick: the forward keeps only O and L):
//   S = Q K_j^T (fp32, TMEM), m = running row maximum of S * scale * log2e,
//   P = exp2(S * scale * log2e - m), l += rowsum(P), O += P V_j;
//   O = O / l and L = (m + log2 l) * ln 2 at the end.
//
// Layout. A CTA owns 256 queries of one (batch, head) as two 128-row tiles A
// and B. TMEM: S_A [0, 128), S_B [128, 256), O_A [256, 256 + d), O_B after it.
// Two threads own one query row of a tile (the same TMEM lane, in two warps on
// one scheduler), 64 keys of a block each: per block they exchange only their
// halves' maxima (shared memory and an mbarrier of the two warps); each keeps its
// half's running sum, and the two sums are added once at the end. The MMA
// warp alternates the tiles: while tile A's warps turn S_A(j) into P_A(j), the
// tensor cores run O_B += P_B(j-1) V_{j-1} and S_B(j); then the roles swap.
// P is written back over the S columns it came from as a 16-bit image (eight
// rounded columns, then eight residual columns per 16-key MMA K step; the
// residual MMAs run only where a probability may exceed 1/64 of the row sum,
// as in the other kernels), and the O MMA reads it from TMEM. The next S MMA
// of a tile is issued right behind that tile's O MMA: tcgen05 MMAs issued by
// one thread execute in order, so the O MMA has read the image before S
// overwrites it.
//
// The row maximum's reference moves only when the block maximum exceeds it by
// more than 2^8 (so probabilities relative to a stale reference stay below 2^8);
// then the row of O is rescaled in TMEM after that tile's previous O MMA.
//
// Warp roles (576 threads): warp 0 issues TMA loads (Q_A, Q_B once; K and V
// per key block into rings), warp 1 owns TMEM and issues every MMA; warps 2-9
// are tile A's softmax warps (2-5 the first 64 keys of each block, 6-9 the last
// 64), warps 10-17 tile B's. A warp reaches the TMEM lanes of its quarter
// (warp % 4), so the two warps of a row share a scheduler. This path serves 16-bit inputs with d in {64, 128}, fixed-length or
// packed sequences, without dropout, ALiBi, an attention bias or a window.
#include "fa_internal.h"

namespace fa {

constexpr int kFwdThreads = 576;
constexpr int kFwdRows = 256;  // queries per CTA (two 128-row tiles)
// CTAs are launched in groups of 16 (batch, head) units, tiles outermost within a
// group (heaviest first). The forward streams K and V once per 256-query tile, so
// it gains more from the balance of larger groups than from the L2 sharing of the
// backward's groups of 8 (measured at bf16 causal d = 128: 1x32x8192 0.537 ->
// 0.528 ms, 4x16x2048 0.117 -> 0.107 ms, 1x8x32768 1.86-1.92 -> 1.82 ms).
constexpr int kFwdUnitGroup = 16;
// The reference maximum of a row moves only when a block's maximum exceeds it
// by more than this (log2 units), bounding relative probabilities by 2^8.
constexpr float kFwdRescaleLog2 = 8.f;

__device__ __forceinline__ float lg2_fwd(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct FwdCfg {
  static constexpr int kPanels = D / 64;
  static constexpr uint32_t kPanel = 128 * 128;            // 16 KB: 128 rows x 64 elements
  static constexpr uint32_t kTile = kPanels * kPanel;      // one 128-row tile of Q, K or V
  static constexpr int kNK = D == 64 ? 4 : 2;              // K ring stages
  static constexpr int kNV = D == 64 ? 4 : 2;              // V ring stages
  static constexpr uint32_t oQA = 0;
  static constexpr uint32_t oQB = kTile;
  static constexpr uint32_t oK = 2 * kTile;
  static constexpr uint32_t oV = oK + kNK * kTile;
  static constexpr uint32_t oBar = oV + kNV * kTile;
  static constexpr int bQ = 0;                             // Q_A, Q_B landed
  static constexpr int bKFull = 1;
  static constexpr int bKEmpty = bKFull + kNK;
  static constexpr int bVFull = bKEmpty + kNK;
  static constexpr int bVEmpty = bVFull + kNV;
  static constexpr int bSFull = bVEmpty + kNV;             // [2 tiles] S(j) landed
  static constexpr int bPFull = bSFull + 2;                // [2] P image of block j written
  static constexpr int bODone = bPFull + 2;                // [2] O MMA of block j done
  static constexpr int bDrain = bODone + 2;
  static constexpr int bXchg = bDrain + 1;                 // [tile][lane quarter][block parity] row-maximum exchange
  static constexpr int bSum = bXchg + 16;                  // [tile][lane quarter] final row-sum exchange
  static constexpr int kBars = bSum + 8;
  static constexpr uint32_t oTmemSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oTmemSlot + 8;
  static constexpr uint32_t oFlags = (oAbort + 8 + 15) & ~15u;  // [tile][8 warps] split votes
  // row-maximum exchange between the two warps of a row: [tile][block parity][half][128 rows],
  // then the final row sums [tile][half][128 rows]
  static constexpr uint32_t oXchg = oFlags + 2 * 8 * 4;
  static constexpr uint32_t kSmem = oXchg + (2 * 2 * 2 + 2 * 2) * 128 * 4 + 1024;  // + slack for 1024-byte alignment
  static_assert(kSmem <= 227u * 1024u, "shared memory budget exceeded");
};

template <int D, bool kBf16>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_pingpong_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oAbort);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + C::oFlags);
  auto bar = [&](int idx) -> uint32_t { return sb + C::oBar + 8u * idx; };

  // Unit: (batch * head, or sequence * head of packed input; 256-query tile),
  // the last (heaviest under a causal mask) tiles first. Tile A holds queries
  // q0 .. q0+127 of the unit, tile B q0+128 .. q0+255. A tile past the end of a
  // short sequence has no work: the CTA leaves before any setup.
  Unit u;
  if (!unit_decode(p, blockIdx.x, kFwdRows, true, u, kFwdUnitGroup)) return;
  const int b = u.b, h = u.h;
  const int Nl = u.n;  // rows of this (batch, head) or sequence
  const int q0 = u.tile * kFwdRows;
  const bool hasB = q0 + 128 < Nl;
  // Key blocks of 128: tile X sees blocks 0 .. last[X] (causal: up to its diagonal).
  const int nkb = (Nl + 127) / 128;
  const int lastA = p.causal ? min(nkb - 1, q0 / 128) : nkb - 1;
  const int lastB = hasB ? (p.causal ? min(nkb - 1, q0 / 128 + 1) : nkb - 1) : -1;
  const int nblk = max(lastA, lastB) + 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bQ), 1);
    for (int s = 0; s < C::kNK; ++s) {
      mbar_init(bar(C::bKFull + s), 1);
      mbar_init(bar(C::bKEmpty + s), 1);
    }
    for (int s = 0; s < C::kNV; ++s) {
      mbar_init(bar(C::bVFull + s), 1);
      mbar_init(bar(C::bVEmpty + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::bSFull + x), 1);
      mbar_init(bar(C::bPFull + x), 256);  // the tile's eight softmax warps
      mbar_init(bar(C::bODone + x), 1);
    }
    mbar_init(bar(C::bDrain), 1);
    for (int x = 0; x < 16; ++x) mbar_init(bar(C::bXchg + x), 64);  // the two warps of a row quarter
    for (int x = 0; x < 8; ++x) mbar_init(bar(C::bSum + x), 64);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::oTmemSlot);

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::bQ), (hasB ? 2 : 1) * C::kTile);
      for (int pn = 0; pn < C::kPanels; ++pn) {
        tma_load_4d(sb + C::oQA + pn * C::kPanel, &tmQ, bar(C::bQ), 64 * pn, u.row0 + q0, h, b);
        if (hasB) tma_load_4d(sb + C::oQB + pn * C::kPanel, &tmQ, bar(C::bQ), 64 * pn, u.row0 + q0 + 128, h, b);
      }
      int issuedK = 0, issuedV = 0;
      bool ok = true;
      for (int j = 0; ok && j < nblk; ++j) {
        const int sk = j % C::kNK, sv = j % C::kNV;
        if (!mbar_wait(bar(C::bKEmpty + sk), ((j / C::kNK) & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(bar(C::bKFull + sk), C::kTile);
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_4d(sb + C::oK + sk * C::kTile + pn * C::kPanel, &tmK, bar(C::bKFull + sk), 64 * pn,
                      u.row0 + 128 * j, h, b);
        issuedK = j + 1;
        if (!mbar_wait(bar(C::bVEmpty + sv), ((j / C::kNV) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(C::bVFull + sv), C::kTile);
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_4d(sb + C::oV + sv * C::kTile + pn * C::kPanel, &tmV, bar(C::bVFull + sv), 64 * pn,
                      u.row0 + 128 * j, h, b);
        issuedV = j + 1;
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        mbar_wait_drain(bar(C::bQ), 0, p.status);
        for (int j = max(0, issuedK - C::kNK); j < issuedK; ++j)
          mbar_wait_drain(bar(C::bKFull + j % C::kNK), (j / C::kNK) & 1, p.status);
        for (int j = max(0, issuedV - C::kNV); j < issuedV; ++j)
          mbar_wait_drain(bar(C::bVFull + j % C::kNV), (j / C::kNV) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer --------------------------------
    // S_X(j) = Q_X K_j^T: M = 128 queries, N = 128 keys, K = d (both K-major).
    // O_X += P_X(j) V_j: M = 128, N = d, K = 128 keys; A = the P image in TMEM,
    // B = V_j read MN-major. Order: S_A(0), S_B(0); then per block j:
    // O_A(j), S_A(j+1), O_B(j), S_B(j+1).
    constexpr uint32_t idS = make_idesc(128, 128, kBf16, false, false);
    constexpr uint32_t idO = make_idesc(128, D, kBf16, false, true);
    const uint64_t dQA = make_sdesc(sb + C::oQA, 16, 1024), dQB = make_sdesc(sb + C::oQB, 16, 1024);
    const uint64_t dK0 = make_sdesc(sb + C::oK, 16, 1024);
    const uint64_t dV0 = make_sdesc(sb + C::oV, C::kPanel, 1024);
    bool ok = warp_wait<kIssuerPoll>(bar(C::bQ), 0, abort_flag, p.status);
    // S of tile x (0 = A, 1 = B) for block j; K_j must have landed.
    auto issue_s = [&](int x, int j) {
      const uint64_t kd = desc_add(dK0, (j % C::kNK) * C::kTile);
      const uint64_t qd = x ? dQB : dQA;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        tc_mma_ss_w(tmem + 128 * x, desc_add(qd, (k >> 2) * C::kPanel + (k & 3) * 32),
                    desc_add(kd, (k >> 2) * C::kPanel + (k & 3) * 32), idS, k > 0 ? 1u : 0u);
      tc_commit_w(bar(C::bSFull + x));
    };
    auto issue_o = [&](int x, int j) {
      const uint64_t vd = desc_add(dV0, (j % C::kNV) * C::kTile);
      const uint32_t tO = tmem + 256 + D * x, tP = tmem + 128 * x;
      const int4* f4 = reinterpret_cast<const int4*>(const_cast<const int*>(flags) + 8 * x);
      const int4 fa = f4[0], fb = f4[1];
      const bool split = (fa.x | fa.y | fa.z | fa.w | fb.x | fb.y | fb.z | fb.w) != 0;
      const uint32_t first = j > 0 ? 1u : 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        tc_mma_ts_w(tO, tP + 16 * k, desc_add(vd, 2048 * k), idO, k > 0 ? 1u : first);
      if (split) {
#pragma unroll
        for (int k = 0; k < 8; ++k) tc_mma_ts_w(tO, tP + 16 * k + 8, desc_add(vd, 2048 * k), idO, 1u);
      }
      tc_commit_w(bar(C::bODone + x));
    };
    if (ok) ok = warp_wait<kIssuerPoll>(bar(C::bKFull), 0, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      issue_s(0, 0);
      if (lastB >= 0) issue_s(1, 0);
      tc_commit_w(bar(C::bKEmpty));  // K_0 read by both S MMAs
    }
    for (int j = 0; ok && j < nblk; ++j) {
      const int sv = j % C::kNV;
      // K_{j+1} for the next S MMAs
      const bool nextA = j + 1 <= lastA, nextB = j + 1 <= lastB;
      if (!warp_wait<kIssuerPoll>(bar(C::bVFull + sv), (j / C::kNV) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      if (nextA || nextB) {
        const int sk = (j + 1) % C::kNK;
        if (!warp_wait<kIssuerPoll>(bar(C::bKFull + sk), ((j + 1) / C::kNK) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
      }
      if (j <= lastA) {
        if (!warp_wait<kIssuerPoll>(bar(C::bPFull + 0), j & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_o(0, j);
        if (nextA) issue_s(0, j + 1);
      }
      if (j <= lastB) {
        if (!warp_wait<kIssuerPoll>(bar(C::bPFull + 1), j & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_o(1, j);
        if (nextB) issue_s(1, j + 1);
      }
      tc_commit_w(bar(C::bVEmpty + sv));                               // V_j read by both O MMAs
      if (nextA || nextB) tc_commit_w(bar(C::bKEmpty + (j + 1) % C::kNK));  // K_{j+1} read by the S MMAs
    }
    // Every MMA this warp issued is complete before the CTA frees TMEM and exits.
    tc_commit_w(bar(C::bDrain));
    if (lane == 0) mbar_wait_drain(bar(C::bDrain), 0, p.status);
    __syncwarp();
  } else {
    // ------------------------------ softmax warps ------------------------------
    // warps 2-17; a warp reaches TMEM lanes 32 (warp % 4) .. + 31
    const int x = (warp - 2) >> 3;         // tile
    const int half = ((warp - 2) >> 2) & 1;  // keys [64 half, 64 half + 64) of a block
    const int wq = warp & 3;
    const int il = wq * 32 + lane;  // row in the tile, TMEM lane
    const int i = q0 + 128 * x + il;
    const int last = x ? lastB : lastA;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + 128 * x + 64 * half;          // this warp's 64 S columns
    const uint32_t tO = tmem + lane_off + 256 + D * x + (D / 2) * half;  // and D/2 O columns
    float* xchg = reinterpret_cast<float*>(smem + C::oXchg);
    const int pq = 4 * x + wq;  // the two warps holding rows 32 wq .. 32 wq + 31 of tile x
    const float c2 = p.scale_log2;
    float mref = -INFINITY, lsum = 0.f;  // lsum: this half's part of the row sum
    bool ok = true;
    // Waits block (the hardware suspends the warp): each tile's warps idle about
    // half the time, and spinning would take issue slots from the other tile's
    // warps on the same scheduler.
    for (int j = 0; j <= last; ++j) {
      if (!warp_wait<false>(bar(C::bSFull + x), j & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // keys 128 j + 64 half .. + 63 of this warp; the allowed ones are those
      // below the diagonal and the unit's end (with packed input the keys past
      // the end belong to the next sequence): local columns 0 .. hi - 1.
      const int kb = 128 * j + 64 * half;
      const int hi = min(Nl, p.causal ? i + 1 : Nl) - kb;
      // Pass 1: this half's maximum of S over the allowed keys.
      float hmax = -INFINITY;
      {
        uint32_t s0[32], s1[32];
        tmem_ld32(tS, s0);
        tmem_ld32(tS + 32, s1);
        tmem_ld_wait2(s0, s1);
        if (hi >= 64) {
          float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            m0 = fmax3(m0, __uint_as_float(s0[e]), __uint_as_float(s0[e + 1]));
            m1 = fmax3(m1, __uint_as_float(s1[e]), __uint_as_float(s1[e + 1]));
          }
          hmax = fmaxf(m0, m1);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            hmax = (e < hi) ? fmaxf(hmax, __uint_as_float(s0[e])) : hmax;
            hmax = (32 + e < hi) ? fmaxf(hmax, __uint_as_float(s1[e])) : hmax;
          }
        }
      }
      // The block maximum of the row: this half's and the other warp's (slots
      // alternate with the block parity, so a slot is rewritten only after the
      // partner has passed the next exchange, i.e. has read it).
      float* xs = xchg + ((x * 2 + (j & 1)) * 2) * 128;
      xs[half * 128 + il] = hmax;
      warp_arrive(bar(C::bXchg + 2 * pq + (j & 1)));
      if (!warp_wait<false>(bar(C::bXchg + 2 * pq + (j & 1)), (j >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const float bmax = fmaxf(hmax, xs[(half ^ 1) * 128 + il]) * c2;  // scale > 0 on this path
      // Lazy rescale: the reference moves when the block maximum exceeds it by
      // more than 2^8 (always on the first block: every processed block holds an
      // allowed key for every row, so the reference is finite from then on).
      // Both warps of a row take the same decision; each rescales its D/2 O columns.
      const bool mv = bmax > mref + kFwdRescaleLog2;
      const float alpha = mv ? ex2_approx(mref - bmax) : 1.f;  // 0 when mref = -inf
      // (warp-wide decision: the wait and the TMEM accesses below are collective)
      if (j > 0 && __any_sync(0xffffffffu, mv && mref != -INFINITY)) {
        // this tile's O MMA of block j-1 is done before its rows are rescaled
        if (!warp_wait<false>(bar(C::bODone + x), (j - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          uint32_t r[32];
          tmem_ld32(tO + 32 * cc, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(tO + 32 * cc, r);
        }
      }
      if (mv) {
        lsum *= alpha;
        mref = bmax;
      }
      // Pass 2, 32 keys at a time: P = exp2(S * scale * log2e - mref) (0 where
      // masked), this half's running sum, and the 16-bit image of the two MMA K
      // steps over the same columns. A chunk writes residual columns where the
      // block's largest probability may exceed 1/64 of this half's sum so far (a
      // part of the final row sum, so the bound holds for the final P); zeros
      // otherwise.
      const uint64_t cc2 = f2_pack(c2, c2), nm2 = f2_pack(-mref, -mref);
      // the largest P of this block for this row (its block maximum against the reference)
      const float pmax = ex2_approx(bmax - mref);
      bool split = false;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t cur[32];
        __syncwarp();
        tmem_ld32(tS + 32 * q, cur);
        tmem_ld_wait(cur);
        uint64_t sum2 = f2_pack(0.f, 0.f);
        if (hi >= 64) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float p0, p1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(cur[e]), __uint_as_float(cur[e + 1])), cc2, nm2), p0, p1);
            p0 = ex2_approx(p0);
            p1 = ex2_approx(p1);
            sum2 = f2_add(sum2, f2_pack(p0, p1));
            cur[e] = __float_as_uint(p0);
            cur[e + 1] = __float_as_uint(p1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float p0, p1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(cur[e]), __uint_as_float(cur[e + 1])), cc2, nm2), p0, p1);
            p0 = (32 * q + e < hi) ? ex2_approx(p0) : 0.f;
            p1 = (32 * q + e + 1 < hi) ? ex2_approx(p1) : 0.f;
            sum2 = f2_add(sum2, f2_pack(p0, p1));
            cur[e] = __float_as_uint(p0);
            cur[e + 1] = __float_as_uint(p1);
          }
        }
        __syncwarp();
        float s0, s1;
        f2_unpack(sum2, s0, s1);
        lsum += s0 + s1;
        const bool sp = __any_sync(0xffffffffu, pmax > kSplitThreshold * lsum);
        split |= sp;
        // (sp is warp-uniform: a real branch, the residuals are computed only when needed)
        if (sp) {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t w[16];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float a = __uint_as_float(cur[16 * k + 2 * t]), c = __uint_as_float(cur[16 * k + 2 * t + 1]);
              w[t] = pack2<kBf16>(a, c);
              w[8 + t] = pack2_residual<kBf16>(a, c, w[t]);
            }
            tmem_st16(tS + 32 * q + 16 * k, w);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t w[16];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              w[t] = pack2<kBf16>(__uint_as_float(cur[16 * k + 2 * t]), __uint_as_float(cur[16 * k + 2 * t + 1]));
              w[8 + t] = 0u;
            }
            tmem_st16(tS + 32 * q + 16 * k, w);
          }
        }
      }
      tmem_st_wait();
      if (lane == 0) flags[8 * x + 4 * half + wq] = split ? 1 : 0;
      tc_fence_before();
      warp_arrive(bar(C::bPFull + x));
    }
    // Epilogue: the row sum of both halves; O = O / l (bf16/fp16), this warp's
    // D/2 columns; L = (mref + log2 l) * ln 2, written by the first half's warp.
    if (ok && last >= 0) {
      float* xl = xchg + 8 * 128 + (x * 2) * 128;
      xl[half * 128 + il] = lsum;
      warp_arrive(bar(C::bSum + pq));
      ok = warp_wait<false>(bar(C::bSum + pq), 0, abort_flag, p.status);
      const float ltot = lsum + xl[(half ^ 1) * 128 + il];
      if (ok) ok = warp_wait<false>(bar(C::bODone + x), last & 1, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
        uint16_t* dst = static_cast<uint16_t*>(p.out) + (long long)b * p.sb + (long long)(u.row0 + i) * p.sn +
                        (long long)h * p.sh + (D / 2) * half;
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          uint32_t r[32];
          tmem_ld32(tO + 32 * cc, r);
          tmem_ld_wait(r);
          uint32_t w[16];
#pragma unroll
          for (int t = 0; t < 16; ++t)
            w[t] = pack2<kBf16>(__uint_as_float(r[2 * t]) * inv, __uint_as_float(r[2 * t + 1]) * inv);
          if (i < Nl) {
            uint4* g = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
            for (int t = 0; t < 4; ++t) g[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
          }
        }
        if (half == 0 && i < Nl)
          p.lse_out[u.lse + i] = ltot > 0.f ? (mref + lg2_fwd(ltot)) * 0.6931471805599453f : -INFINITY;
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

template <int D, bool kBf16>
static cudaError_t launch_fwd_t(const AttnParams& p, const CUtensorMap* maps, cudaStream_t st) {
  using C = FwdCfg<D>;
  auto kern = fwd_pingpong_kernel<D, kBf16>;
  const int smem = (int)(C::kSmem > kMinSmemOneCtaPerSm ? C::kSmem : kMinSmemOneCtaPerSm);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rows = p.cu_seqlens ? p.max_seqlen : p.N;
  const long long grid = (long long)((rows + kFwdRows - 1) / kFwdRows) * (p.cu_seqlens ? p.nseq * p.H : p.B * p.H);
  kern<<<(unsigned)grid, kFwdThreads, smem, st>>>(p, maps[0], maps[1], maps[2]);
  return cudaGetLastError();
}

// Whether the ping-pong forward serves these parameters: 16-bit inputs with d
// in {64, 128} (fixed-length or packed), a positive scale, no dropout, ALiBi,
// attention bias or window, and a grid that fits.
bool fwd_pingpong_supported(const AttnParams& p) {
  const int rows = p.cu_seqlens ? p.max_seqlen : p.N;
  return (p.d == 64 || p.d == 128) && p.drop.on == 0 && p.alibi == nullptr && p.bias == nullptr && p.window == 0 &&
         p.scale > 0.f &&
         (long long)((rows + kFwdRows - 1) / kFwdRows) * (p.cu_seqlens ? p.nseq * p.H : p.B * p.H) <= 0x7fffffffll;
}

// maps: Q, K, V with boxes of 128 rows x 64 elements (128-byte swizzle).
cudaError_t launch_fwd_pingpong(const AttnParams& p, bool bf16, const CUtensorMap* maps, cudaStream_t st) {
  if (p.d == 128) return bf16 ? launch_fwd_t<128, true>(p, maps, st) : launch_fwd_t<128, false>(p, maps, st);
  return bf16 ? launch_fwd_t<64, true>(p, maps, st) : launch_fwd_t<64, false>(p, maps, st);
}

}  // namespace fa
