// Bandwidth-bound helpers of the backward pass and the CUDA-core fp32 path.
//
// * preprocess: D_i = rowsum(dO o O) in fp32 ("FlashAttention backward",
//   §The gradients, and the one scalar that makes them local: one cheap pass
//   over dO and O before the main loop), stored negated, plus -L*log2(e) into
//   a padded workspace vector and, in the atomic and ordered dQ modes, the zero
//   fill of the fp32 dQ accumulator (and, ordered, of the chunk counters and
//   the unit ticket). Both vectors are kept negated so that the consumers
//   use them as addends (S*scale*log2e + (-L*log2e) is one FMA, dP + (-D) one
//   add, also in packed two-wide form).
// * dq_convert: dQ = scale * dQ_accum, rounded to the tensor dtype (atomic mode).
// * fp32 kernels: forward (two passes: row statistics, then O) and the
//   key-major dK/dV plus query-major dQ kernels of the backward, on CUDA cores.
//   fp32 needs ~1e-7 relative accuracy, which the tf32 tensor-core kind cannot
//   give, so this path multiplies in FFMA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;

// -L * log2(e) for the backward's exp2 addend. A row with no finite score
// (L = -inf, possible only when an attention bias masks every key) gets -inf,
// not +inf, so that its probabilities come out 0 even where a biased score is
// -inf (-inf + inf would be NaN).
__device__ __forceinline__ float neg_l2(float L) { return L == -INFINITY ? L : -(L * kLog2e); }
constexpr float kLn2 = 0.6931471805599453f;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per (b, i, h) row; rows enumerated in [B, n_pad, H] order so that a
// contiguous [B, N, H, d] tensor is read front to back. The row index and its
// decomposition are 64-bit and the warps stride over the rows, so that any
// B * H * n_pad the size limits admit is covered (a 32-bit row index would
// wrap once B * H * n_pad passes 2^27 rows at 8 warps a block).
template <typename T>
__global__ void __launch_bounds__(256) preprocess_kernel(const __grid_constant__ AttnParams p) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.B * p.n_pad * p.H;
  const long long stride = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += stride) {
    const long long bi = row / p.H;              // b * n_pad + i
    const int h = (int)(row - bi * p.H);
    const long long b = bi / p.n_pad;
    const int i = (int)(bi - b * p.n_pad);
    const long long bh = b * p.H + h;
    const long long ws = bh * p.n_pad + i;
    float acc = 0.f;
    if (i < p.N) {
      const long long off = b * p.sb + (long long)i * p.sn + (long long)h * p.sh;
      const T* o = static_cast<const T*>(p.o) + off;
      const T* g = static_cast<const T*>(p.dout) + off;
      if (sizeof(T) == 2 && (p.d & 63) == 0) {
        // 16-bit types, d in {64, 128}: lanes read 2 or 4 contiguous elements.
        const int per = p.d >> 5;
        for (int e = 0; e < per; e += 2) {
          const int k = lane * per + e;
          const uint32_t ow = *reinterpret_cast<const uint32_t*>(o + k);
          const uint32_t gw = *reinterpret_cast<const uint32_t*>(g + k);
          const T* o2 = reinterpret_cast<const T*>(&ow);
          const T* g2 = reinterpret_cast<const T*>(&gw);
          acc = fmaf(to_f32(o2[0]), to_f32(g2[0]), acc);
          acc = fmaf(to_f32(o2[1]), to_f32(g2[1]), acc);
        }
      } else {
        for (int k = lane; k < p.d; k += 32) acc = fmaf(to_f32(o[k]), to_f32(g[k]), acc);
      }
      acc = warp_sum(acc);
    }
    if (lane == 0) {
      p.ws_nD[ws] = -acc;
      p.ws_nL2[ws] = (i < p.N) ? neg_l2(p.lse[bh * p.N + i]) : __int_as_float(0xff800000);
      // ordered dQ: the contribution counter of each 32-row chunk and the unit ticket start at 0
      if (p.dq_flags != nullptr && (i & 31) == 0) p.dq_flags[bh * (p.n_pad / 32) + i / 32] = 0u;
      if (p.dq_ticket != nullptr && row == 0) *p.dq_ticket = 0u;
    }
    if (p.ws_dq != nullptr) {
      float* dq = p.ws_dq + ws * p.d;
      for (int k = lane; k < p.d; k += 32) dq[k] = 0.f;
    }
  }
}

// 16-bit tensors with d in {64, 128}: a group of d/8 lanes owns one row and
// each lane reads 16 bytes of O and of dO, so a warp moves whole 128-byte lines.
// Rows are enumerated in [B*H, n_pad] order (positions fastest), which keeps
// the workspace vectors and L contiguous (measured faster than streaming the
// [B, N, H, d] tensors front to back); every thread takes kVecRows rows and
// issues all of their loads before reducing, to keep enough bytes in flight.
constexpr int kVecRows = 4;

// Rows of one (batch, head) per block: 8 warps x (32 / (d/8)) rows x kVecRows.
template <int D>
constexpr int vec_block_rows() { return 8 * (32 / (D / 8)) * kVecRows; }

template <int D>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = D / 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T>
__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const T* a2 = reinterpret_cast<const T*>(&aw[x]);
    const T* b2 = reinterpret_cast<const T*>(&bw[x]);
    acc = fmaf(to_f32(a2[0]), to_f32(b2[0]), acc);
    acc = fmaf(to_f32(a2[1]), to_f32(b2[1]), acc);
  }
  return acc;
}

// Grid: x = block of vec_block_rows<D>() positions, y = batch * head.
template <typename T, int D>
__global__ void __launch_bounds__(256) preprocess_vec_kernel(const __grid_constant__ AttnParams p) {
  constexpr int G = D / 8;            // lanes per row
  constexpr int kRowsPerWarp = 32 / G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ib = blockIdx.x * vec_block_rows<D>() + warp * (kRowsPerWarp * kVecRows) + lane / G;
  const int e0 = (lane % G) * 8;
  // y = batch * head, or sequence * head for packed variable-length input; rows
  // below are local to it (n of them, padded to `pad` workspace rows).
  int bh, row0 = 0, n = p.N, pad = p.n_pad;
  long long ws0, lse0;
  if (p.cu_seqlens == nullptr) {
    bh = blockIdx.y;
    ws0 = (long long)bh * p.n_pad;
    lse0 = (long long)bh * p.N;
  } else {
    const int sq = blockIdx.y / p.H, h = blockIdx.y % p.H;
    const int s0 = min(max(p.cu_seqlens[sq], 0), p.N), s1 = min(max(p.cu_seqlens[sq + 1], s0), p.N);
    bh = h;  // B = 1
    row0 = s0;
    n = min(s1 - s0, p.max_seqlen);
    pad = p.seq_pad;
    ws0 = ((long long)h * p.nseq + sq) * p.seq_pad;
    lse0 = (long long)h * p.N + s0;
  }
  const T* o = static_cast<const T*>(p.o) + (long long)(bh / p.H) * p.sb + (long long)(bh % p.H) * p.sh +
               (long long)row0 * p.sn + e0;
  const T* g = static_cast<const T*>(p.dout) + (o - static_cast<const T*>(p.o));
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    if (p.dq_ticket != nullptr) *p.dq_ticket = 0u;
    if (p.unit_ctr != nullptr)
      for (int x = 0; x < 4; ++x) p.unit_ctr[x] = 0u;
  }
  uint4 ov[kVecRows], gv[kVecRows];
#pragma unroll
  for (int r = 0; r < kVecRows; ++r) {
    const int i = ib + r * kRowsPerWarp;
    ov[r] = gv[r] = make_uint4(0u, 0u, 0u, 0u);
    if (i < n) {
      ov[r] = __ldg(reinterpret_cast<const uint4*>(o + (long long)i * p.sn));
      gv[r] = __ldg(reinterpret_cast<const uint4*>(g + (long long)i * p.sn));
    }
  }
#pragma unroll
  for (int r = 0; r < kVecRows; ++r) {
    const int i = ib + r * kRowsPerWarp;
    const float acc = group_sum<D>(dot8<T>(ov[r], gv[r], 0.f));
    if (i >= pad) continue;
    if (e0 == 0) {
      p.ws_nD[ws0 + i] = -acc;
      p.ws_nL2[ws0 + i] = (i < n) ? neg_l2(p.lse[lse0 + i]) : __int_as_float(0xff800000);
      // ordered dQ: the contribution counter of each 32-row chunk starts at 0
      if (p.dq_flags != nullptr && (i & 31) == 0) p.dq_flags[(long long)blockIdx.y * (pad / 32) + i / 32] = 0u;
    }
    // (packed input: the dQ accumulator is zeroed separately)
    if (p.ws_dq != nullptr && p.cu_seqlens == nullptr) {
      float4* dq = reinterpret_cast<float4*>(p.ws_dq + (ws0 + i) * D + e0);
      dq[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      dq[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// dQ = scale * dQ_accum for 16-bit outputs with d in {64, 128}, eight elements a
// lane; the grid is laid out as for preprocess_vec_kernel.
template <typename T, int D>
__global__ void __launch_bounds__(256) dq_convert_vec_kernel(const __grid_constant__ AttnParams p) {
  constexpr int G = D / 8;
  constexpr int kRowsPerWarp = 32 / G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int bh = blockIdx.y;
  const int ib = blockIdx.x * vec_block_rows<D>() + warp * (kRowsPerWarp * kVecRows) + lane / G;
  const int e0 = (lane % G) * 8;
  const float* src = p.ws_dq + (long long)bh * p.n_pad * D + e0;
  T* dst = static_cast<T*>(p.out) + (long long)(bh / p.H) * p.sb + (long long)(bh % p.H) * p.sh + e0;
  float4 a[kVecRows], c[kVecRows];
#pragma unroll
  for (int r = 0; r < kVecRows; ++r) {
    const int i = ib + r * kRowsPerWarp;
    if (i < p.N) {
      const float4* s4 = reinterpret_cast<const float4*>(src + (long long)i * D);
      a[r] = __ldg(s4);
      c[r] = __ldg(s4 + 1);
    }
  }
#pragma unroll
  for (int r = 0; r < kVecRows; ++r) {
    const int i = ib + r * kRowsPerWarp;
    if (i >= p.N) continue;
    const float v[8] = {a[r].x, a[r].y, a[r].z, a[r].w, c[r].x, c[r].y, c[r].z, c[r].w};
    uint32_t w[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const T lo = from_f32<T>(v[2 * x] * p.scale), hi = from_f32<T>(v[2 * x + 1] * p.scale);
      w[x] = (uint32_t)(*reinterpret_cast<const uint16_t*>(&lo)) |
             ((uint32_t)(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
    }
    *reinterpret_cast<uint4*>(dst + (long long)i * p.sn) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The general case (other dtypes or head dimensions): one warp per (b, i, h)
// row, 64-bit row index, warps striding over the rows as in preprocess_kernel.
template <typename T>
__global__ void __launch_bounds__(256) dq_convert_kernel(const __grid_constant__ AttnParams p) {
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.B * p.N * p.H;
  const long long stride = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += stride) {
    const long long bi = row / p.H;              // b * N + i
    const int h = (int)(row - bi * p.H);
    const long long b = bi / p.N;
    const int i = (int)(bi - b * p.N);
    const float* src = p.ws_dq + ((b * p.H + h) * p.n_pad + i) * p.d;
    T* dst = static_cast<T*>(p.out) + b * p.sb + (long long)i * p.sn + (long long)h * p.sh;
    for (int k = lane; k < p.d; k += 32) dst[k] = from_f32<T>(src[k] * p.scale);
  }
}

// ------------------------------- fp32 path ---------------------------------
constexpr int kF32Warps = 4;  // rows per block (one warp each)

__device__ __forceinline__ const float* row_ptr(const AttnParams& p, const void* base, int b, int i, int h) {
  return static_cast<const float*>(base) + (long long)b * p.sb + (long long)i * p.sn + (long long)h * p.sh;
}

__device__ __forceinline__ float dot_row(const float* __restrict__ a_smem, const float* __restrict__ g, int d) {
  float acc = 0.f;
  for (int k = 0; k < d; ++k) acc = fmaf(a_smem[k], g[k], acc);
  return acc;
}

// ALiBi slope of (batch b, head h) in the log2 domain (0 without ALiBi): the
// score of (i, j) gains -m * |i - j| after the scale.
__device__ __forceinline__ float alibi_slope_log2(const AttnParams& p, int b, int h) {
  return p.alibi ? __ldg(p.alibi + (long long)b * p.alibi_sb + h) * kLog2e : 0.f;
}

// Attention bias of (query i, key j) in the log2 domain (0 without a bias).
__device__ __forceinline__ float bias_log2_f32(const AttnParams& p, int b, int h, int i, int j) {
  if (!p.bias) return 0.f;
  const float* row = static_cast<const float*>(p.bias) + (long long)b * p.bias_sb + (long long)h * p.bias_sh +
                     (long long)i * p.bias_sn;
  return __ldg(row + j) * kLog2e;
}

// Forward, one warp per query row: pass 1 row max and sum of exp2 (lanes take
// keys lane, lane+32, ...), pass 2 O = sum_j P~_ij V_j with lanes owning head
// dimensions and P broadcast by shuffles.
__global__ void __launch_bounds__(32 * kF32Warps) fwd_f32_kernel(const __grid_constant__ AttnParams p) {
  __shared__ float qrow[kF32Warps][128];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kF32Warps + w;
  if (row >= (long long)p.B * p.H * p.N) return;
  const int i = row % p.N, bh = row / p.N, b = bh / p.H, h = bh % p.H;
  const float* q = row_ptr(p, p.q, b, i, h);
  for (int k = lane; k < p.d; k += 32) qrow[w][k] = q[k];
  __syncwarp();
  const int jlo = p.window > 0 ? max(0, i - p.window + 1) : 0;
  const int jhi = p.causal ? i : p.N - 1;
  const float am = alibi_slope_log2(p, b, h);
  float m = -INFINITY, l = 0.f;
  for (int j = jlo + lane; j <= jhi; j += 32) {
    const float x = fmaf(-am, fabsf((float)(i - j)), dot_row(qrow[w], row_ptr(p, p.k, b, j, h), p.d) * p.scale_log2) +
                    bias_log2_f32(p, b, h, i, j);
    if (x == -INFINITY) continue;  // a pair the bias masks out
    const float mn = fmaxf(m, x);
    l = l * ex2_approx(m - mn) + ex2_approx(x - mn);
    m = mn;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, o), lo = __shfl_xor_sync(0xffffffffu, l, o);
    const float mn = fmaxf(m, mo);
    if (mn == -INFINITY) continue;
    l = l * ex2_approx(m - mn) + lo * ex2_approx(mo - mn);
    m = mn;
  }
  const bool live = l > 0.f;
  float lg;
  asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(live ? l : 1.f));
  const float L2 = live ? m + lg : __int_as_float(0x7f800000);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int jb = jlo; jb <= jhi; jb += 32) {
    const int j = jb + lane;
    float pj = 0.f;
    if (j <= jhi) {
      pj = ex2_approx(fmaf(-am, fabsf((float)(i - j)), dot_row(qrow[w], row_ptr(p, p.k, b, j, h), p.d) * p.scale_log2) +
                      bias_log2_f32(p, b, h, i, j) - L2);
      if (p.drop.on) pj = dropout_keep(p.drop, bh, p.N, i, j) ? pj * p.drop.rp : 0.f;
    }
    const int cnt = min(32, jhi - jb + 1);
    for (int t = 0; t < cnt; ++t) {
      const float pb = __shfl_sync(0xffffffffu, pj, t);
      const float* vr = row_ptr(p, p.v, b, jb + t, h);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = lane + 32 * u;
        if (k < p.d) acc[u] = fmaf(pb, vr[k], acc[u]);
      }
    }
  }
  float* o = static_cast<float*>(p.out) + (long long)b * p.sb + (long long)i * p.sn + (long long)h * p.sh;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int k = lane + 32 * u;
    if (k < p.d) o[k] = acc[u];
  }
  if (lane == 0) p.lse_out[(long long)bh * p.N + i] = live ? L2 * kLn2 : -INFINITY;
}

// dK, dV, one warp per key row j: lanes take queries, the per-pair P~ and dS
// are broadcast by shuffles and accumulated into lane-owned head dimensions.
__global__ void __launch_bounds__(32 * kF32Warps) bwd_dkdv_f32_kernel(const __grid_constant__ AttnParams p) {
  __shared__ float krow[kF32Warps][128];
  __shared__ float vrow[kF32Warps][128];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kF32Warps + w;
  if (row >= (long long)p.B * p.H * p.N) return;
  const int j = row % p.N, bh = row / p.N, b = bh / p.H, h = bh % p.H;
  const float* kk = row_ptr(p, p.k, b, j, h);
  const float* vv = row_ptr(p, p.v, b, j, h);
  for (int k = lane; k < p.d; k += 32) {
    krow[w][k] = kk[k];
    vrow[w][k] = vv[k];
  }
  __syncwarp();
  const int ilo = p.causal ? j : 0;
  const int ihi = p.window > 0 ? min(p.N - 1, j + p.window - 1) : p.N - 1;
  const float* nL2 = p.ws_nL2 + (long long)bh * p.n_pad;
  const float* nD = p.ws_nD + (long long)bh * p.n_pad;
  const float am = alibi_slope_log2(p, b, h);
  float dk[4] = {0.f, 0.f, 0.f, 0.f}, dv[4] = {0.f, 0.f, 0.f, 0.f};
  for (int ib = ilo; ib <= ihi; ib += 32) {
    const int i = ib + lane;
    float pt = 0.f, ds = 0.f;
    if (i <= ihi) {
      const float pv = ex2_approx(
          fmaf(-am, fabsf((float)(i - j)), dot_row(krow[w], row_ptr(p, p.q, b, i, h), p.d) * p.scale_log2) +
          bias_log2_f32(p, b, h, i, j) + nL2[i]);
      float dp = dot_row(vrow[w], row_ptr(p, p.dout, b, i, h), p.d);
      pt = pv;
      if (p.drop.on) {
        const bool keep = dropout_keep(p.drop, bh, p.N, i, j);
        pt = keep ? pv * p.drop.rp : 0.f;
        dp = keep ? dp * p.drop.rp : 0.f;
      }
      ds = pv * (dp + nD[i]);
    }
    const int cnt = min(32, ihi - ib + 1);
    for (int t = 0; t < cnt; ++t) {
      const float pb = __shfl_sync(0xffffffffu, pt, t), sb = __shfl_sync(0xffffffffu, ds, t);
      const float* qr = row_ptr(p, p.q, b, ib + t, h);
      const float* gr = row_ptr(p, p.dout, b, ib + t, h);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = lane + 32 * u;
        if (k < p.d) {
          dv[u] = fmaf(pb, gr[k], dv[u]);
          dk[u] = fmaf(sb, qr[k], dk[u]);
        }
      }
    }
  }
  const long long off = (long long)b * p.sb + (long long)j * p.sn + (long long)h * p.sh;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int k = lane + 32 * u;
    if (k < p.d) {
      static_cast<float*>(p.dk)[off + k] = dk[u] * p.scale;
      static_cast<float*>(p.dv)[off + k] = dv[u];
    }
  }
}

// dQ, one warp per query row i (query-major: deterministic, no atomics).
__global__ void __launch_bounds__(32 * kF32Warps) bwd_dq_f32_kernel(const __grid_constant__ AttnParams p) {
  __shared__ float qrow[kF32Warps][128];
  __shared__ float grow[kF32Warps][128];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kF32Warps + w;
  if (row >= (long long)p.B * p.H * p.N) return;
  const int i = row % p.N, bh = row / p.N, b = bh / p.H, h = bh % p.H;
  const float* q = row_ptr(p, p.q, b, i, h);
  const float* g = row_ptr(p, p.dout, b, i, h);
  for (int k = lane; k < p.d; k += 32) {
    qrow[w][k] = q[k];
    grow[w][k] = g[k];
  }
  __syncwarp();
  const int jlo = p.window > 0 ? max(0, i - p.window + 1) : 0;
  const int jhi = p.causal ? i : p.N - 1;
  const float nL2 = p.ws_nL2[(long long)bh * p.n_pad + i];
  const float nD = p.ws_nD[(long long)bh * p.n_pad + i];
  const float am = alibi_slope_log2(p, b, h);
  float dq[4] = {0.f, 0.f, 0.f, 0.f};
  for (int jb = jlo; jb <= jhi; jb += 32) {
    const int j = jb + lane;
    float ds = 0.f;
    if (j <= jhi) {
      const float pv = ex2_approx(
          fmaf(-am, fabsf((float)(i - j)), dot_row(qrow[w], row_ptr(p, p.k, b, j, h), p.d) * p.scale_log2) +
          bias_log2_f32(p, b, h, i, j) + nL2);
      float dp = dot_row(grow[w], row_ptr(p, p.v, b, j, h), p.d);
      if (p.drop.on) dp = dropout_keep(p.drop, bh, p.N, i, j) ? dp * p.drop.rp : 0.f;
      ds = pv * (dp + nD);
    }
    const int cnt = min(32, jhi - jb + 1);
    for (int t = 0; t < cnt; ++t) {
      const float sb = __shfl_sync(0xffffffffu, ds, t);
      const float* kr = row_ptr(p, p.k, b, jb + t, h);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = lane + 32 * u;
        if (k < p.d) dq[u] = fmaf(sb, kr[k], dq[u]);
      }
    }
  }
  float* o = static_cast<float*>(p.out) + (long long)b * p.sb + (long long)i * p.sn + (long long)h * p.sh;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int k = lane + 32 * u;
    if (k < p.d) o[k] = dq[u] * p.scale;
  }
}

// ------------------------------- launchers ---------------------------------
// Grid of a row-striding kernel: enough blocks to cover the rows, at most 2^20
// (the kernel's warps stride over the rest).
static inline unsigned grid_for_rows_strided(long long rows, int rows_per_block) {
  const long long g = (rows + rows_per_block - 1) / rows_per_block;
  return (unsigned)(g < (1ll << 20) ? (g > 0 ? g : 1) : (1ll << 20));
}

cudaError_t launch_preprocess(const AttnParams& p, int dtype, cudaStream_t st) {
  const long long rows = (long long)p.B * p.n_pad * p.H;
  // packed variable-length input: y = sequence * head, x over seq_pad rows
  const int prow = p.cu_seqlens ? p.seq_pad : p.n_pad;
  const int units = p.cu_seqlens ? p.nseq * p.H : p.B * p.H;
  if (dtype != 0 && (p.d == 64 || p.d == 128) && units <= 65535) {
    const dim3 g((unsigned)((prow + vec_block_rows<128>() - 1) / vec_block_rows<128>()), (unsigned)units);
    const dim3 g64((unsigned)((prow + vec_block_rows<64>() - 1) / vec_block_rows<64>()), (unsigned)units);
    if (p.d == 128)
      dtype == 1 ? preprocess_vec_kernel<__half, 128><<<g, 256, 0, st>>>(p)
                 : preprocess_vec_kernel<__nv_bfloat16, 128><<<g, 256, 0, st>>>(p);
    else
      dtype == 1 ? preprocess_vec_kernel<__half, 64><<<g64, 256, 0, st>>>(p)
                 : preprocess_vec_kernel<__nv_bfloat16, 64><<<g64, 256, 0, st>>>(p);
    return cudaGetLastError();
  }
  const unsigned grid = grid_for_rows_strided(rows, 8);
  if (dtype == 0) preprocess_kernel<float><<<grid, 256, 0, st>>>(p);
  else if (dtype == 1) preprocess_kernel<__half><<<grid, 256, 0, st>>>(p);
  else preprocess_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const AttnParams& p, int dtype, cudaStream_t st) {
  if (dtype != 0 && (p.d == 64 || p.d == 128) && p.B * p.H <= 65535) {
    const dim3 g((unsigned)((p.n_pad + vec_block_rows<128>() - 1) / vec_block_rows<128>()), (unsigned)(p.B * p.H));
    const dim3 g64((unsigned)((p.n_pad + vec_block_rows<64>() - 1) / vec_block_rows<64>()), (unsigned)(p.B * p.H));
    if (p.d == 128)
      dtype == 1 ? dq_convert_vec_kernel<__half, 128><<<g, 256, 0, st>>>(p)
                 : dq_convert_vec_kernel<__nv_bfloat16, 128><<<g, 256, 0, st>>>(p);
    else
      dtype == 1 ? dq_convert_vec_kernel<__half, 64><<<g64, 256, 0, st>>>(p)
                 : dq_convert_vec_kernel<__nv_bfloat16, 64><<<g64, 256, 0, st>>>(p);
    return cudaGetLastError();
  }
  const long long rows = (long long)p.B * p.N * p.H;
  const unsigned grid = grid_for_rows_strided(rows, 8);
  if (dtype == 0) dq_convert_kernel<float><<<grid, 256, 0, st>>>(p);
  else if (dtype == 1) dq_convert_kernel<__half><<<grid, 256, 0, st>>>(p);
  else dq_convert_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_f32(const AttnParams& p, cudaStream_t st) {
  const long long blocks = ((long long)p.B * p.H * p.N + kF32Warps - 1) / kF32Warps;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;  // one warp per row: the grid must fit
  const unsigned grid = (unsigned)blocks;
  fwd_f32_kernel<<<grid, 32 * kF32Warps, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv_f32(const AttnParams& p, cudaStream_t st) {
  const long long blocks = ((long long)p.B * p.H * p.N + kF32Warps - 1) / kF32Warps;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;  // one warp per row: the grid must fit
  const unsigned grid = (unsigned)blocks;
  bwd_dkdv_f32_kernel<<<grid, 32 * kF32Warps, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_f32(const AttnParams& p, cudaStream_t st) {
  const long long blocks = ((long long)p.B * p.H * p.N + kF32Warps - 1) / kF32Warps;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;  // one warp per row: the grid must fit
  const unsigned grid = (unsigned)blocks;
  bwd_dq_f32_kernel<<<grid, 32 * kF32Warps, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
