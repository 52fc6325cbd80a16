// Parameters passed by value from the C-ABI layer to the kernels.
#pragma once

#include <stdint.h>

#include <type_traits>

#include "device_common.cuh"

namespace fa {

// Tile geometry of the tensor-core kernels.
constexpr int kRowsKV = 128;    // keys per CTA in the key/value-major kernel (TMEM lanes)
constexpr int kStepQ = 64;      // queries per inner step of that kernel
constexpr int kRowsQ = 128;     // queries per CTA in the query-major kernels (TMEM lanes)
constexpr int kStepKV = 128;    // keys per inner step of those kernels
constexpr int kPadRows = 128;   // per-head row padding of the L / D workspace vectors
// Every tensor-core CTA allocates all 512 TMEM columns; requesting more than half
// of the SM's shared memory keeps it alone on its SM.
constexpr unsigned kMinSmemOneCtaPerSm = 120u * 1024u;

struct AttnParams {
  int B, H, N, d;
  int64_t sb, sn, sh;     // element strides of every [B, N, H, d] tensor (d stride is 1)
  int n_pad;              // N rounded up to kPadRows
  float scale;            // softmax scale applied to Q.K
  float scale_log2;       // scale * log2(e)
  int causal;             // keep j <= i
  int window;             // > 0: keep j > i - window
  DropoutParams drop;
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;       // [B, H, N] natural-log log-sum-exp
  void* out;              // forward: O; backward: dQ
  void* dk;
  void* dv;
  float* lse_out;         // forward: L written here
  float* ws_nL2;          // [B*H, n_pad]  -L * log2(e), -inf past N (negated: feeds an FMA addend)
  float* ws_nD;           // [B*H, n_pad]  -rowsum(dO o O), 0 past N (negated: feeds an add)
  float* ws_dq;           // [B*H, n_pad, d] fp32 dQ accumulator (atomic and ordered modes) or null
  // Ordered dQ mode (null otherwise): one counter per (unit, 32-row query chunk)
  // of the completed contributions to that chunk of the accumulator, and the
  // ticket from which the key/value-major CTAs take their units in order. Both
  // zeroed by the preprocess.
  unsigned int* dq_flags;
  unsigned int* dq_ticket;
  // Persistent backward kernels (null: units in a fixed stride over the grid):
  // four counters in the workspace, zeroed by the preprocess: [0] the next unit
  // ticket and [1] the CTAs done of the key/value-major kernel, [2], [3] the
  // same for the query-major dQ kernel. The last CTA of a launch resets its pair.
  unsigned int* unit_ctr;
  unsigned int* status;   // device status word (timeout bits)
  // Packed variable-length input (null cu_seqlens otherwise): the tensors are
  // [total, H, d] (B = 1, N = total), sequence s occupies packed rows
  // [cu_seqlens[s], cu_seqlens[s+1]), attention stays within a sequence, L is
  // [H, total], and the L / D workspace rows of (h, s) start at
  // (h * nseq + s) * seq_pad (seq_pad = max_seqlen rounded up to kPadRows).
  const int* cu_seqlens;
  int nseq;
  int max_seqlen;
  int seq_pad;
  // ALiBi slopes (null: no position bias): the score of (i, j) gains
  // -m * |i - j| after the scale, m = alibi[seq * alibi_sb + h] with seq the
  // batch index (or the sequence index of packed input); alibi_sb = 0 shares
  // one slope per head across the batch.
  const float* alibi;
  int64_t alibi_sb;
  // Additive attention bias (null: none): the score of (i, j) gains
  // bias[b, h, i, j] after the scale, in the tensors' dtype, element strides
  // bias_sb / bias_sh (0 broadcasts over batches / heads) and bias_sn per
  // query row; keys are contiguous. -inf entries mask pairs out.
  const void* bias;
  int64_t bias_sb, bias_sh, bias_sn;
};

// One CTA's unit: a tile of rows of one (batch, head), or of one (sequence,
// head) with packed variable-length input. Rows are local to the unit; row0 is
// the unit's first row in the [B, N, H, d] (or packed) tensors, n its length,
// ws its L / D workspace row base, acc its dQ-accumulator row base, lse its
// base index in L.
struct Unit {
  int tile, b, h, bh, seq, row0, n;
  long long ws, acc, lse;
};

// Units (one (batch, head) or (sequence, head) each) are launched in groups
// of kUnitGroup: within a group tiles are outermost (heaviest first), so the
// CTAs resident at one time cover about 152 / kUnitGroup tiles of each of a
// few units and share those units' streamed operands through L2, while the
// heavy tiles of every group still start early.
constexpr int kUnitGroup = 8;

// Decodes block `idx` of a grid of ntiles * units CTAs. reverse_tiles != 0
// numbers the tiles from the last one down in launch order (heaviest first for
// the query-major kernels under a causal mask). `group` units share a group
// (default kUnitGroup; group >= units puts the tiles outermost over all units).
// Returns false for tiles past the end of a short sequence (the CTA has no work).
__device__ __forceinline__ bool unit_decode(const AttnParams& p, int idx, int tile_rows, bool reverse_tiles,
                                            Unit& u, int group = kUnitGroup) {
  const bool packed = p.cu_seqlens != nullptr;
  const int units = packed ? p.nseq * p.H : p.B * p.H;
  const int ntiles = ((packed ? p.max_seqlen : p.N) + tile_rows - 1) / tile_rows;
  group = min(group, units);
  const int g = idx / (group * ntiles), r = idx - g * (group * ntiles);
  const int gsize = min(group, units - g * group);  // the last group may be short
  u.tile = r / gsize;
  if (reverse_tiles) u.tile = ntiles - 1 - u.tile;
  const int unit = g * group + r % gsize;
  if (!packed) {
    u.bh = unit;
    u.b = u.bh / p.H;
    u.h = u.bh % p.H;
    u.seq = u.b;
    u.row0 = 0;
    u.n = p.N;
    u.ws = (long long)u.bh * p.n_pad;
    u.acc = u.ws;
    u.lse = (long long)u.bh * p.N;
    return true;
  }
  const int sq = unit / p.H;
  u.h = unit % p.H;
  u.seq = sq;
  u.b = 0;
  u.bh = u.h;
  // Clamp the offsets into [0, N] and the length to max_seqlen, so that a
  // malformed cu_seqlens cannot move any access outside the tensors.
  const int s0 = min(max(p.cu_seqlens[sq], 0), p.N), s1 = min(max(p.cu_seqlens[sq + 1], s0), p.N);
  u.row0 = s0;
  u.n = min(s1 - s0, p.max_seqlen);
  u.ws = ((long long)u.h * p.nseq + sq) * p.seq_pad;
  u.acc = (long long)u.h * p.n_pad + s0;
  u.lse = (long long)u.h * p.N + s0;
  return u.tile * tile_rows < u.n;
}

// ALiBi slope of a unit in score units: m / scale, so that the bias folds into
// the raw scores S = Q.K before the kernels' scale * log2(e) (the host requires
// scale > 0 with ALiBi).
__device__ __forceinline__ float alibi_slope_raw(const AttnParams& p, const Unit& u) {
  return __ldg(p.alibi + (long long)u.seq * p.alibi_sb + u.h) / p.scale;
}

// ALiBi on 16 raw scores of one TMEM row: s_e -= slope_raw * |d0 + kSign * e|,
// where d0 + kSign * e is i - j of column e (query-major rows: d0 = i - j_first,
// kSign = -1; key-major rows: d0 = i_first - j, kSign = +1).
template <int kSign>
__device__ __forceinline__ void alibi_fold16(uint32_t (&sr)[16], float d0, float slope_raw) {
#pragma unroll
  for (int e = 0; e < 16; ++e)
    sr[e] = __float_as_uint(fmaf(-slope_raw, fabsf(d0 + (float)(kSign * e)), __uint_as_float(sr[e])));
}

// ALiBi ramp on 16 raw scores: s_e += slope * (kX0 + e), kX0 the chunk column
// of e = 0 (one FMA with an immediate a score).
template <int kX0>
__device__ __forceinline__ void alibi_ramp16(uint32_t (&sr)[16], float slope) {
#pragma unroll
  for (int e = 0; e < 16; ++e) sr[e] = __float_as_uint(fmaf(slope, (float)(kX0 + e), __uint_as_float(sr[e])));
}

// 16-bit value (bf16 or fp16 bits in the low half) to fp32.
template <bool kBf16>
__device__ __forceinline__ float h16_bits_to_f32(uint32_t bits) {
  if constexpr (kBf16) {
    return __uint_as_float(bits << 16);
  } else {
    float f;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.f32.f16 %0, t;\n\t}" : "=f"(f) : "r"(bits));
    return f;
  }
}

// Attention bias on 16 raw scores of one TMEM row, read from a bias tile in
// shared memory: value e at addr + e * row_bytes, folded in score units
// (s += bias / scale, so that the kernels' scale * log2(e) restores it).
template <bool kBf16>
__device__ __forceinline__ void bias_fold16_smem(uint32_t (&sr)[16], uint32_t addr, uint32_t row_bytes,
                                                 float inv_scale) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr + (uint32_t)e * row_bytes));
    sr[e] = __float_as_uint(fmaf(h16_bits_to_f32<kBf16>(v), inv_scale, __uint_as_float(sr[e])));
  }
}

// The same from 16 consecutive 16-bit values held in registers (8 words).
template <bool kBf16>
__device__ __forceinline__ void bias_fold16_regs(uint32_t (&sr)[16], const uint32_t* w, float inv_scale) {
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    const float lo = h16_bits_to_f32<kBf16>(w[x] & 0xFFFFu), hi = h16_bits_to_f32<kBf16>(w[x] >> 16);
    sr[2 * x] = __float_as_uint(fmaf(lo, inv_scale, __uint_as_float(sr[2 * x])));
    sr[2 * x + 1] = __float_as_uint(fmaf(hi, inv_scale, __uint_as_float(sr[2 * x + 1])));
  }
}

// Allowed (query i, key j) pair under the causal / sliding-window mask.
__device__ __forceinline__ bool pair_allowed(const AttnParams& p, int i, int j) {
  return j < p.N && i < p.N && (!p.causal || j <= i) && (p.window <= 0 || j > i - p.window);
}

}  // namespace fa
