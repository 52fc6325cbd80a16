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
  float* ws_dq;           // [B*H, n_pad, d] fp32 dQ accumulator (atomic mode) or null
  unsigned int* status;   // device status word (timeout bits)
};

// Allowed (query i, key j) pair under the causal / sliding-window mask.
__device__ __forceinline__ bool pair_allowed(const AttnParams& p, int i, int j) {
  return j < p.N && i < p.N && (!p.causal || j <= i) && (p.window <= 0 || j > i - p.window);
}

}  // namespace fa
