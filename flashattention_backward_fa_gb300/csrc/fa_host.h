// Host-side entry shared by the C-ABI translation units.
#pragma once
#include "fa.h"

namespace fa {

// Optional inputs of the forward and backward:
//  * ALiBi slopes (m = alibi[seq * alibi_sb + h]);
//  * an additive attention bias tensor with element strides bias_st
//    (b, n = per query row, h; 0 broadcasts), in the tensors' dtype;
//  * philox_bh_off, added to every (batch * H + head) index that keys a
//    dropout mask, so a call on a slice of the heads (B = 1) or of the batch
//    draws the whole problem's masks.
struct Extras {
  const float* alibi = nullptr;
  int64_t alibi_sb = 0;
  const void* bias = nullptr;
  fa_strides bias_st = {0, 0, 0};
  uint32_t philox_bh_off = 0;
};

// The whole backward (preprocess, dK/dV, dQ) on `stream`. With
// allow_side_stream, the deterministic 16-bit path runs its dQ kernel on a
// second, library-owned stream beside the dK/dV kernel (fork after the
// preprocess, join before returning); without it every kernel goes on `stream`
// and nothing is created.
int bwd_run(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
            float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
            const Extras& ex, int deterministic, void* workspace, size_t workspace_bytes, void* stream,
            bool allow_side_stream);

// One backward stage (fa_bwd_stage with the optional inputs of Extras).
int bwd_stage_run(fa_bwd_stage_id stage, const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                  uint64_t seed, uint64_t offset, const Extras& ex, int deterministic, void* workspace,
                  size_t workspace_bytes, void* stream, bool check_ptrs = true);

// The forward with the optional inputs of Extras.
int fwd_run(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
            fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p, uint64_t seed,
            uint64_t offset, const Extras& ex, void* stream);

// The shape, dtype, stride and scalar checks every entry point applies.
int check_bwd_args(int B, int H, int N, int d, fa_strides strides, fa_dtype dtype, float scale, int window,
                   float dropout_p);

}  // namespace fa
