// C ABI of libfa.so: argument validation, workspace layout, TMA descriptor
// creation and kernel dispatch. Declarations and the contract: include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "fa.h"
#include "fa_host.h"
#include "fa_internal.h"

namespace fa {
cudaError_t launch_preprocess(const AttnParams& p, int dtype, cudaStream_t st);
cudaError_t launch_dq_convert(const AttnParams& p, int dtype, cudaStream_t st);
cudaError_t launch_fwd_f32(const AttnParams& p, cudaStream_t st);
cudaError_t launch_bwd_dkdv_f32(const AttnParams& p, cudaStream_t st);
cudaError_t launch_bwd_dq_f32(const AttnParams& p, cudaStream_t st);
cudaError_t launch_bwd_dkdv_tc(const AttnParams& p, bool bf16, bool atomic, const CUtensorMap* maps,
                               cudaStream_t st);
cudaError_t launch_qmajor_tc(const AttnParams& p, bool bf16, bool dq_mode, const CUtensorMap* maps,
                             cudaStream_t st);
bool fwd_pingpong_supported(const AttnParams& p);
cudaError_t launch_fwd_pingpong(const AttnParams& p, bool bf16, const CUtensorMap* maps, cudaStream_t st);
}  // namespace fa

namespace {

using fa::AttnParams;

// Device status word, one per device context; kernels get its address.
__device__ unsigned int g_status_word = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};

int status_ptr(unsigned int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return FA_ERR_CUDA;
    g_status_ptr[dev] = static_cast<unsigned int*>(ptr);
  }
  *out = g_status_ptr[dev];
  return FA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D map over a [B, N, H, d] tensor (dims innermost first: d, N, H, B), 128-byte
// swizzle, boxes of 64 head-dim elements x `rows` sequence rows.
bool make_map(CUtensorMap* m, const void* base, const AttnParams& p, bool bf16, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)p.d, (cuuint64_t)p.N, (cuuint64_t)p.H, (cuuint64_t)p.B};
  const cuuint64_t strides[3] = {(cuuint64_t)p.sn * 2, (cuuint64_t)p.sh * 2, (cuuint64_t)p.sb * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The attention bias as a 4-D map (keys, query rows, heads, batches); a
// broadcast dimension (stride 0) becomes a dimension of size 1; rows and keys
// past N read as 0. Key-major kernel: boxes of kStepQ rows x kRowsKV keys,
// unswizzled. Query-major kernels: boxes of kRowsQ rows x 64 keys, 128-byte
// swizzle.
bool make_bias_map(CUtensorMap* m, const AttnParams& p, bool bf16, bool query_major) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t nh = p.bias_sh ? (cuuint64_t)p.H : 1, nb = p.bias_sb ? (cuuint64_t)p.B : 1;
  const cuuint64_t plane = (cuuint64_t)p.bias_sn * p.N * 2;  // bytes of one [N, N] plane (stride of size-1 dims)
  const cuuint64_t dims[4] = {(cuuint64_t)p.N, (cuuint64_t)p.N, nh, nb};
  const cuuint64_t strides[3] = {(cuuint64_t)p.bias_sn * 2, p.bias_sh ? (cuuint64_t)p.bias_sh * 2 : plane,
                                 p.bias_sb ? (cuuint64_t)p.bias_sb * 2 : plane};
  const cuuint32_t box[4] = {query_major ? 64u : (cuuint32_t)fa::kRowsKV,
                             query_major ? (cuuint32_t)fa::kRowsQ : (cuuint32_t)fa::kStepQ, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
             const_cast<void*>(p.bias), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             query_major ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
inline int pad_rows(int N) { return (N + fa::kPadRows - 1) / fa::kPadRows * fa::kPadRows; }

// The dQ algorithm a `deterministic` argument selects (fa.h, FA_DQ_*). fp32 has
// one path (query-major, deterministic) whatever is asked.
enum class DqAlgo { kAtomic, kRecompute, kOrdered };

DqAlgo dq_algo(int dtype, int deterministic) {
  if (dtype == FA_F32) return DqAlgo::kRecompute;
  if (deterministic == FA_DQ_ATOMIC) return DqAlgo::kAtomic;
  if (deterministic == FA_DQ_ORDERED) return DqAlgo::kOrdered;
  return DqAlgo::kRecompute;  // FA_DQ_DETERMINISTIC, FA_DQ_RECOMPUTE
}

bool valid_dq_mode(int deterministic) {
  return deterministic == FA_DQ_ATOMIC || deterministic == FA_DQ_DETERMINISTIC || deterministic == FA_DQ_RECOMPUTE ||
         deterministic == FA_DQ_ORDERED;
}

bool needs_dq_accum(int dtype, int deterministic) { return dq_algo(dtype, deterministic) != DqAlgo::kRecompute; }

struct WsLayout {
  size_t off_L2, off_D, off_ctr, off_dq, off_flags, off_ticket, total;
};

// [-L*log2e | -D | the persistent kernels' unit counters | fp32 dQ accumulator
// (atomic, ordered) | chunk counters and the unit ticket (ordered)], each part
// 256-byte aligned.
WsLayout ws_layout(int B, int H, int N, int d, int dtype, int deterministic) {
  const size_t rows = (size_t)B * H * pad_rows(N);
  WsLayout w;
  w.off_L2 = 0;
  w.off_D = round256(rows * 4);
  w.off_ctr = w.off_D + round256(rows * 4);
  w.off_dq = w.off_ctr + 256;
  w.off_flags = w.off_dq + (needs_dq_accum(dtype, deterministic) ? round256(rows * (size_t)d * 4) : 0);
  const bool ordered = dq_algo(dtype, deterministic) == DqAlgo::kOrdered;
  w.off_ticket = w.off_flags + (ordered ? round256(rows / 32 * 4) : 0);
  w.total = w.off_ticket + (ordered ? 256 : 0);
  return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor-map encoding (cuTensorMapEncodeTiled) is a driver call that needs a
// current context on the calling thread. A thread whose CUDA calls so far bound
// none (pointer queries, this library's cached lookups) would see it fail, so
// every entry point makes the current device's primary context current first:
// cudaSetDevice initialises that context and binds it to the thread.
int bind_device_context() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

// Every buffer a kernel touches must be memory of the current device (or
// managed memory): a host or another device's pointer would make the kernels
// fault. Checked last, after the cheap argument checks and before any launch.
// Null entries are optional inputs that are absent.
int check_device_ptrs(std::initializer_list<const void*> ptrs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  for (const void* ptr : ptrs) {
    if (!ptr) continue;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
      cudaGetLastError();  // not a pointer the runtime knows: clear the (non-sticky) error
      return FA_ERR_INVALID_ARG;
    }
    if (at.type == cudaMemoryTypeManaged) continue;
    if (at.type != cudaMemoryTypeDevice || at.device != dev) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

// Validation shared by the forward and the backward. Returns FA_OK or an error.
int check_common(int B, int H, int N, int d, fa_strides s, int dtype, float scale, int window, float dropout_p) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_F32 ? d > 128 : (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
  if (s.b < 1 || s.n < 1 || s.h < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (window < 0) return FA_ERR_INVALID_ARG;
  if (!(dropout_p >= 0.f && dropout_p < 1.f)) return FA_ERR_INVALID_ARG;
  // Index arithmetic stays in 32-bit grids and 64-bit offsets.
  if ((long long)B * H > (1ll << 24) || N > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_F32 && ((s.b | s.n | s.h) & 7)) return FA_ERR_ALIGNMENT;
  return FA_OK;
}

void fill_params(AttnParams& p, int B, int H, int N, int d, fa_strides s, float scale, int causal, int window,
                 float dropout_p, uint64_t seed, uint64_t offset) {
  std::memset(&p, 0, sizeof(p));
  p.B = B;
  p.H = H;
  p.N = N;
  p.d = d;
  p.sb = s.b;
  p.sn = s.n;
  p.sh = s.h;
  p.n_pad = pad_rows(N);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.window = window;
  p.drop.on = dropout_p > 0.f ? 1u : 0u;
  p.drop.threshold = (uint32_t)std::floor((double)dropout_p * 65536.0);  // < 2^16 for dropout_p < 1
  p.drop.rp = 1.f / (1.f - dropout_p);
  p.drop.seed_lo = (uint32_t)seed;
  p.drop.seed_hi = (uint32_t)(seed >> 32);
  p.drop.off_lo = (uint32_t)offset;
  p.drop.off_hi = (uint32_t)(offset >> 32);
}

// ALiBi slopes: fp32, 4-byte aligned, a non-negative batch (or sequence)
// stride; the kernels fold the bias into the raw scores as m / scale, so the
// scale must be positive.
int check_alibi(const float* alibi, int64_t alibi_sb, float scale) {
  if (!alibi) return FA_OK;
  if (reinterpret_cast<uintptr_t>(alibi) & 3u) return FA_ERR_ALIGNMENT;
  if (alibi_sb < 0) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Attention bias: strides non-negative with rows at least N keys apart; the
// 16-bit kernels read it with 16-byte loads and TMA, so there the base is
// 16-byte aligned and every stride a multiple of 8 elements; folded in score
// units as bias / scale, so the scale must be positive.
int check_bias(const void* bias, fa_strides st, int N, int dtype, float scale) {
  if (!bias) return FA_OK;
  if (st.b < 0 || st.h < 0 || st.n < N) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_F32) return (reinterpret_cast<uintptr_t>(bias) & 3u) ? FA_ERR_ALIGNMENT : FA_OK;
  if ((reinterpret_cast<uintptr_t>(bias) & 15u) || ((st.b | st.h | st.n) & 7)) return FA_ERR_ALIGNMENT;
  return FA_OK;
}

void apply_extras(AttnParams& p, const fa::Extras& ex) {
  p.drop.bh_off = ex.philox_bh_off;
  p.alibi = ex.alibi;
  p.alibi_sb = ex.alibi_sb;
  p.bias = ex.bias;
  p.bias_sb = ex.bias_st.b;
  p.bias_sh = ex.bias_st.h;
  p.bias_sn = ex.bias_st.n;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// The fp32 dQ accumulator as a 3-D map (d, rows per head, heads): rows per head
// n_pad (packed input: the per-head accumulator rows), heads B*H (packed: H);
// boxes of d x 32 rows, unswizzled, for the key/value-major kernel's TMA
// reduce-adds of its staged [32 rows][d] tiles.
bool make_dq_accum_map(CUtensorMap* m, const AttnParams& p) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t nz = p.cu_seqlens ? (cuuint64_t)p.H : (cuuint64_t)p.B * p.H;
  const cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.n_pad, nz};
  const cuuint64_t strides[2] = {(cuuint64_t)p.d * 4, (cuuint64_t)p.n_pad * p.d * 4};
  const cuuint32_t box[3] = {(cuuint32_t)p.d, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.ws_dq, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches one backward stage for fully validated and filled parameters.
int launch_stage(fa_bwd_stage_id stage, const AttnParams& p, int dtype, int deterministic, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (stage == FA_BWD_PREPROCESS) return cuda_rc(fa::launch_preprocess(p, dtype, st));
  if (dtype == FA_F32)
    return cuda_rc(stage == FA_BWD_DKDV ? fa::launch_bwd_dkdv_f32(p, st) : fa::launch_bwd_dq_f32(p, st));
  const bool bf16 = dtype == FA_BF16;
  const bool accum = dq_algo(dtype, deterministic) != DqAlgo::kRecompute;
  if (stage == FA_BWD_DKDV) {
    CUtensorMap maps[6];
    if (!make_map(&maps[0], p.q, p, bf16, fa::kStepQ) || !make_map(&maps[1], p.k, p, bf16, fa::kRowsKV) ||
        !make_map(&maps[2], p.v, p, bf16, fa::kRowsKV) || !make_map(&maps[3], p.dout, p, bf16, fa::kStepQ))
      return FA_ERR_CUDA;
    if (p.bias ? !make_bias_map(&maps[4], p, bf16, false) : false) return FA_ERR_CUDA;
    if (!p.bias) maps[4] = maps[0];  // unused
    if (accum ? !make_dq_accum_map(&maps[5], p) : false) return FA_ERR_CUDA;
    if (!accum) maps[5] = maps[0];  // unused
    return cuda_rc(fa::launch_bwd_dkdv_tc(p, bf16, accum, maps, st));
  }
  if (accum) return cuda_rc(fa::launch_dq_convert(p, dtype, st));
  CUtensorMap maps[5];
  if (!make_map(&maps[0], p.q, p, bf16, fa::kRowsQ) || !make_map(&maps[1], p.k, p, bf16, fa::kStepKV) ||
      !make_map(&maps[2], p.v, p, bf16, fa::kStepKV) || !make_map(&maps[3], p.dout, p, bf16, fa::kRowsQ))
    return FA_ERR_CUDA;
  if (p.bias ? !make_bias_map(&maps[4], p, bf16, true) : false) return FA_ERR_CUDA;
  if (!p.bias) maps[4] = maps[0];  // unused
  return cuda_rc(fa::launch_qmajor_tc(p, bf16, true, maps, st));
}

// A second stream per device on which the deterministic backward runs its dQ
// kernel beside the dK/dV kernel (fork after the preprocess, join before
// returning), so that the two grids share the tail of each other's last wave
// instead of running back to back. Created on first use and kept.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxDevices];
// Guards g_side and serialises each fork/join enqueue sequence. Distinct from
// g_mu, which the stage launches below take themselves.
std::mutex g_side_mu;

// Caller holds g_side_mu.
int side_stream_locked(SideStream** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  SideStream& ss = g_side[dev];
  if (!ss.stream) {
    if (cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  *out = &ss;
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_version(void) { return 100; }

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension, dtype or size";
    case FA_ERR_ALIGNMENT: return "pointer or stride violates the alignment rules";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FA_ERR_CUDA: return "CUDA call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
    default: return "unknown error code";
  }
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d, fa_dtype dtype, int deterministic) {
  if (B < 1 || H < 1 || N < 1 || d < 1 || d > 128) return 0;
  if (!valid_dq_mode(deterministic)) return 0;
  if (dtype != FA_F32 && dtype != FA_F16 && dtype != FA_BF16) return 0;
  if ((long long)B * H > (1ll << 24) || N > (1 << 30)) return 0;  // beyond the size limits (and pad_rows' int range)
  return ws_layout(B, H, N, d, dtype, deterministic).total;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
           uint64_t seed, uint64_t offset, void* stream) {
  return fa::fwd_run(q, k, v, o, lse, B, H, N, d, strides, dtype, scale, causal, window, dropout_p, seed, offset,
                     fa::Extras{}, stream);
}

int fa_fwd_alibi(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                 uint64_t seed, uint64_t offset, const float* alibi_slopes, int64_t alibi_stride_b, void* stream) {
  fa::Extras ex;
  ex.alibi = alibi_slopes;
  ex.alibi_sb = alibi_stride_b;
  return fa::fwd_run(q, k, v, o, lse, B, H, N, d, strides, dtype, scale, causal, window, dropout_p, seed, offset,
                     ex, stream);
}

int fa_fwd_bias(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                uint64_t seed, uint64_t offset, const void* bias, fa_strides bias_strides, void* stream) {
  if (!bias) return FA_ERR_INVALID_ARG;
  fa::Extras ex;
  ex.bias = bias;
  ex.bias_st = bias_strides;
  return fa::fwd_run(q, k, v, o, lse, B, H, N, d, strides, dtype, scale, causal, window, dropout_p, seed, offset,
                     ex, stream);
}

int fa_bwd_stage(fa_bwd_stage_id stage, const void* q, const void* k, const void* v, const void* o,
                 const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                 uint64_t seed, uint64_t offset, int deterministic, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return fa::bwd_stage_run(stage, q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, strides, dtype, scale, causal,
                           window, dropout_p, seed, offset, fa::Extras{}, deterministic, workspace, workspace_bytes,
                           stream);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
           float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
           int deterministic, void* workspace, size_t workspace_bytes, void* stream) {
  return fa::bwd_run(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, strides, dtype, scale, causal, window,
                     dropout_p, seed, offset, fa::Extras{}, deterministic, workspace, workspace_bytes, stream, true);
}

int fa_bwd_alibi(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
                 float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
                 const float* alibi_slopes, int64_t alibi_stride_b, int deterministic, void* workspace,
                 size_t workspace_bytes, void* stream) {
  fa::Extras ex;
  ex.alibi = alibi_slopes;
  ex.alibi_sb = alibi_stride_b;
  return fa::bwd_run(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, strides, dtype, scale, causal, window,
                     dropout_p, seed, offset, ex, deterministic, workspace, workspace_bytes, stream, true);
}

int fa_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
                float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
                const void* bias, fa_strides bias_strides, int deterministic, void* workspace,
                size_t workspace_bytes, void* stream) {
  if (!bias) return FA_ERR_INVALID_ARG;
  fa::Extras ex;
  ex.bias = bias;
  ex.bias_st = bias_strides;
  return fa::bwd_run(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, strides, dtype, scale, causal, window,
                     dropout_p, seed, offset, ex, deterministic, workspace, workspace_bytes, stream, true);
}

}  // extern "C"

namespace fa {

int bwd_stage_run(fa_bwd_stage_id stage, const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                  uint64_t seed, uint64_t offset, const Extras& ex, int deterministic, void* workspace,
                  size_t workspace_bytes, void* stream, bool check_ptrs) {
  int rc = check_common(B, H, N, d, strides, dtype, scale, window, dropout_p);
  if (rc) return rc;
  if ((rc = check_alibi(ex.alibi, ex.alibi_sb, scale))) return rc;
  if ((rc = check_bias(ex.bias, ex.bias_st, N, dtype, scale))) return rc;
  if (stage != FA_BWD_PREPROCESS && stage != FA_BWD_DKDV && stage != FA_BWD_DQ) return FA_ERR_INVALID_ARG;
  if (!valid_dq_mode(deterministic)) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  const void* all[] = {q, k, v, o, dout, lse, dq, dk, dv};
  for (const void* ptr : all)
    if (!aligned16(ptr)) return FA_ERR_ALIGNMENT;
  const WsLayout w = ws_layout(B, H, N, d, dtype, deterministic);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < w.total)
    return FA_ERR_WORKSPACE;
  if (check_ptrs && (rc = check_device_ptrs({q, k, v, o, dout, lse, dq, dk, dv, workspace, ex.alibi, ex.bias})))
    return rc;
  if ((rc = bind_device_context())) return rc;
  AttnParams p;
  fill_params(p, B, H, N, d, strides, scale, causal, window, dropout_p, seed, offset);
  apply_extras(p, ex);
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.out = dq;
  p.dk = dk;
  p.dv = dv;
  char* ws = static_cast<char*>(workspace);
  p.ws_nL2 = reinterpret_cast<float*>(ws + w.off_L2);
  p.ws_nD = reinterpret_cast<float*>(ws + w.off_D);
  p.ws_dq = needs_dq_accum(dtype, deterministic) ? reinterpret_cast<float*>(ws + w.off_dq) : nullptr;
  p.unit_ctr = reinterpret_cast<unsigned int*>(ws + w.off_ctr);
  if (dq_algo(dtype, deterministic) == DqAlgo::kOrdered) {
    p.dq_flags = reinterpret_cast<unsigned int*>(ws + w.off_flags);
    p.dq_ticket = reinterpret_cast<unsigned int*>(ws + w.off_ticket);
  }
  if ((rc = status_ptr(&p.status))) return rc;
  return launch_stage(stage, p, dtype, deterministic, stream);
}

int fwd_run(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
            fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p, uint64_t seed,
            uint64_t offset, const Extras& ex, void* stream) {
  int rc = check_common(B, H, N, d, strides, dtype, scale, window, dropout_p);
  if (rc) return rc;
  if ((rc = check_alibi(ex.alibi, ex.alibi_sb, scale))) return rc;
  if ((rc = check_bias(ex.bias, ex.bias_st, N, dtype, scale))) return rc;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_ALIGNMENT;
  if ((rc = check_device_ptrs({q, k, v, o, lse, ex.alibi, ex.bias}))) return rc;
  if ((rc = bind_device_context())) return rc;
  AttnParams p;
  fill_params(p, B, H, N, d, strides, scale, causal, window, dropout_p, seed, offset);
  apply_extras(p, ex);
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = o;
  p.lse_out = lse;
  if ((rc = status_ptr(&p.status))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == FA_F32) return cuda_rc(fa::launch_fwd_f32(p, st));
  const bool bf16 = dtype == FA_BF16;
  CUtensorMap maps[5];
  if (!make_map(&maps[0], q, p, bf16, fa::kRowsQ) || !make_map(&maps[1], k, p, bf16, fa::kStepKV) ||
      !make_map(&maps[2], v, p, bf16, fa::kStepKV))
    return FA_ERR_CUDA;
  // the common case (no dropout, ALiBi, bias or window): two query tiles per CTA in ping-pong
  if (fa::fwd_pingpong_supported(p)) return cuda_rc(fa::launch_fwd_pingpong(p, bf16, maps, st));
  maps[3] = maps[0];
  if (p.bias ? !make_bias_map(&maps[4], p, bf16, true) : false) return FA_ERR_CUDA;
  if (!p.bias) maps[4] = maps[0];  // unused
  return cuda_rc(fa::launch_qmajor_tc(p, bf16, false, maps, st));
}

int check_bwd_args(int B, int H, int N, int d, fa_strides strides, fa_dtype dtype, float scale, int window,
                   float dropout_p) {
  return check_common(B, H, N, d, strides, dtype, scale, window, dropout_p);
}

}  // namespace fa

namespace {

// Failure-detection self-test (fa_selftest_timeout): one CTA of two warps holds
// 32 TMEM columns and waits on an mbarrier that nothing ever arrives on. Warp 1
// polls (test_wait), warp 0 blocks (try_wait), as the row-math and MMA-issuing
// warps of the attention kernels do. The first wait to pass the wall-clock
// limit sets the timeout bit and the CTA's abort flag; the other leaves at its
// next abort check. Thread 0 then runs the bounded drain wait on the same
// barrier, which gives up after the limit as well. Warp 0 frees TMEM and the
// CTA exits, leaving the context usable.
__global__ void __launch_bounds__(64, 1) selftest_timeout_kernel(unsigned int* status, int* outcome) {
  __shared__ __align__(8) unsigned long long bar_word;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5;
  const uint32_t bar = fa::smem_u32(&bar_word);
  if (threadIdx.x == 0) {
    fa::mbar_init(bar, 1);
    abort_flag = 0;
    fa::fence_mbar_init();
  }
  if (warp == 0) {
    fa::tmem_alloc(fa::smem_u32(&tmem_slot), 32);
    fa::tmem_relinquish();
  }
  fa::tc_fence_before();
  __syncthreads();
  fa::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const bool ok = warp == 1 ? fa::warp_wait<true>(bar, 0, &abort_flag, status)
                            : fa::warp_wait<false>(bar, 0, &abort_flag, status);
  if ((threadIdx.x & 31) == 0) atomicOr(outcome, ok ? 0 : (1 << warp));
  if (threadIdx.x == 0) fa::mbar_wait_drain(bar, 0, status);
  fa::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    fa::tc_fence_after();
    fa::tmem_dealloc(tmem, 32);
  }
}

}  // namespace

extern "C" {

int fa_selftest_timeout(int* outcome, void* stream) {
  if (!outcome) return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  selftest_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(status, outcome);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_get_device_status(unsigned int* status, int clear) {
  if (!status) return FA_ERR_INVALID_ARG;
  unsigned int* ptr = nullptr;
  int rc = status_ptr(&ptr);
  if (rc) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpy(status, ptr, sizeof(unsigned int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (clear && cudaMemset(ptr, 0, sizeof(unsigned int)) != cudaSuccess) return FA_ERR_CUDA;
  return (*status & fa::kStatusTimeout) ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"

namespace {

// The three stages in order; the deterministic 16-bit backward forks its dQ
// kernel onto the side stream (see SideStream).
template <typename StageFn>
int run_backward(StageFn stage, int deterministic, int dtype, bool allow_side_stream, void* stream) {
  int rc = stage(FA_BWD_PREPROCESS, stream);
  if (rc) return rc;
  if (!allow_side_stream || dq_algo(dtype, deterministic) != DqAlgo::kRecompute || dtype == FA_F32) {
    if ((rc = stage(FA_BWD_DKDV, stream))) return rc;
    return stage(FA_BWD_DQ, stream);
  }
  // Fork: the dQ kernel waits for the preprocess on the side stream while the
  // dK/dV kernel follows it on the caller's stream; join before returning. The
  // enqueue sequence is serialised because the fork/join events are shared.
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream* ss = nullptr;
  if ((rc = side_stream_locked(&ss))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaEventRecord(ss->fork, st) != cudaSuccess || cudaStreamWaitEvent(ss->stream, ss->fork, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  if ((rc = stage(FA_BWD_DKDV, stream))) return rc;
  if ((rc = stage(FA_BWD_DQ, ss->stream))) return rc;
  if (cudaEventRecord(ss->join, ss->stream) != cudaSuccess || cudaStreamWaitEvent(st, ss->join, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

namespace fa {

int bwd_run(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
            float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
            const Extras& ex, int deterministic, void* workspace, size_t workspace_bytes, void* stream,
            bool allow_side_stream) {
  auto stage = [&](fa_bwd_stage_id s, void* st) {
    // The buffers are the same for all three steps: the first one checks them.
    return bwd_stage_run(s, q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, strides, dtype, scale, causal, window,
                         dropout_p, seed, offset, ex, deterministic, workspace, workspace_bytes, st,
                         s == FA_BWD_PREPROCESS);
  };
  return run_backward(stage, deterministic, dtype, allow_side_stream, stream);
}

}  // namespace fa

// ------------------------- packed variable-length -------------------------
namespace {

struct VarlenWs {
  int seq_pad, acc_rows;
  size_t off_L2, off_D, off_ctr, off_dq, off_flags, off_ticket, total;
};

VarlenWs varlen_ws_layout(int nseq, int max_seqlen, int total, int H, int d, int deterministic) {
  VarlenWs w;
  w.seq_pad = pad_rows(max_seqlen);
  w.acc_rows = pad_rows(total) + fa::kPadRows;  // a tile may run past its sequence's last row
  const size_t vec = (size_t)H * nseq * w.seq_pad * 4;
  w.off_L2 = 0;
  w.off_D = round256(vec);
  w.off_ctr = w.off_D + round256(vec);
  w.off_dq = w.off_ctr + 256;
  const DqAlgo a = dq_algo(FA_BF16, deterministic);
  w.off_flags = w.off_dq + (a != DqAlgo::kRecompute ? round256((size_t)H * w.acc_rows * d * 4) : 0);
  w.off_ticket = w.off_flags + (a == DqAlgo::kOrdered ? round256(vec / 32) : 0);
  w.total = w.off_ticket + (a == DqAlgo::kOrdered ? 256 : 0);
  return w;
}

// Validation and parameters common to the varlen forward and backward.
int varlen_params(AttnParams& p, const int* cu_seqlens, int nseq, int max_seqlen, int total, int H, int d,
                  int64_t stride_n, int64_t stride_h, fa_dtype dtype, float scale, int causal, int window,
                  const float* alibi, int64_t alibi_ss) {
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FA_ERR_INVALID_ARG;
  if (nseq < 1 || max_seqlen < 1 || total < 1 || H < 1) return FA_ERR_INVALID_ARG;
  if ((long long)nseq * H > 65535) return FA_ERR_UNSUPPORTED;
  // one CTA per (128-row tile of max_seqlen, sequence, head) in a 1-D grid
  if ((long long)pad_rows(max_seqlen) / fa::kPadRows * nseq * H > 0x7fffffffll) return FA_ERR_UNSUPPORTED;
  const fa_strides s = {stride_n, stride_n, stride_h};  // B = 1: the batch stride is never used
  int rc = check_common(1, H, total, d, s, dtype, scale, window, 0.f);
  if (rc) return rc;
  if ((rc = check_alibi(alibi, alibi_ss, scale))) return rc;
  fill_params(p, 1, H, total, d, s, scale, causal, window, 0.f, 0, 0);
  p.alibi = alibi;
  p.alibi_sb = alibi_ss;
  p.cu_seqlens = cu_seqlens;
  p.nseq = nseq;
  p.max_seqlen = max_seqlen;
  p.seq_pad = pad_rows(max_seqlen);
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_varlen_bwd_workspace_size(int nseq, int max_seqlen, int total, int H, int d, fa_dtype dtype,
                                    int deterministic) {
  if (nseq < 1 || max_seqlen < 1 || total < 1 || H < 1 || (d != 64 && d != 128)) return 0;
  if (dtype != FA_F16 && dtype != FA_BF16) return 0;
  if (!valid_dq_mode(deterministic)) return 0;
  return varlen_ws_layout(nseq, max_seqlen, total, H, d, deterministic).total;
}

int fa_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens, int nseq,
                  int max_seqlen, int total, int H, int d, int64_t stride_n, int64_t stride_h, fa_dtype dtype,
                  float scale, int causal, int window, const float* alibi_slopes, int64_t alibi_stride_seq,
                  void* stream) {
  AttnParams p;
  int rc = varlen_params(p, cu_seqlens, nseq, max_seqlen, total, H, d, stride_n, stride_h, dtype, scale, causal,
                         window, alibi_slopes, alibi_stride_seq);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_ALIGNMENT;
  if ((rc = check_device_ptrs({q, k, v, o, lse, cu_seqlens, alibi_slopes}))) return rc;
  if ((rc = bind_device_context())) return rc;
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = o;
  p.lse_out = lse;
  if ((rc = status_ptr(&p.status))) return rc;
  const bool bf16 = dtype == FA_BF16;
  CUtensorMap maps[5];
  if (!make_map(&maps[0], q, p, bf16, fa::kRowsQ) || !make_map(&maps[1], k, p, bf16, fa::kStepKV) ||
      !make_map(&maps[2], v, p, bf16, fa::kStepKV))
    return FA_ERR_CUDA;
  if (fa::fwd_pingpong_supported(p)) return cuda_rc(fa::launch_fwd_pingpong(p, bf16, maps, static_cast<cudaStream_t>(stream)));
  maps[3] = maps[0];
  maps[4] = maps[0];  // no attention bias on packed input
  return cuda_rc(fa::launch_qmajor_tc(p, bf16, false, maps, static_cast<cudaStream_t>(stream)));
}

int fa_varlen_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, const int* cu_seqlens, int nseq, int max_seqlen, int total, int H,
                  int d, int64_t stride_n, int64_t stride_h, fa_dtype dtype, float scale, int causal, int window,
                  const float* alibi_slopes, int64_t alibi_stride_seq, int deterministic, void* workspace,
                  size_t workspace_bytes, void* stream) {
  AttnParams p;
  int rc = varlen_params(p, cu_seqlens, nseq, max_seqlen, total, H, d, stride_n, stride_h, dtype, scale, causal,
                         window, alibi_slopes, alibi_stride_seq);
  if (rc) return rc;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!valid_dq_mode(deterministic)) return FA_ERR_INVALID_ARG;
  const void* all[] = {q, k, v, o, dout, lse, dq, dk, dv};
  for (const void* ptr : all)
    if (!aligned16(ptr)) return FA_ERR_ALIGNMENT;
  const VarlenWs w = varlen_ws_layout(nseq, max_seqlen, total, H, d, deterministic);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < w.total)
    return FA_ERR_WORKSPACE;
  if ((rc = check_device_ptrs({q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens, alibi_slopes}))) return rc;
  if ((rc = bind_device_context())) return rc;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.out = dq;
  p.dk = dk;
  p.dv = dv;
  p.n_pad = w.acc_rows;  // dQ accumulator rows per head (packed rows + tail)
  char* ws = static_cast<char*>(workspace);
  p.ws_nL2 = reinterpret_cast<float*>(ws + w.off_L2);
  p.ws_nD = reinterpret_cast<float*>(ws + w.off_D);
  const DqAlgo algo = dq_algo(dtype, deterministic);
  p.ws_dq = algo == DqAlgo::kRecompute ? nullptr : reinterpret_cast<float*>(ws + w.off_dq);
  p.unit_ctr = reinterpret_cast<unsigned int*>(ws + w.off_ctr);
  if (algo == DqAlgo::kOrdered) {
    p.dq_flags = reinterpret_cast<unsigned int*>(ws + w.off_flags);
    p.dq_ticket = reinterpret_cast<unsigned int*>(ws + w.off_ticket);
  }
  if ((rc = status_ptr(&p.status))) return rc;
  const size_t acc_bytes = (size_t)H * w.acc_rows * d * 4;
  auto stage = [&](fa_bwd_stage_id s, void* st) {
    if (s == FA_BWD_PREPROCESS && p.ws_dq &&
        cudaMemsetAsync(p.ws_dq, 0, acc_bytes, static_cast<cudaStream_t>(st)) != cudaSuccess)
      return (int)FA_ERR_CUDA;
    return launch_stage(s, p, dtype, deterministic, st);
  };
  return run_backward(stage, deterministic, dtype, true, stream);
}

}  // extern "C"
