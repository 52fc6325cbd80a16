/*
 * fa.h — C ABI of the GB300 (sm_103a) FlashAttention forward/backward library (libfa.so).
 *
 * What is computed. For every batch b and head h of [B, N, H, d] tensors:
 *   S = scale * Q K^T; pairs outside the mask get S = -inf
 *   L_i = log sum_j exp(S_ij)                         (natural log, before dropout)
 *   P = exp(S - L);  P~ = P o Z / (1 - p)             (Z: dropout keep-mask)
 *   O = P~ V
 * and the backward, from the saved state (O, L) and the upstream gradient dO:
 *   D_i = sum_k dO_ik O_ik
 *   dV = P~^T dO;  dP = (dO V^T) o Z / (1 - p);  dS = P o (dP - D)
 *   dQ = scale * dS K;  dK = scale * dS^T Q
 * Sources: "FlashAttention backward" (GPU-kernels lesson 29), §What the forward
 * left behind (O and L are the saved state; P = exp(S - L)) and §The gradients,
 * and the one scalar that makes them local (the formulas and D); "Lecture 7 —
 * Backward Pass and Validation", §The math, §Mask behaviour, §Dropout,
 * §Determinism; "Implementing Flash Attention's Backward Pass in Raw CUDA",
 * §Deriving the gradients. The N x N matrix P is never materialised.
 *
 * Masks. causal != 0 keeps pairs j <= i (top-left aligned, square attention).
 * window > 0 keeps pairs j > i - window; with causal this is the two-sided
 * sliding window i - window < j <= i. window == 0 means no window.
 *
 * Dropout. 0 <= dropout_p < 1. The keep decision of element (b, h, i, j)
 * uses Philox4x32-10 (Salmon et al., SC'11) with
 *   key     = (lo32(seed), hi32(seed))
 *   counter = (lo32(g), hi32(g), lo32(offset), hi32(offset)),
 *   g       = ((b*H + h)*N + i) * ceil(N/8) + floor(j/8)
 * One call serves eight keys: key j takes 16-bit half (j mod 2) (the low half
 * for even j) of output word ((j mod 8) div 2), and the element is kept iff
 * that half >= floor(dropout_p * 2^16). Kept elements are scaled by
 * 1/(1 - dropout_p). fa_fwd and fa_bwd draw the same mask for the same
 * (seed, offset).
 *
 * Layout. Q, K, V, O, dO, dQ, dK, dV share one element-stride triple
 * fa_strides {b, n, h}: element (b, i, h, k) lives at b*s.b + i*s.n + h*s.h + k
 * (the head dimension is contiguous). [B, N, H, d] contiguous is
 * {N*H*d, H*d, d}; [B, H, N, d] contiguous is {H*N*d, d, N*d}.
 * L (lse) is a contiguous fp32 [B, H, N] array.
 *
 * Supported. fp16 / bf16: d in {64, 128}, tensor-core (tcgen05) kernels.
 * fp32: 1 <= d <= 128, CUDA-core kernels. Any N >= 1, B >= 1, H >= 1 up to
 * B*H <= 2^24 and N <= 2^30 (FA_ERR_UNSUPPORTED beyond: the kernels index in
 * 32-bit grids and 64-bit offsets).
 * Alignment: every tensor base 16-byte aligned; for fp16/bf16 every stride a
 * multiple of 8 elements (the TMA rule of 16-byte strides); for fp32 strides
 * only need to be positive.
 *
 * Ownership and execution. The caller owns every buffer, and no call
 * allocates device memory. The library does hold a little module state per
 * device: the device status word (see fa_get_device_status), the fixed 8 MiB (+256 B)
 * scratch array of fa_bwd_noalloc (shared by all of its calls, which keeps the
 * last call's contents; see its declaration), and, created on first use, one
 * side stream with two events for the deterministic fa_bwd and two copy
 * streams for fa_bwd_host. All pointers are
 * device pointers of the current device (or managed memory), except the host
 * buffers of fa_bwd_host. After the other argument checks, and before anything
 * is launched, every buffer is looked up with cudaPointerGetAttributes: a host
 * pointer, another device's pointer or an unknown address returns
 * FA_ERR_INVALID_ARG. Calls are asynchronous on `stream` (a cudaStream_t, NULL =
 * the legacy default stream). Outputs are overwritten, never accumulated into.
 * Return value: FA_OK, or a negative FA_ERR_* code when an argument is
 * rejected (nothing is launched) or a launch fails. Faults during execution
 * surface at the caller's next synchronisation, as for any CUDA call. A kernel
 * whose internal bounded wait gives up sets a device status bit that
 * fa_get_device_status() reports as FA_ERR_TIMEOUT. No C++ exception crosses
 * this boundary. Thread-safe.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_F32 = 0, FA_F16 = 1, FA_BF16 = 2 } fa_dtype;

enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad mask/dropout value */
  FA_ERR_UNSUPPORTED = -2, /* head dimension or dtype this library does not handle */
  FA_ERR_ALIGNMENT = -3,   /* base pointer or stride violates the alignment rules */
  FA_ERR_WORKSPACE = -4,   /* workspace missing, misaligned (256 B) or too small */
  FA_ERR_CUDA = -5,        /* a CUDA runtime/driver call or kernel launch failed */
  FA_ERR_TIMEOUT = -6      /* a kernel's bounded wait gave up (see fa_get_device_status) */
};

/* dQ algorithms, selected by the `deterministic` argument of the backward
 * entry points ("FlashAttention backward", §The loop structure: who
 * accumulates cleanly, who needs atomics; "Lecture 7 — Backward Pass and
 * Validation", §Determinism):
 *  FA_DQ_ATOMIC (0): the key/value-major kernel also forms dQ^T = K^T dS^T per
 *    tile and adds it into an fp32 accumulator with TMA reduce-adds in no fixed
 *    order, then a conversion pass scales and rounds it. Five contractions per
 *    tile pair; dQ may differ in the last bits between runs.
 *  FA_DQ_DETERMINISTIC (1): the library's deterministic default, currently
 *    FA_DQ_RECOMPUTE.
 *  FA_DQ_RECOMPUTE (2): a separate query-major kernel recomputes S and dP and
 *    accumulates dQ on chip. Seven contractions per tile pair; bit-identical
 *    run to run.
 *  FA_DQ_ORDERED (3): as FA_DQ_ATOMIC, but the contributions of the key blocks
 *    to each 32-row query chunk are added in ascending key-block order (each
 *    waits for its predecessors through a counter in the workspace), so the
 *    fp32 sums, and dQ, are bit-identical run to run. Five contractions per
 *    tile pair.
 * dK and dV are deterministic in every mode. fp32 inputs always take the
 * query-major path. Other values return FA_ERR_INVALID_ARG (and a workspace
 * size of 0). */
#define FA_DQ_ATOMIC 0
#define FA_DQ_DETERMINISTIC 1
#define FA_DQ_RECOMPUTE 2
#define FA_DQ_ORDERED 3

/* Element strides of the [B, N, H, d] tensors; the d stride is 1. */
typedef struct {
  int64_t b, n, h;
} fa_strides;

/* Bytes of device workspace fa_bwd needs: two fp32 vectors of B*H*roundup(N,128)
 * (L*log2(e) and D), plus, for fp16/bf16 with FA_DQ_ATOMIC or FA_DQ_ORDERED,
 * the fp32 dQ accumulator of B*H*roundup(N,128)*d floats, plus, for
 * FA_DQ_ORDERED, one 32-bit counter per 32 padded rows and a 256-byte slot for
 * the unit ticket. Returns 0 for invalid sizes or modes. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d, fa_dtype dtype, int deterministic);

/* Forward: writes O ([B, N, H, d], dtype) and lse ([B, H, N] fp32, natural
 * log). Produces the saved state the backward consumes. */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
           uint64_t seed, uint64_t offset, void* stream);

/* Backward: from Q, K, V, the forward's O and lse, and dO, writes dQ, dK, dV
 * (same dtype and strides). `deterministic` selects the dQ algorithm (FA_DQ_*
 * above; nonzero values are bit-reproducible run to run). `workspace` must be
 * 256-byte aligned and hold fa_bwd_workspace_size(...) bytes for the same
 * mode; its contents on entry do not matter. Runs fa_bwd_stage
 * (FA_BWD_PREPROCESS), (FA_BWD_DKDV), (FA_BWD_DQ) in order on `stream`; with
 * FA_DQ_RECOMPUTE the dQ kernel runs on a library-owned side stream beside the
 * dK/dV kernel, joined back into `stream` before the call returns. */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
           float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
           int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/* The three steps of fa_bwd, for callers that schedule or time them apart.
 * Arguments as fa_bwd; the stages must run in order with the same arguments.
 *  FA_BWD_PREPROCESS: D_i = rowsum(dO o O) and lse*log2(e) into the workspace;
 *                     zero-fills the dQ accumulator (FA_DQ_ATOMIC, FA_DQ_ORDERED)
 *                     and the chunk counters and unit ticket (FA_DQ_ORDERED).
 *  FA_BWD_DKDV:       key/value-major kernel: dK, dV (and the dQ adds of
 *                     FA_DQ_ATOMIC / FA_DQ_ORDERED). With FA_DQ_ORDERED it must
 *                     follow a FA_BWD_PREPROCESS on the same workspace (it
 *                     consumes the ticket the preprocess resets; a second
 *                     launch without one does no work and sets status bit 2).
 *  FA_BWD_DQ:         FA_DQ_RECOMPUTE: query-major dQ kernel; FA_DQ_ATOMIC /
 *                     FA_DQ_ORDERED: dQ = scale * accumulator, rounded to the
 *                     dtype. */
typedef enum { FA_BWD_PREPROCESS = 0, FA_BWD_DKDV = 1, FA_BWD_DQ = 2 } fa_bwd_stage_id;

int fa_bwd_stage(fa_bwd_stage_id stage, const void* q, const void* k, const void* v, const void* o,
                 const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                 uint64_t seed, uint64_t offset, int deterministic, void* workspace, size_t workspace_bytes,
                 void* stream);

/* fa_bwd_noalloc: the deterministic backward for callers that cannot allocate
 * device memory when they run it (a pre-planned memory arena that forbids new
 * allocations, a runtime recording work before any allocator exists, an
 * embedding that hands over only the tensors). The pages describe no such
 * entry point; it is this library's own. Arguments as fa_bwd, without the
 * deterministic flag (always FA_DQ_RECOMPUTE) and without a workspace: the
 * scratch (D and lse*log2(e) vectors, four unit counters) lives in one fixed
 * device array of 8 MiB + 256 bytes inside the library, so the call allocates
 * nothing. Limit:
 * B*H*roundup(N,128) <= 1048576; larger problems return FA_ERR_WORKSPACE and
 * launch nothing. All calls on a device share the array (each call overwrites
 * what it reads, nothing needs clearing); calls that overlap on the GPU race,
 * so order them. The first call on a device looks up the array's address
 * (once per device): make it before any stream capture. */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                   uint64_t seed, uint64_t offset, void* stream);

/* ---------------------------------------------------------------------------
 * Backward from host buffers: fa_bwd with Q, K, V, O, dO, L and dQ, dK, dV in
 * HOST memory (same shapes, strides, dtypes and scalars as fa_bwd; L
 * contiguous fp32 [B, H, N]). The call uploads the inputs into a caller-owned
 * device staging buffer, runs the backward there and downloads the gradients,
 * all enqueued on `stream` and asynchronous to the host: the host buffers must
 * stay valid, and the outputs are ready, once `stream` has completed the work.
 * The problem is cut into up to four groups (of heads when B = 1, of batch
 * entries otherwise) so that the upload of one group, the backward of the
 * previous one and the download of the one before run at the same time on
 * two library-owned copy streams and `stream`. Page-locked host memory
 * (cudaHostAlloc / cudaHostRegister) is needed for that overlap; pageable
 * memory is accepted, with copies that then synchronise with the host.
 * dev_buf: device memory of fa_bwd_host_buffer_size(...) bytes, 256-byte
 * aligned, owned by the caller; its contents after the call are unspecified.
 * Results equal fa_bwd's bit for bit in deterministic mode (dropout masks
 * included). Errors as fa_bwd (FA_ERR_WORKSPACE for dev_buf).
 * ------------------------------------------------------------------------- */
size_t fa_bwd_host_buffer_size(int B, int H, int N, int d, fa_dtype dtype, int deterministic);
int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
                float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
                int deterministic, void* dev_buf, size_t dev_buf_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * ALiBi position bias ("Lecture 7 — Backward Pass and Validation", §Use it in
 * the real stack, names ALiBi among the cases a complete harness covers; the
 * pages give no formula, so the usual linear bias is taken): the score of
 * query i and key j becomes scale * q_i.k_j - m * |i - j| before the mask and
 * the softmax, with m = alibi_slopes[b * alibi_stride_b + h] (fp32, device
 * memory, 4-byte aligned; alibi_stride_b = 0 shares one slope per head across
 * the batch, H otherwise for a [B, H] array). The slopes are constants: the
 * gradients keep their form with the biased P. Requires scale > 0
 * (FA_ERR_UNSUPPORTED otherwise); a null alibi_slopes is plain attention.
 * Every other argument, layout and error as fa_fwd / fa_bwd.
 * ------------------------------------------------------------------------- */
int fa_fwd_alibi(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                 uint64_t seed, uint64_t offset, const float* alibi_slopes, int64_t alibi_stride_b, void* stream);
int fa_bwd_alibi(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
                 float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
                 const float* alibi_slopes, int64_t alibi_stride_b, int deterministic, void* workspace,
                 size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Additive attention bias ("Lecture 7 — Backward Pass and Validation", §Mask
 * behaviour: custom masks enter as an attn_bias and need their own test path):
 * the score of query i and key j becomes scale * q_i.k_j + bias[b, h, i, j]
 * before the mask and the softmax; -inf entries mask pairs out (a row with
 * every key masked gets O = 0, L = -inf and no gradient). The bias is a
 * constant: no gradient is computed for it.
 * bias: device memory in the tensors' dtype, logically [B, H, N, N] with keys
 * contiguous and element strides bias_strides = {b, n (per query row), h}; a
 * stride of 0 for b or h broadcasts one plane over the batch or the heads.
 * Requires scale > 0 and bias_strides.n >= N; for 16-bit dtypes a 16-byte
 * aligned base and strides that are multiples of 8 elements (a [N, N] plane
 * with N not a multiple of 8 is passed as a view of rows padded to one;
 * FA_ERR_ALIGNMENT otherwise); fp32: a 4-byte aligned base, any strides.
 * Errors as fa_fwd / fa_bwd (FA_ERR_INVALID_ARG for a null bias).
 * ------------------------------------------------------------------------- */
int fa_fwd_bias(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                fa_strides strides, fa_dtype dtype, float scale, int causal, int window, float dropout_p,
                uint64_t seed, uint64_t offset, const void* bias, fa_strides bias_strides, void* stream);
int fa_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
                float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
                const void* bias, fa_strides bias_strides, int deterministic, void* workspace,
                size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Packed variable-length sequences ("Lecture 7 — Backward Pass and
 * Validation", §Use it in the real stack, lists varlen among the cases a
 * complete harness covers; the math per sequence is that of fa_fwd / fa_bwd).
 *
 * nseq sequences of different lengths share one packed [total, H, d] tensor
 * per operand: sequence s occupies rows [cu_seqlens[s], cu_seqlens[s+1]), and
 * attention (with the causal / window mask, positions local to the sequence)
 * never crosses a sequence boundary. cu_seqlens is a DEVICE int32 array of
 * nseq + 1 nondecreasing offsets with cu_seqlens[0] = 0, cu_seqlens[nseq] =
 * total and every length <= max_seqlen; the library cannot check device
 * contents, so it clamps offsets into [0, total] and lengths to max_seqlen (a
 * malformed array gives wrong gradients, never an out-of-bounds access).
 * stride_n / stride_h are element strides of the packed tensors (d stride 1,
 * multiples of 8). lse is contiguous fp32 [H, total]. 16-bit dtypes, d in
 * {64, 128}, nseq * H <= 65535, no dropout (dropout_p is not an argument).
 * Optional ALiBi slopes as for fa_fwd_alibi, indexed by sequence:
 * m = alibi_slopes[s * alibi_stride_seq + h] (null: no bias).
 * Errors as fa_fwd / fa_bwd; the caller owns every buffer.
 * ------------------------------------------------------------------------- */
size_t fa_varlen_bwd_workspace_size(int nseq, int max_seqlen, int total, int H, int d, fa_dtype dtype,
                                    int deterministic);
/* Forward: O [total, H, d] and lse [H, total] per sequence. */
int fa_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens, int nseq,
                  int max_seqlen, int total, int H, int d, int64_t stride_n, int64_t stride_h, fa_dtype dtype,
                  float scale, int causal, int window, const float* alibi_slopes, int64_t alibi_stride_seq,
                  void* stream);
/* Backward: dQ, dK, dV [total, H, d] per sequence; deterministic and atomic dQ
 * as fa_bwd; workspace of fa_varlen_bwd_workspace_size(...) bytes, 256-byte
 * aligned. */
int fa_varlen_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, const int* cu_seqlens, int nseq, int max_seqlen, int total, int H,
                  int d, int64_t stride_n, int64_t stride_h, fa_dtype dtype, float scale, int causal, int window,
                  const float* alibi_slopes, int64_t alibi_stride_seq, int deterministic, void* workspace,
                  size_t workspace_bytes, void* stream);

/* Reads (and with clear != 0 resets) the status word of the current device.
 * Call after synchronising the streams the kernels ran on. *status receives
 * the raw bits (1 = a bounded wait timed out; 2 = an FA_DQ_ORDERED dK/dV
 * launch found its unit ticket not reset and did nothing). Returns FA_OK, FA_ERR_TIMEOUT
 * when the timeout bit is set, or FA_ERR_CUDA. This call synchronises the device. */
int fa_get_device_status(unsigned int* status, int clear);

/* Self-test of the failure detection (the bounded waits of the tensor-core
 * kernels). Launches, on `stream`, one CTA of two warps that allocates 32 TMEM
 * columns and waits on an mbarrier that nothing arrives on: one warp with the
 * polling wait of the row-math warps, one with the blocking wait of the
 * MMA-issuing warps. After the wall-clock limit of a wait (4 s) the kernel sets
 * the timeout bit of the device status word and its CTA's abort flag, then
 * runs the bounded drain wait (another 4 s), frees its TMEM and returns, so the
 * context stays usable. `outcome` is a device int the caller zeroes; the kernel
 * ORs in bit w for each warp w whose wait gave up (3 = both). Afterwards
 * fa_get_device_status reports FA_ERR_TIMEOUT. Returns FA_OK, or FA_ERR_CUDA if
 * the launch failed. No other state is touched; about 8 s of GPU time. */
int fa_selftest_timeout(int* outcome, void* stream);

/* Static string for an FA_* code. */
const char* fa_strerror(int code);

/* Library ABI version (major*100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
