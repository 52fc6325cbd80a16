// fa_bwd_host: the backward from host buffers, with the host<->device copies
// overlapped with the computation.
//
// The problem is cut into groups that the backward treats independently:
// groups of heads when B = 1, groups of batch entries otherwise (see Split). Each group's
// inputs go up on a host-to-device copy stream, its backward runs on the
// caller's stream, and its gradients come down on a device-to-host copy
// stream, so the upload of group g + 1, the backward of group g and the
// download of group g - 1 run at the same time. Events order the three
// streams; the caller's stream waits for the last download before the call's
// work is complete. The device side lives in a caller-owned staging buffer
// (dense [B, N, H, d] copies of every tensor, L by group, and one group's
// workspace):
// the library allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_host.h"

namespace {

constexpr int kMaxDevicesHost = 64;

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t esize_of(fa_dtype dt) { return dt == FA_F32 ? 4 : 2; }

// How the problem is cut: groups of heads (B = 1) or batch entries (B > 1),
// group g covering units [first[g], first[g] + n[g]). The uploads are the
// bottleneck and what follows the last upload (the last group's backward and
// download) is exposed, so the groups shrink at the end: groups of a quarter
// of the units, then the remainder halved down to an eighth (32 heads: 8, 8,
// 8, 4, 2, 2). A group's tensors start (h0 * d) or (b0 * N * H * d) elements
// into the dense staging copies and the kernels need 16-byte aligned tensor
// pointers: where a cut would break that, the problem stays in one group.
constexpr int kMaxGroups = 8;

struct Split {
  bool by_head;
  int count, groups, max_n;
  int first[kMaxGroups], n[kMaxGroups];
};

Split make_split(int B, int H, int N, int d, fa_dtype dt) {
  Split s;
  s.by_head = B == 1;
  s.count = s.by_head ? H : B;
  const size_t step = s.by_head ? (size_t)d * esize_of(dt) : (size_t)N * H * d * esize_of(dt);
  s.groups = 0;
  auto add = [&](int n) {
    s.first[s.groups] = s.groups ? s.first[s.groups - 1] + s.n[s.groups - 1] : 0;
    s.n[s.groups++] = n;
  };
  if (step % 16 != 0 || s.count < 2) {
    add(s.count);
  } else {
    const int per = (s.count + 3) / 4, floor_n = (per + 3) / 4;
    int left = s.count;
    while (left > per && s.groups < kMaxGroups - 3) {
      add(per);
      left -= per;
    }
    // the remainder (at most `per` units, or what the group limit leaves): halve it
    while (left > 0) {
      int n = (left + 1) / 2;
      if (n < floor_n || s.groups == kMaxGroups - 1) n = left;
      add(n);
      left -= n;
    }
  }
  s.max_n = 0;
  for (int g = 0; g < s.groups; ++g) s.max_n = s.n[g] > s.max_n ? s.n[g] : s.max_n;
  return s;
}

struct StagingLayout {
  size_t tensor, off[8], off_lse, lse_group, off_ws, ws, total;  // off: q k v o dO dq dk dv
};

StagingLayout staging_layout(int B, int H, int N, int d, fa_dtype dt, int deterministic) {
  StagingLayout L;
  L.tensor = (size_t)B * N * H * d * esize_of(dt);
  size_t at = 0;
  for (int t = 0; t < 8; ++t) {
    L.off[t] = at;
    at += round256(L.tensor);
  }
  // L: one 256-byte aligned slot per group (the kernels read L through
  // 16-byte aligned pointers; a group's rows start h0 * N or b0 * H * N floats in)
  const Split s = make_split(B, H, N, d, dt);
  L.off_lse = at;
  L.lse_group = round256((size_t)(s.by_head ? s.max_n : (size_t)s.max_n * H) * N * 4);
  at += (size_t)s.groups * L.lse_group;
  L.ws = s.by_head ? fa_bwd_workspace_size(1, s.max_n, N, d, dt, deterministic)
                   : fa_bwd_workspace_size(s.max_n, H, N, d, dt, deterministic);
  L.off_ws = at;
  L.total = at + round256(L.ws);
  return L;
}

struct HostPipe {
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaEvent_t in[kMaxGroups] = {}, done[kMaxGroups] = {};
};
HostPipe g_pipe[kMaxDevicesHost];
// Guards g_pipe and serialises each call's enqueue sequence (the events are shared).
std::mutex g_pipe_mu;

int pipe_locked(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesHost) return FA_ERR_CUDA;
  HostPipe& hp = g_pipe[dev];
  if (!hp.up) {
    if (cudaStreamCreateWithFlags(&hp.up, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.down, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.join, cudaEventDisableTiming) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int g = 0; g < kMaxGroups; ++g)
      if (cudaEventCreateWithFlags(&hp.in[g], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.done[g], cudaEventDisableTiming) != cudaSuccess)
        return FA_ERR_CUDA;
  }
  *out = &hp;
  return FA_OK;
}

// Copies one group's slice of a [B, N, H, d] tensor between the host layout
// (element strides hs) and the dense device layout. Heads [h0, h0 + nh) of
// batch entries [b0, b0 + nb).
cudaError_t copy_slice(char* dev, const fa_strides& hs, char* host, int b0, int nb, int h0, int nh, int H, int N,
                       int d, size_t es, bool to_device, cudaStream_t st) {
  const size_t dev_row = (size_t)H * d * es;  // dense pitch of one position
  const cudaMemcpyKind kind = to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost;
  for (int b = b0; b < b0 + nb; ++b) {
    char* dbase = dev + ((size_t)b * N * H + h0) * d * es;
    char* hbase = host + ((size_t)b * hs.b + (size_t)h0 * hs.h) * es;
    cudaError_t e;
    if (hs.h == d) {
      // heads adjacent within a position: N rows of nh * d elements
      const size_t width = (size_t)nh * d * es, hp = (size_t)hs.n * es;
      e = to_device ? cudaMemcpy2DAsync(dbase, dev_row, hbase, hp, width, N, kind, st)
                    : cudaMemcpy2DAsync(hbase, hp, dbase, dev_row, width, N, kind, st);
      if (e != cudaSuccess) return e;
    } else {
      for (int h = 0; h < nh; ++h) {
        char* dh = dbase + (size_t)h * d * es;
        char* hh = hbase + (size_t)h * hs.h * es;
        const size_t width = (size_t)d * es, hp = (size_t)hs.n * es;
        e = to_device ? cudaMemcpy2DAsync(dh, dev_row, hh, hp, width, N, kind, st)
                      : cudaMemcpy2DAsync(hh, hp, dh, dev_row, width, N, kind, st);
        if (e != cudaSuccess) return e;
      }
    }
  }
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t fa_bwd_host_buffer_size(int B, int H, int N, int d, fa_dtype dtype, int deterministic) {
  if (fa_bwd_workspace_size(B, H, N, d, dtype, deterministic) == 0) return 0;
  return staging_layout(B, H, N, d, dtype, deterministic).total;
}

int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_strides strides, fa_dtype dtype,
                float scale, int causal, int window, float dropout_p, uint64_t seed, uint64_t offset,
                int deterministic, void* dev_buf, size_t dev_buf_bytes, void* stream) {
  int rc = fa::check_bwd_args(B, H, N, d, strides, dtype, scale, window, dropout_p);
  if (rc) return rc;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  const StagingLayout L = staging_layout(B, H, N, d, dtype, deterministic);
  if (!dev_buf || (reinterpret_cast<uintptr_t>(dev_buf) & 255u) || dev_buf_bytes < L.total) return FA_ERR_WORKSPACE;
  const Split sp = make_split(B, H, N, d, dtype);
  const size_t es = esize_of(dtype);
  char* base = static_cast<char*>(dev_buf);
  const fa_strides dense = {(int64_t)N * H * d, (int64_t)H * d, (int64_t)d};
  const void* hin[5] = {q, k, v, o, dout};
  void* hout[3] = {dq, dk, dv};
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* hp = nullptr;
  if ((rc = pipe_locked(&hp))) return rc;
  // Everything already queued on the caller's stream (earlier users of the
  // staging buffer) precedes the uploads.
  if (cudaEventRecord(hp->fork, st) != cudaSuccess || cudaStreamWaitEvent(hp->up, hp->fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->down, hp->fork, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  for (int g = 0; g < sp.groups; ++g) {
    const int first = sp.first[g], n = sp.n[g];
    const int b0 = sp.by_head ? 0 : first, nb = sp.by_head ? 1 : n;
    const int h0 = sp.by_head ? first : 0, nh = sp.by_head ? n : H;
    // upload: the five [B, N, H, d] inputs and L rows of the group
    for (int t = 0; t < 5; ++t)
      if (copy_slice(base + L.off[t], strides, const_cast<char*>(static_cast<const char*>(hin[t])), b0, nb, h0, nh,
                     H, N, d, es, true, hp->up) != cudaSuccess)
        return FA_ERR_CUDA;
    const size_t lse_first = ((size_t)b0 * H + h0) * N, lse_count = (size_t)nb * nh * N;  // contiguous
    float* lse_dev = reinterpret_cast<float*>(base + L.off_lse + (size_t)g * L.lse_group);
    if (cudaMemcpyAsync(lse_dev, lse + lse_first, lse_count * 4, cudaMemcpyHostToDevice, hp->up) != cudaSuccess ||
        cudaEventRecord(hp->in[g], hp->up) != cudaSuccess || cudaStreamWaitEvent(st, hp->in[g], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    // backward of the group on the caller's stream (groups share the workspace, in stream order)
    const size_t elem0 = ((size_t)b0 * N * H + h0) * d * es;
    auto at = [&](int t) { return static_cast<void*>(base + L.off[t] + elem0); };
    fa::Extras ex;
    ex.philox_bh_off = (uint32_t)(b0 * H + h0);
    rc = fa::bwd_run(at(0), at(1), at(2), at(3), at(4), lse_dev,
                     at(5), at(6), at(7), nb, nh, N, d, dense, dtype, scale, causal, window, dropout_p, seed, offset,
                     ex, deterministic, base + L.off_ws, L.ws, stream, true);
    if (rc) return rc;
    // download: the group's dQ, dK, dV
    if (cudaEventRecord(hp->done[g], st) != cudaSuccess || cudaStreamWaitEvent(hp->down, hp->done[g], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int t = 0; t < 3; ++t)
      if (copy_slice(base + L.off[5 + t], strides, static_cast<char*>(hout[t]), b0, nb, h0, nh, H, N, d, es, false,
                     hp->down) != cudaSuccess)
        return FA_ERR_CUDA;
  }
  if (cudaEventRecord(hp->join, hp->down) != cudaSuccess || cudaStreamWaitEvent(st, hp->join, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
