"""Thin ctypes binding over libfa.so (the C ABI declared in include/fa.h).

Argument marshalling only: shapes, strides and pointers of torch tensors are
passed to the C entry points, which validate them and launch the CUDA kernels
on the caller's current stream. torch supplies device memory and streams;
every step of the computation runs in the library's kernels. There is no
fallback: if the library is missing or the tensors are not on a CUDA device,
these functions raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libfa.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fa.h")

FA_F32, FA_F16, FA_BF16 = 0, 1, 2
FA_BWD_PREPROCESS, FA_BWD_DKDV, FA_BWD_DQ = 0, 1, 2
# dQ algorithms (the `deterministic` argument of the backward calls, fa.h FA_DQ_*)
FA_DQ_ATOMIC, FA_DQ_DETERMINISTIC, FA_DQ_RECOMPUTE, FA_DQ_ORDERED = 0, 1, 2, 3


def _dq_mode(deterministic) -> int:
    """A `deterministic` argument as the C ABI's dQ mode: True / False are
    FA_DQ_DETERMINISTIC / FA_DQ_ATOMIC; integers pass through (FA_DQ_*)."""
    if isinstance(deterministic, bool):
        return FA_DQ_DETERMINISTIC if deterministic else FA_DQ_ATOMIC
    mode = int(deterministic)
    if mode not in (FA_DQ_ATOMIC, FA_DQ_DETERMINISTIC, FA_DQ_RECOMPUTE, FA_DQ_ORDERED):
        raise ValueError(f"deterministic must be a bool or one of FA_DQ_* (0..3), not {deterministic!r}")
    return mode
ERROR_CODES = {
    0: "FA_OK", -1: "FA_ERR_INVALID_ARG", -2: "FA_ERR_UNSUPPORTED", -3: "FA_ERR_ALIGNMENT",
    -4: "FA_ERR_WORKSPACE", -5: "FA_ERR_CUDA", -6: "FA_ERR_TIMEOUT",
}
_TORCH_TO_FA = {torch.float32: FA_F32, torch.float16: FA_F16, torch.bfloat16: FA_BF16}


class FaStrides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("n", ctypes.c_int64), ("h", ctypes.c_int64)]


class FaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_CODES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libfa.so and declare the C signatures; raises if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libfa.so not found at {path}: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i, f, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t
    lib.fa_version.argtypes, lib.fa_version.restype = [], i
    lib.fa_strerror.argtypes, lib.fa_strerror.restype = [i], ctypes.c_char_p
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, FaStrides, i, f, i, i, f, u64, u64, vp]
    lib.fa_fwd.restype = i
    bwd_args = [vp] * 9 + [i, i, i, i, FaStrides, i, f, i, i, f, u64, u64, i, vp, sz, vp]
    lib.fa_bwd.argtypes, lib.fa_bwd.restype = bwd_args, i
    lib.fa_bwd_stage.argtypes, lib.fa_bwd_stage.restype = [i] + bwd_args, i
    lib.fa_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i]
    lib.fa_get_device_status.restype = i
    lib.fa_selftest_timeout.argtypes, lib.fa_selftest_timeout.restype = [vp, vp], i
    lib.fa_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, FaStrides, i, f, i, i, f, u64, u64, vp]
    lib.fa_bwd_noalloc.restype = i
    i64 = ctypes.c_int64
    lib.fa_varlen_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.fa_varlen_bwd_workspace_size.restype = sz
    lib.fa_varlen_fwd.argtypes = [vp] * 6 + [i, i, i, i, i, i64, i64, i, f, i, i, vp, i64, vp]
    lib.fa_varlen_fwd.restype = i
    lib.fa_varlen_bwd.argtypes = [vp] * 10 + [i, i, i, i, i, i64, i64, i, f, i, i, vp, i64, i, vp, sz, vp]
    lib.fa_varlen_bwd.restype = i
    lib.fa_bwd_host_buffer_size.argtypes = [i, i, i, i, i, i]
    lib.fa_bwd_host_buffer_size.restype = sz
    lib.fa_bwd_host.argtypes = bwd_args
    lib.fa_bwd_host.restype = i
    lib.fa_fwd_bias.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, FaStrides, i, f, i, i, f, u64, u64, vp, FaStrides,
                                vp]
    lib.fa_fwd_bias.restype = i
    lib.fa_bwd_bias.argtypes = [vp] * 9 + [i, i, i, i, FaStrides, i, f, i, i, f, u64, u64, vp, FaStrides, i, vp,
                                           sz, vp]
    lib.fa_bwd_bias.restype = i
    lib.fa_fwd_alibi.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, FaStrides, i, f, i, i, f, u64, u64, vp, i64, vp]
    lib.fa_fwd_alibi.restype = i
    lib.fa_bwd_alibi.argtypes = [vp] * 9 + [i, i, i, i, FaStrides, i, f, i, i, f, u64, u64, vp, i64, i, vp, sz,
                                            vp]
    lib.fa_bwd_alibi.restype = i
    _lib = lib
    return lib


def header_functions(path: str = HEADER_PATH):
    """Names of the functions include/fa.h declares (used to check the exports)."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def fa_strerror(code: int) -> str:
    return load_library().fa_strerror(int(code)).decode()


def _check(code: int):
    if code != 0:
        raise FaError(code, fa_strerror(code))


def _layout(t: torch.Tensor):
    if t.dim() != 4:
        raise ValueError("attention tensors are [B, N, H, d]")
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if t.stride(3) != 1:
        raise ValueError("the head dimension must be contiguous")
    B, N, H, d = t.shape
    return (B, N, H, d), FaStrides(t.stride(0), t.stride(1), t.stride(2))


def _same_layout(ref: torch.Tensor, *others: torch.Tensor):
    shp, st = _layout(ref)
    for o in others:
        s2, st2 = _layout(o)
        if s2 != shp or (st2.b, st2.n, st2.h) != (st.b, st.n, st.h) or o.dtype != ref.dtype:
            raise ValueError("all [B, N, H, d] tensors must share shape, strides and dtype")
        if o.device != ref.device:
            raise ValueError("all tensors must live on the same CUDA device")
    if ref.device.index is not None and ref.device.index != torch.cuda.current_device():
        raise ValueError(f"tensors live on {ref.device} but the current device is cuda:{torch.cuda.current_device()}"
                         " (use torch.cuda.device(...))")
    return shp, st


def _on_device(t: torch.Tensor, ref: torch.Tensor, name: str):
    if not t.is_cuda or t.device != ref.device:
        raise ValueError(f"{name} must be a CUDA tensor on {ref.device}")


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _alibi(slopes, lead: int, H: int, device):
    """(pointer, lead stride) of ALiBi slopes shaped [H] or [lead, H] (fp32 CUDA), or (None, 0)."""
    if slopes is None:
        return None, 0
    if slopes.dtype != torch.float32 or not slopes.is_cuda or slopes.device != device:
        raise ValueError("alibi_slopes must be a float32 tensor on the tensors' device")
    if slopes.dim() == 1 and slopes.shape[0] == H and slopes.stride(0) == 1:
        return slopes.data_ptr(), 0
    if slopes.dim() == 2 and tuple(slopes.shape) == (lead, H) and slopes.stride(1) == 1:
        return slopes.data_ptr(), slopes.stride(0)
    raise ValueError(f"alibi_slopes must be [H] or [{lead}, H] with a contiguous head dimension")


def _bias(bias, q):
    """(pointer, FaStrides(b, n, h)) of an attention bias shaped [B or 1, H or 1, N, N]."""
    B, N, H, _ = q.shape
    if bias.dtype != q.dtype or not bias.is_cuda or bias.device != q.device:
        raise ValueError("attn_bias must be a CUDA tensor of the tensors' dtype on their device")
    if bias.dim() != 4 or bias.shape[0] not in (1, B) or bias.shape[1] not in (1, H) or \
            tuple(bias.shape[2:]) != (N, N) or bias.stride(3) != 1:
        raise ValueError(f"attn_bias must be [B or 1, H or 1, {N}, {N}] with contiguous keys")
    sb = bias.stride(0) if bias.shape[0] > 1 else 0
    sh = bias.stride(1) if bias.shape[1] > 1 else 0
    return bias.data_ptr(), FaStrides(sb, bias.stride(2), sh)


def default_scale(d: int) -> float:
    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int, dtype, deterministic: bool = True) -> int:
    code = _TORCH_TO_FA[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load_library().fa_bwd_workspace_size(B, H, N, d, code, _dq_mode(deterministic)))


def fa_fwd(q, k, v, o, lse, scale=None, causal=False, window=0, dropout_p=0.0, seed=0, offset=0, stream=None,
           alibi_slopes=None, attn_bias=None):
    """Forward through the C ABI: fills o ([B,N,H,d]) and lse ([B,H,N] fp32).

    ``alibi_slopes`` (fp32 [H] or [B, H]) adds -m|i - j| to the scaled scores (fa_fwd_alibi).
    """
    (B, N, H, d), st = _same_layout(q, k, v, o)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    _on_device(lse, q, "lse")
    lib = load_library()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, st,
            _TORCH_TO_FA[q.dtype], default_scale(d) if scale is None else float(scale), int(causal), int(window),
            float(dropout_p), int(seed), int(offset))
    if alibi_slopes is not None and attn_bias is not None:
        raise ValueError("pass either alibi_slopes or attn_bias (fold ALiBi into the bias to combine them)")
    if attn_bias is not None:
        _check(lib.fa_fwd_bias(*args, *_bias(attn_bias, q), _stream(stream)))
    elif alibi_slopes is None:
        _check(lib.fa_fwd(*args, _stream(stream)))
    else:
        _check(lib.fa_fwd_alibi(*args, *_alibi(alibi_slopes, B, H, q.device), _stream(stream)))


def _bwd_args(q, k, v, o, do, lse, dq, dk, dv, scale, causal, window, dropout_p, seed, offset, deterministic,
              workspace, stream):
    (B, N, H, d), st = _same_layout(q, k, v, o, do, dq, dk, dv)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    _on_device(lse, q, "lse")
    _on_device(workspace, q, "workspace")
    return (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr(), B, H, N, d, st, _TORCH_TO_FA[q.dtype],
            default_scale(d) if scale is None else float(scale), int(causal), int(window), float(dropout_p),
            int(seed), int(offset), _dq_mode(deterministic), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream(stream))


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, scale=None, causal=False, window=0, dropout_p=0.0,
           seed=0, offset=0, deterministic=True, stream=None, alibi_slopes=None, attn_bias=None):
    """Backward through the C ABI: fills dq, dk, dv. ``workspace`` is a uint8 CUDA tensor.

    ``alibi_slopes`` as for :func:`fa_fwd` (fa_bwd_alibi)."""
    a = _bwd_args(q, k, v, o, do, lse, dq, dk, dv, scale, causal, window, dropout_p, seed, offset, deterministic,
                  workspace, stream)
    if alibi_slopes is not None and attn_bias is not None:
        raise ValueError("pass either alibi_slopes or attn_bias (fold ALiBi into the bias to combine them)")
    if attn_bias is not None:
        _check(load_library().fa_bwd_bias(*a[:21], *_bias(attn_bias, q), *a[21:]))
    elif alibi_slopes is None:
        _check(load_library().fa_bwd(*a))
    else:
        # fa_bwd_alibi takes the slopes before `deterministic`
        _check(load_library().fa_bwd_alibi(*a[:21], *_alibi(alibi_slopes, q.shape[0], q.shape[2], q.device),
                                           *a[21:]))


def fa_bwd_stage(stage, q, k, v, o, do, lse, dq, dk, dv, workspace, scale=None, causal=False, window=0,
                 dropout_p=0.0, seed=0, offset=0, deterministic=True, stream=None):
    """One of the three backward steps (FA_BWD_PREPROCESS, FA_BWD_DKDV, FA_BWD_DQ)."""
    _check(load_library().fa_bwd_stage(int(stage), *_bwd_args(q, k, v, o, do, lse, dq, dk, dv, scale, causal,
                                                              window, dropout_p, seed, offset, deterministic,
                                                              workspace, stream)))


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, scale=None, causal=False, window=0, dropout_p=0.0, seed=0,
                   offset=0, stream=None):
    """Deterministic backward with the library's fixed internal scratch instead of a workspace.

    For callers that cannot allocate device memory when they run the backward.
    Limit B*H*roundup(N,128) <= 1048576; calls sharing a device must not overlap.
    """
    (B, N, H, d), st = _same_layout(q, k, v, o, do, dq, dk, dv)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    _on_device(lse, q, "lse")
    _check(load_library().fa_bwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
        dk.data_ptr(), dv.data_ptr(), B, H, N, d, st, _TORCH_TO_FA[q.dtype],
        default_scale(d) if scale is None else float(scale), int(causal), int(window), float(dropout_p), int(seed),
        int(offset), _stream(stream)))


def _host_layout(ref: torch.Tensor, *others: torch.Tensor):
    if ref.dim() != 4 or ref.is_cuda or ref.stride(3) != 1:
        raise ValueError("host tensors are CPU [B, N, H, d] with a contiguous head dimension")
    for o in others:
        if o.is_cuda or tuple(o.shape) != tuple(ref.shape) or o.stride() != ref.stride() or o.dtype != ref.dtype:
            raise ValueError("all host [B, N, H, d] tensors must share shape, strides and dtype")
    B, N, H, d = ref.shape
    return (B, N, H, d), FaStrides(ref.stride(0), ref.stride(1), ref.stride(2))


def fa_bwd_host_buffer_size(B: int, H: int, N: int, d: int, dtype, deterministic: bool = True) -> int:
    code = _TORCH_TO_FA[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load_library().fa_bwd_host_buffer_size(B, H, N, d, code, _dq_mode(deterministic)))


def fa_bwd_host(q, k, v, o, do, lse, dq, dk, dv, dev_buf, scale=None, causal=False, window=0, dropout_p=0.0,
                seed=0, offset=0, deterministic=True, stream=None):
    """Backward from host (CPU) tensors through fa_bwd_host: uploads, computes and downloads
    on ``stream`` with the copies overlapped; pin the host tensors for that overlap.
    ``dev_buf`` is a uint8 CUDA tensor of fa_bwd_host_buffer_size(...) bytes. The outputs
    are ready once the stream has completed the work."""
    (B, N, H, d), st = _host_layout(q, k, v, o, do, dq, dk, dv)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous() or lse.is_cuda:
        raise ValueError("lse must be a contiguous float32 CPU [B, H, N] tensor")
    if not dev_buf.is_cuda or dev_buf.device.index not in (None, torch.cuda.current_device()):
        raise ValueError("dev_buf must be device memory of the current device")
    _check(load_library().fa_bwd_host(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
        dk.data_ptr(), dv.data_ptr(), B, H, N, d, st, _TORCH_TO_FA[q.dtype],
        default_scale(d) if scale is None else float(scale), int(causal), int(window), float(dropout_p), int(seed),
        int(offset), _dq_mode(deterministic), dev_buf.data_ptr(), dev_buf.numel() * dev_buf.element_size(),
        _stream(stream)))


def fa_get_device_status(clear: bool = True) -> int:
    """Raw device status bits of the current device (synchronises it)."""
    s = ctypes.c_uint(0)
    code = load_library().fa_get_device_status(ctypes.byref(s), int(clear))
    if code not in (0, -6):
        _check(code)
    return int(s.value)


def fa_selftest_timeout(device=None, stream=None) -> int:
    """Run the bounded-wait self-test kernel (about 8 s) and return its outcome bits.

    Bit w is set when warp w's wait gave up (3 = both). The device status word
    then carries the timeout bit: read and clear it with fa_get_device_status().
    """
    outcome = torch.zeros(1, dtype=torch.int32, device=device if device is not None else "cuda")
    _check(load_library().fa_selftest_timeout(outcome.data_ptr(), _stream(stream)))
    return int(outcome.item())


def alloc_workspace(q: torch.Tensor, deterministic: bool = True) -> torch.Tensor:
    B, N, H, d = q.shape
    nbytes = fa_bwd_workspace_size(B, H, N, d, q.dtype, deterministic)
    return torch.empty(nbytes, dtype=torch.uint8, device=q.device)


def attention_forward(q, k, v, scale=None, causal=False, window=0, dropout_p=0.0, seed=0, offset=0,
                      alibi_slopes=None, attn_bias=None):
    """Allocate O and L and run the forward; returns (o, lse)."""
    B, N, H, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, scale, causal, window, dropout_p, seed, offset, alibi_slopes=alibi_slopes,
           attn_bias=attn_bias)
    return o, lse


def attention_backward(q, k, v, o, do, lse, scale=None, causal=False, window=0, dropout_p=0.0, seed=0, offset=0,
                       deterministic=True, workspace=None, alibi_slopes=None, attn_bias=None):
    """Allocate dQ, dK, dV (and the workspace unless given) and run the backward."""
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = alloc_workspace(q, deterministic)
    fa_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, scale, causal, window, dropout_p, seed, offset,
           deterministic, alibi_slopes=alibi_slopes, attn_bias=attn_bias)
    return dq, dk, dv


# ----------------------- packed variable-length input -----------------------
def _varlen_layout(ref: torch.Tensor, cu_seqlens: torch.Tensor, *others: torch.Tensor):
    """Checks packed [total, H, d] tensors and the int32 cu_seqlens; returns (total, H, d, sn, sh, nseq)."""
    if ref.dim() != 3 or not ref.is_cuda or ref.stride(2) != 1:
        raise ValueError("packed tensors are CUDA [total, H, d] with a contiguous head dimension")
    for o in others:
        if tuple(o.shape) != tuple(ref.shape) or o.stride() != ref.stride() or o.dtype != ref.dtype:
            raise ValueError("all packed tensors must share shape, strides and dtype")
        _on_device(o, ref, "every packed tensor")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_cuda \
            or not cu_seqlens.is_contiguous() or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a contiguous int32 CUDA tensor of nseq + 1 offsets")
    _on_device(cu_seqlens, ref, "cu_seqlens")
    total, H, d = ref.shape
    return total, H, d, ref.stride(0), ref.stride(1), cu_seqlens.numel() - 1


def _varlen_lse_check(lse, H, total):
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, total) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [H, total] tensor")


def fa_varlen_bwd_workspace_size(nseq: int, max_seqlen: int, total: int, H: int, d: int, dtype,
                                 deterministic: bool = True) -> int:
    code = _TORCH_TO_FA[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load_library().fa_varlen_bwd_workspace_size(nseq, max_seqlen, total, H, d, code,
                                                           _dq_mode(deterministic)))


def fa_varlen_fwd(q, k, v, o, lse, cu_seqlens, max_seqlen, scale=None, causal=False, window=0, stream=None,
                  alibi_slopes=None):
    """Forward over packed sequences: fills o ([total, H, d]) and lse ([H, total] fp32).

    ``alibi_slopes``: fp32 [H] or [nseq, H], or None."""
    total, H, d, sn, sh, nseq = _varlen_layout(q, cu_seqlens, k, v, o)
    _varlen_lse_check(lse, H, total)
    _check(load_library().fa_varlen_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), cu_seqlens.data_ptr(), nseq,
        int(max_seqlen), total, H, d, sn, sh, _TORCH_TO_FA[q.dtype], default_scale(d) if scale is None else
        float(scale), int(causal), int(window), *_alibi(alibi_slopes, nseq, H, q.device), _stream(stream)))


def fa_varlen_bwd(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens, max_seqlen, workspace, scale=None, causal=False,
                  window=0, deterministic=True, stream=None, alibi_slopes=None):
    """Backward over packed sequences: fills dq, dk, dv. ``workspace`` is a uint8 CUDA tensor."""
    total, H, d, sn, sh, nseq = _varlen_layout(q, cu_seqlens, k, v, o, do, dq, dk, dv)
    _varlen_lse_check(lse, H, total)
    _check(load_library().fa_varlen_bwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
        dk.data_ptr(), dv.data_ptr(), cu_seqlens.data_ptr(), nseq, int(max_seqlen), total, H, d, sn, sh,
        _TORCH_TO_FA[q.dtype], default_scale(d) if scale is None else float(scale), int(causal), int(window),
        *_alibi(alibi_slopes, nseq, H, q.device), _dq_mode(deterministic), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def varlen_attention_forward(q, k, v, cu_seqlens, max_seqlen, scale=None, causal=False, window=0,
                             alibi_slopes=None):
    """Allocate O and L and run the packed forward; returns (o, lse)."""
    total, H, _ = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    fa_varlen_fwd(q, k, v, o, lse, cu_seqlens, max_seqlen, scale, causal, window, alibi_slopes=alibi_slopes)
    return o, lse


def varlen_attention_backward(q, k, v, o, do, lse, cu_seqlens, max_seqlen, scale=None, causal=False, window=0,
                              deterministic=True, alibi_slopes=None):
    """Allocate dQ, dK, dV and the workspace and run the packed backward."""
    total, H, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = fa_varlen_bwd_workspace_size(cu_seqlens.numel() - 1, max_seqlen, total, H, d, q.dtype, deterministic)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    fa_varlen_bwd(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens, max_seqlen, ws, scale, causal, window,
                  deterministic, alibi_slopes=alibi_slopes)
    return dq, dk, dv


class _FlashAttnFunc(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, scale, causal, window, dropout_p, seed, offset, deterministic, alibi_slopes, attn_bias):
        o, lse = attention_forward(q, k, v, scale, causal, window, dropout_p, seed, offset, alibi_slopes, attn_bias)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.cfg = (scale, causal, window, dropout_p, seed, offset, deterministic, alibi_slopes, attn_bias)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        scale, causal, window, dropout_p, seed, offset, deterministic, alibi_slopes, attn_bias = ctx.cfg
        if do.stride() != q.stride():
            do = _match_layout(do, q)
        dq, dk, dv = attention_backward(q, k, v, o, do, lse, scale, causal, window, dropout_p, seed, offset,
                                        deterministic, alibi_slopes=alibi_slopes, attn_bias=attn_bias)
        return dq, dk, dv, None, None, None, None, None, None, None, None, None


def _match_layout(t: torch.Tensor, ref: torch.Tensor) -> torch.Tensor:
    out = torch.empty_strided(ref.shape, ref.stride(), dtype=ref.dtype, device=ref.device)
    out.copy_(t)
    return out


def flash_attn_func(q, k, v, causal=False, window=0, dropout_p=0.0, softmax_scale=None, seed=0, offset=0,
                    deterministic=True, alibi_slopes=None, attn_bias=None):
    """Attention on [B, S, H, D] tensors with autograd (forward fa_fwd, backward fa_bwd).

    ``alibi_slopes`` (fp32 [H] or [B, H]) adds -m|i - j| to the scaled scores; ``attn_bias``
    ([B or 1, H or 1, S, S], the tensors' dtype, -inf masks) adds itself. Neither is differentiated."""
    k = k if k.stride() == q.stride() else _match_layout(k, q)
    v = v if v.stride() == q.stride() else _match_layout(v, q)
    return _FlashAttnFunc.apply(q, k, v, softmax_scale, causal, window, dropout_p, seed, offset, deterministic,
                                alibi_slopes, attn_bias)


class _FlashAttnVarlenFunc(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens, max_seqlen, scale, causal, window, deterministic, alibi_slopes):
        o, lse = varlen_attention_forward(q, k, v, cu_seqlens, max_seqlen, scale, causal, window, alibi_slopes)
        ctx.save_for_backward(q, k, v, o, lse, cu_seqlens)
        ctx.cfg = (max_seqlen, scale, causal, window, deterministic, alibi_slopes)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, cu_seqlens = ctx.saved_tensors
        max_seqlen, scale, causal, window, deterministic, alibi_slopes = ctx.cfg
        if do.stride() != q.stride():
            do = _match_layout(do, q)
        dq, dk, dv = varlen_attention_backward(q, k, v, o, do, lse, cu_seqlens, max_seqlen, scale, causal, window,
                                               deterministic, alibi_slopes)
        return dq, dk, dv, None, None, None, None, None, None, None


def flash_attn_varlen_func(q, k, v, cu_seqlens, max_seqlen, causal=False, window=0, softmax_scale=None,
                           deterministic=True, alibi_slopes=None):
    """Attention over packed sequences ([total, H, D] tensors, int32 cu_seqlens on the
    device) with autograd (forward fa_varlen_fwd, backward fa_varlen_bwd)."""
    k = k if k.stride() == q.stride() else _match_layout(k, q)
    v = v if v.stride() == q.stride() else _match_layout(v, q)
    return _FlashAttnVarlenFunc.apply(q, k, v, cu_seqlens, int(max_seqlen), softmax_scale, causal, window,
                                      deterministic, alibi_slopes)
