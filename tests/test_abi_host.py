"""Host-only checks of the C ABI: the library builds and loads, exports every
function include/fa.h declares, and rejects bad arguments with the documented
codes before touching any GPU (none of these calls reaches the CUDA runtime).
"""
import ctypes
import os
import shutil

import pytest

import flashattention_backward_fa_gb300 as fa
from flashattention_backward_fa_gb300 import binding

F32, F16, BF16 = fa.FA_F32, fa.FA_F16, fa.FA_BF16
OK, EINVAL, EUNSUP, EALIGN, EWS = 0, -1, -2, -3, -4


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("no nvcc to build the library")
        from flashattention_backward_fa_gb300.build import build_library
        build_library()
    return fa.load_library()


def test_exports_every_declared_function(lib):
    names = binding.header_functions()
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_strerror", "fa_bwd_stage"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_strerror(lib):
    assert lib.fa_version() >= 100
    for code in (OK, EINVAL, EUNSUP, EALIGN, EWS, -5, -6):
        s = fa.fa_strerror(code)
        assert s and s != "unknown error code"
    assert fa.fa_strerror(-99) == "unknown error code"


def _rows(N):
    return (N + 127) // 128 * 128


@pytest.mark.parametrize("B,H,N,d", [(1, 32, 8192, 128), (4, 16, 2048, 128), (2, 16, 4096, 64), (1, 1, 1, 64),
                                     (3, 5, 777, 128)])
def test_workspace_size(lib, B, H, N, d):
    r = B * H * _rows(N)
    vec = (r * 4 + 255) // 256 * 256
    ctr = 256  # the persistent kernels' unit counters
    assert fa.fa_bwd_workspace_size(B, H, N, d, BF16, True) == 2 * vec + ctr
    assert fa.fa_bwd_workspace_size(B, H, N, d, BF16, False) == 2 * vec + ctr + (r * d * 4 + 255) // 256 * 256
    assert fa.fa_bwd_workspace_size(B, H, N, d, F32, False) == 2 * vec + ctr  # fp32 never accumulates dQ atomically
    assert fa.fa_bwd_workspace_size(0, H, N, d, BF16, True) == 0
    assert fa.fa_bwd_workspace_size(B, H, N, 129, BF16, True) == 0


def _strides(N, H, d):
    return fa.FaStrides(N * H * d, H * d, d)


P = 0x10000  # a fake, 16-byte-aligned "device" address: validation rejects before any use


def _fwd(lib, *, q=P, k=P, v=P, o=P, lse=P, B=1, H=2, N=64, d=128, st=None, dt=BF16, scale=0.1, causal=0,
         window=0, p=0.0):
    st = st or _strides(N, H, d)
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, st, dt, scale, causal, window, p, 0, 0, None)


def _bwd(lib, *, ptrs=None, B=1, H=2, N=64, d=128, st=None, dt=BF16, scale=0.1, window=0, p=0.0, det=1,
         ws=0x100000, ws_bytes=1 << 30, stage=None):
    ptrs = ptrs or [P] * 9
    st = st or _strides(N, H, d)
    args = [*ptrs, B, H, N, d, st, dt, scale, 1, window, p, 0, 0, det, ws, ws_bytes, None]
    return lib.fa_bwd(*args) if stage is None else lib.fa_bwd_stage(stage, *args)


def test_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, B=0) == EINVAL
    assert _fwd(lib, N=0) == EINVAL
    assert _fwd(lib, d=96) == EUNSUP
    assert _fwd(lib, d=256) == EUNSUP
    assert _fwd(lib, dt=7) == EUNSUP
    assert _fwd(lib, dt=F32, d=129) == EUNSUP
    assert _fwd(lib, q=0) == EINVAL
    assert _fwd(lib, lse=0) == EINVAL
    assert _fwd(lib, q=P + 8) == EALIGN
    assert _fwd(lib, st=fa.FaStrides(64 * 2 * 128, 2 * 128 + 4, 128)) == EALIGN
    assert _fwd(lib, window=-1) == EINVAL
    assert _fwd(lib, p=1.0) == EINVAL
    assert _fwd(lib, p=-0.1) == EINVAL
    assert _fwd(lib, scale=float("nan")) == EINVAL
    assert _fwd(lib, st=fa.FaStrides(0, 128, 128)) == EINVAL


def test_bwd_rejects_bad_arguments(lib):
    assert _bwd(lib, B=0) == EINVAL
    assert _bwd(lib, d=32) == EUNSUP
    assert _bwd(lib, ptrs=[P] * 8 + [0]) == EINVAL
    assert _bwd(lib, ptrs=[P] * 5 + [P + 4] + [P] * 3) == EALIGN
    assert _bwd(lib, ws=0) == EWS
    assert _bwd(lib, ws=0x100000 + 128) == EWS
    need = fa.fa_bwd_workspace_size(1, 2, 64, 128, BF16, True)
    assert _bwd(lib, ws_bytes=need - 1) == EWS
    need_atomic = fa.fa_bwd_workspace_size(1, 2, 64, 128, BF16, False)
    assert _bwd(lib, det=0, ws_bytes=need) == EWS and need_atomic > need
    assert _bwd(lib, p=1.5) == EINVAL
    assert _bwd(lib, stage=7) == EINVAL
    assert _bwd(lib, stage=1, d=80) == EUNSUP


def _vfwd(lib, *, q=P, cu=P, nseq=3, msl=300, total=700, H=2, d=128, sn=256, sh=128, dt=BF16, window=0,
          alibi=None, alibi_ss=0, scale=0.1):
    return lib.fa_varlen_fwd(q, P, P, P, P, cu, nseq, msl, total, H, d, sn, sh, dt, scale, 1, window, alibi,
                             alibi_ss, None)


def _vbwd(lib, *, ptrs=None, cu=P, nseq=3, msl=300, total=700, H=2, d=128, dt=BF16, det=1, ws=0x100000,
          ws_bytes=1 << 30):
    ptrs = ptrs or [P] * 9
    return lib.fa_varlen_bwd(*ptrs, cu, nseq, msl, total, H, d, H * d, d, dt, 0.1, 1, 0, None, 0, det, ws,
                             ws_bytes, None)


def test_varlen_rejects_bad_arguments(lib):
    assert _vfwd(lib, dt=F32) == EUNSUP          # 16-bit only
    assert _vfwd(lib, d=96) == EUNSUP
    assert _vfwd(lib, cu=0) == EINVAL
    assert _vfwd(lib, cu=P + 2) == EINVAL        # int32 offsets must be 4-byte aligned
    assert _vfwd(lib, nseq=0) == EINVAL
    assert _vfwd(lib, msl=0) == EINVAL
    assert _vfwd(lib, total=0) == EINVAL
    assert _vfwd(lib, nseq=40000, H=2) == EUNSUP  # nseq * H bounded by the grid's y extent
    assert _vfwd(lib, sn=260) == EALIGN
    assert _vfwd(lib, window=-1) == EINVAL
    assert _vfwd(lib, q=0) == EINVAL
    assert _vfwd(lib, q=P + 8) == EALIGN
    assert _vbwd(lib, ptrs=[P] * 8 + [0]) == EINVAL
    assert _vbwd(lib, ws=0) == EWS
    need = fa.fa_varlen_bwd_workspace_size(3, 300, 700, 2, 128, BF16, True)
    assert _vbwd(lib, ws_bytes=need - 1) == EWS
    need_atomic = fa.fa_varlen_bwd_workspace_size(3, 300, 700, 2, 128, BF16, False)
    assert _vbwd(lib, det=0, ws_bytes=need) == EWS and need_atomic > need


def test_alibi_rejects_bad_arguments(lib):
    st = _strides(64, 2, 128)

    def fwd(alibi=P, sb=0, scale=0.1, B=1, d=128):
        a = [P] * 5 + [B, 2, 64, d, st, BF16]
        return lib.fa_fwd_alibi(*a, scale, 1, 0, 0.0, 0, 0, alibi, sb, None)
    assert fwd(alibi=P + 2) == EALIGN          # fp32 slopes, 4-byte aligned
    assert fwd(sb=-1) == EINVAL
    assert fwd(scale=0.0) == EUNSUP            # the bias folds in as m / scale
    assert fwd(scale=-0.5) == EUNSUP
    assert fwd(d=96) == EUNSUP                 # the common checks still apply
    assert fwd(B=0) == EINVAL
    assert _vfwd(lib, alibi=P + 1) == EALIGN
    assert _vfwd(lib, alibi=P, scale=0.0) == EUNSUP

    def bwd(alibi=P, sb=0, scale=0.1, ws=0x100000, ws_bytes=1 << 30):
        return lib.fa_bwd_alibi(*([P] * 9), 1, 2, 64, 128, st, BF16, scale, 1, 0, 0.0, 0, 0, alibi, sb, 1, ws,
                                ws_bytes, None)
    assert bwd(alibi=P + 2) == EALIGN
    assert bwd(scale=0.0) == EUNSUP
    assert bwd(ws=0) == EWS


def test_host_backward_rejects_bad_arguments(lib):
    st = _strides(64, 2, 128)

    def call(ptrs=None, B=1, d=128, dt=BF16, buf=0x100000, nbytes=1 << 30, p=0.0):
        ptrs = ptrs or [P] * 9
        return lib.fa_bwd_host(*ptrs, B, 2, 64, d, st, dt, 0.1, 1, 0, p, 0, 0, 1, buf, nbytes, None)
    assert call(B=0) == EINVAL
    assert call(d=96) == EUNSUP
    assert call(p=1.0) == EINVAL
    assert call(ptrs=[P] * 8 + [0]) == EINVAL
    assert call(buf=0) == EWS
    assert call(buf=0x100000 + 64) == EWS              # 256-byte alignment
    need = fa.fa_bwd_host_buffer_size(1, 2, 64, 128, BF16, True)
    assert call(nbytes=need - 1) == EWS
    # staging: 8 dense tensors, L in one 256-byte slot per group, one group's workspace
    # (B = 1: two groups of one head)
    t = 64 * 2 * 128 * 2
    assert need == 8 * t + 2 * 256 + fa.fa_bwd_workspace_size(1, 1, 64, 128, BF16, True)


def test_bias_rejects_bad_arguments(lib):
    N = 64
    st = _strides(N, 2, 128)

    def fwd(bias=P, bst=(0, N, 0), scale=0.1, dt=BF16, d=128):
        return lib.fa_fwd_bias(*([P] * 5), 1, 2, N, d, st, dt, scale, 1, 0, 0.0, 0, 0, bias, fa.FaStrides(*bst), None)
    assert fwd(bias=0) == EINVAL
    assert fwd(bst=(0, N - 8, 0)) == EINVAL      # rows must not overlap
    assert fwd(bst=(-8, N, 0)) == EINVAL
    assert fwd(scale=0.0) == EUNSUP               # folded in score units as bias / scale
    assert fwd(bias=P + 8) == EALIGN              # 16-bit: 16-byte aligned base
    assert fwd(bst=(0, N + 4, 0)) == EALIGN       # 16-bit: strides in multiples of 8 elements
    assert fwd(bst=(12, N, 0)) == EALIGN
    assert fwd(d=96) == EUNSUP
    assert fwd(dt=F32, bias=P + 2) == EALIGN      # fp32: 4-byte aligned

    def bwd(bias=P, bst=(0, N, 0), ws=0x100000):
        return lib.fa_bwd_bias(*([P] * 9), 1, 2, N, 128, st, BF16, 0.1, 1, 0, 0.0, 0, 0, bias, fa.FaStrides(*bst), 1,
                               ws, 1 << 30, None)
    assert bwd(bias=0) == EINVAL
    assert bwd(bias=P + 2) == EALIGN
    assert bwd(ws=0) == EWS


def test_varlen_workspace_size(lib):
    # L and D rows per (head, sequence), each padded to roundup(max_seqlen, 128);
    # atomic mode adds an fp32 dQ accumulator of roundup(total, 128) + 128 rows per head.
    nseq, msl, total, H, d = 3, 300, 700, 4, 128
    vec = H * nseq * 384 * 4
    vec = (vec + 255) // 256 * 256
    ctr = 256  # the persistent kernels' unit counters
    assert fa.fa_varlen_bwd_workspace_size(nseq, msl, total, H, d, BF16, True) == 2 * vec + ctr
    acc = H * (768 + 128) * d * 4
    assert fa.fa_varlen_bwd_workspace_size(nseq, msl, total, H, d, F16, False) == 2 * vec + ctr + acc
    assert fa.fa_varlen_bwd_workspace_size(nseq, msl, total, H, d, F32, True) == 0
    assert fa.fa_varlen_bwd_workspace_size(0, msl, total, H, d, BF16, True) == 0


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 1, 8)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, q, lse)


def test_oracle_not_imported_by_product_path():
    """The package never imports the oracle (its only users are tests, smoke and the bench)."""
    import pathlib
    pkg = pathlib.Path(binding.__file__).parent
    for f in pkg.rglob("*.py"):
        text = f.read_text()
        assert "import oracle" not in text and "from oracle" not in text, f


def test_size_limits_are_unsupported(lib):
    """B*H above 2^24 or N above 2^30 are refused before any pointer is used."""
    assert _fwd(lib, B=1 << 13, H=(1 << 11) + 1, N=64) == EUNSUP
    assert _bwd(lib, B=1 << 13, H=(1 << 11) + 1, N=64) == EUNSUP
    assert _fwd(lib, N=(1 << 30) + 1) == EUNSUP
    assert _bwd(lib, N=(1 << 30) + 1) == EUNSUP
