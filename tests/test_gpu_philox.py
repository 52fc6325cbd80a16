"""Dropout generator pins on a GPU.

* The oracle's Philox4x32-10 (written from Salmon et al., SC'11) against
  cuRAND's device Philox4_32_10: curand_init(seed, subsequence, 4*g) followed
  by curand4() yields the generator output at counter (lo32(g), hi32(g),
  lo32(subsequence), hi32(subsequence)) with key (lo32(seed), hi32(seed)),
  which is this library's layout with subsequence = offset.
* The keep-masks the kernels apply, recovered exactly with identity probes
  (V = I in the forward gives O = P~; dO = I in the backward gives dV^T = P~),
  against the oracle's keep_mask, bit for bit.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import flashattention_backward_fa_gb300 as fa
from gpu_check import DQ_IDS, DQ_MODES
import oracle

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def curand_lib(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("curand") / "libcurand_words.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    os.path.join(HERE, "cuda", "curand_philox_words.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.curand_philox_words.argtypes = [ctypes.c_ulonglong, ctypes.c_ulonglong, ctypes.c_ulonglong, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_uint)]
    return lib


@pytest.mark.parametrize("seed,subseq,g0", [(0, 0, 0), (1234, 0, 0), ((7 << 32) | 99, (5 << 32) | 11, 123456789),
                                            (2 ** 64 - 1, 2 ** 64 - 1, 2 ** 40)])
def test_oracle_philox_matches_curand(curand_lib, seed, subseq, g0):
    n = 4096
    buf = (ctypes.c_uint * (4 * n))()
    assert curand_lib.curand_philox_words(seed, subseq, g0, n, buf) == 0
    got = np.frombuffer(buf, dtype=np.uint32).reshape(n, 4)
    g = np.uint64(g0) + np.arange(n, dtype=np.uint64)
    words = oracle.philox4x32_10(g & np.uint64(0xFFFFFFFF), g >> np.uint64(32), subseq & 0xFFFFFFFF, subseq >> 32,
                                 seed & 0xFFFFFFFF, seed >> 32)
    np.testing.assert_array_equal(got, np.stack(words, axis=1))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_forward_mask_bit_exact(dtype):
    """V = I (N = d): O = P o Z / (1 - p), so the kept set is where O != 0."""
    B, H, N, d, p, seed, off = 2, 3, 64, 64, 0.3, 987654321, 17
    g = torch.Generator().manual_seed(5)
    q = (0.1 * torch.randn(B, N, H, d, generator=g)).to(dtype).cuda()
    k = (0.1 * torch.randn(B, N, H, d, generator=g)).to(dtype).cuda()
    v = torch.eye(N, d).reshape(1, N, 1, d).expand(B, N, H, d).contiguous().to(dtype).cuda()
    o, _ = fa.attention_forward(q, k, v, dropout_p=p, seed=seed, offset=off)
    got = (o.float().cpu() != 0).numpy()
    for b in range(B):
        for h in range(H):
            z = oracle.keep_mask(b, h, H, N, np.arange(N), seed, off, p)
            np.testing.assert_array_equal(got[b, :, h, :], z)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_backward_mask_bit_exact(dtype):
    """dO = I (N = d): dV_j = sum_i P~_ij e_i, so dV[j, i] != 0 exactly where (i, j) is kept."""
    B, H, N, d, p, seed, off = 1, 2, 64, 64, 0.25, 31337, 5
    g = torch.Generator().manual_seed(6)
    q = (0.1 * torch.randn(B, N, H, d, generator=g)).to(dtype).cuda()
    k = (0.1 * torch.randn(B, N, H, d, generator=g)).to(dtype).cuda()
    v = torch.randn(B, N, H, d, generator=g).to(dtype).cuda()
    do = torch.eye(N, d).reshape(1, N, 1, d).expand(B, N, H, d).contiguous().to(dtype).cuda()
    o, lse = fa.attention_forward(q, k, v, dropout_p=p, seed=seed, offset=off)
    for det in DQ_MODES:
        _, _, dv = fa.attention_backward(q, k, v, o, do, lse, dropout_p=p, seed=seed, offset=off, deterministic=det)
        got = (dv.float().cpu() != 0).numpy()
        for h in range(H):
            z = oracle.keep_mask(0, h, H, N, np.arange(N), seed, off, p)
            np.testing.assert_array_equal(got[0, :, h, :].T, z)
