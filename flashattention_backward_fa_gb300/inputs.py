"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random tensors and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can consume its
output without sharing any of the method's code.

Recipe (the same on every machine, because it runs on the CPU generator):
one ``torch.Generator`` per workload seeded with the workload's seed; Q, K, V
and dO are drawn in that order as float32 ``randn`` in [B, N, H, d] order,
dO optionally multiplied by a constant in float32, then each is rounded to the
working dtype (round to nearest even).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    """One attention shape with its mask, dropout and input-generation settings."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "f32" | "f16" | "bf16"
    causal: bool = False
    window: int = 0
    dropout_p: float = 0.0
    philox_seed: int = 0
    philox_offset: int = 0
    input_seed: int = 0
    dout_std: float = 1.0
    notes: str = field(default="", compare=False)

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DTYPES[self.dtype]

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d), rounded to float32 as the host computes it."""
        return float(torch.tensor(1.0, dtype=torch.float32) / torch.sqrt(torch.tensor(float(self.d), dtype=torch.float32)))

    def with_(self, **kw) -> "Workload":
        args = {f: getattr(self, f) for f in self.__dataclass_fields__}
        args.update(kw)
        return Workload(**args)


# The five workloads of this library's parity and performance plan.
WORKLOADS = {
    "fp32_n128_d64": Workload("fp32_n128_d64", 1, 1, 128, 64, "f32", input_seed=0),
    "bf16_causal_b4h16_n2048_d128": Workload("bf16_causal_b4h16_n2048_d128", 4, 16, 2048, 128, "bf16",
                                             causal=True, input_seed=1),
    "bf16_causal_b1h32_n8192_d128": Workload("bf16_causal_b1h32_n8192_d128", 1, 32, 8192, 128, "bf16",
                                             causal=True, input_seed=2),
    "bf16_causal_b1h8_n32768_d128": Workload("bf16_causal_b1h8_n32768_d128", 1, 8, 32768, 128, "bf16",
                                             causal=True, input_seed=3, dout_std=0.01),
    "fp16_window1024_drop0.1_b2h16_n4096_d64": Workload(
        "fp16_window1024_drop0.1_b2h16_n4096_d64", 2, 16, 4096, 64, "f16", causal=True, window=1024,
        dropout_p=0.1, philox_seed=1234, philox_offset=0, input_seed=4),
}
HEADLINE = "bf16_causal_b1h32_n8192_d128"


def make_inputs(w: Workload, device: str = "cpu"):
    """Return (q, k, v, do) as [B, N, H, d] tensors of the workload's dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.input_seed))
    shape = (w.B, w.N, w.H, w.d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.dout_std != 1.0:
        do = do * torch.tensor(w.dout_std, dtype=torch.float32)
    dt = w.torch_dtype
    return tuple(t.to(dt).to(device) for t in (q, k, v, do))


def head_subset(w: Workload, heads):
    """Slice a workload's inputs to some heads (the oracle checks large ones per head)."""
    return w.with_(H=len(heads))


def make_varlen_inputs(lengths, H: int, d: int, dtype: str, seed: int = 0, dout_std: float = 1.0):
    """Packed variable-length inputs: (q, k, v, do) as [total, H, d] tensors of
    ``dtype`` plus cu_seqlens (int32, nseq + 1 offsets), drawn like
    :func:`make_inputs` with the packed shape."""
    lengths = [int(n) for n in lengths]
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (int(cu[-1]), H, d)
    q, k, v, do = (torch.randn(shape, generator=g, dtype=torch.float32) for _ in range(4))
    if dout_std != 1.0:
        do = do * torch.tensor(dout_std, dtype=torch.float32)
    dt = _DTYPES[dtype]
    return q.to(dt), k.to(dt), v.to(dt), do.to(dt), cu


def varlen_lengths(nseq: int, max_seqlen: int, seed: int = 0, min_seqlen: int = 1):
    """A seeded length mix: nseq lengths uniform on [min_seqlen, max_seqlen]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randint(min_seqlen, max_seqlen + 1, (nseq,), generator=g).tolist()
