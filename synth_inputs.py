"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers: it holds none of the method's
arithmetic (no gates, no normalisation, no recurrence). Raw draws are passed to
both sides; the gates (beta, g) and the L2 norm are applied by whichever side
consumes them (the CUDA path or the oracle).

Distributions (the workload descriptions of the pages' prefill and decode
steps): q, k, v, b, a ~ N(0, 1); A_log ~ U(0, ln 16); dt_bias ~ N(0, 0.5^2);
post-conv activations x ~ N(0, 1); decode state ~ N(0, 0.1^2); varlen request
lengths ~ U{64..2048}. Everything is drawn on the CPU from one
``torch.Generator`` per call, so the same seed gives the same bits everywhere.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def chunk_inputs(B: int, T: int, H: int, HV: int, K: int, V: int, M: int, seed: int = 0,
                 dtype: torch.dtype = torch.bfloat16):
    """Raw inputs of the chunked forward, drawn in the order q, k, v, b, a, A_log, dt_bias.

    q [B,T,H,K], k [B,T*M,H,K], v [B,T*M,HV,V] in ``dtype`` (not normalised);
    b [B,T*M,HV] and a [B,T,HV] fp32 gate inputs; A_log, dt_bias [HV] fp32.
    """
    g = _gen(seed)
    q = torch.randn(B, T, H, K, generator=g).to(dtype)
    k = torch.randn(B, T * M, H, K, generator=g).to(dtype)
    v = torch.randn(B, T * M, HV, V, generator=g).to(dtype)
    b = torch.randn(B, T * M, HV, generator=g)
    a = torch.randn(B, T, HV, generator=g)
    A_log = torch.rand(HV, generator=g) * math.log(16.0)
    dt_bias = torch.randn(HV, generator=g) * 0.5
    return {"q": q, "k": k, "v": v, "b": b, "a": a, "A_log": A_log, "dt_bias": dt_bias}


def varlen_lengths(n_seq: int, lo: int = 64, hi: int = 2048, seed: int = 0) -> torch.Tensor:
    """Request lengths ~ U{lo..hi} (int64)."""
    return torch.randint(lo, hi + 1, (n_seq,), generator=_gen(seed))


def cu_seqlens_of(lengths) -> torch.Tensor:
    """Offsets [N+1] (int32) of packed requests with the given lengths."""
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    return cu.to(torch.int32)


def prepare_inputs(n: int, T: int, M: int, H: int, G: int, P: int, N: int, seed: int = 0,
                   dtype: torch.dtype = torch.bfloat16):
    """Post-conv x [n,T,M*H*P+M*G*N+G*N], ba [n,T,M*H+H], A_log [H], dt_bias [H]."""
    g = _gen(seed)
    D = M * H * P + M * G * N + G * N
    x = torch.randn(n, T, D, generator=g).to(dtype)
    ba = torch.randn(n, T, M * H + H, generator=g).to(dtype)
    A_log = torch.rand(H, generator=g) * math.log(16.0)
    dt_bias = torch.randn(H, generator=g) * 0.5
    return {"x": x, "ba": ba, "A_log": A_log, "dt_bias": dt_bias}


def decode_state(n: int, H: int, K: int, V: int, seed: int = 1) -> torch.Tensor:
    """Per-request recurrent state [n,H,K,V] fp32 ~ N(0, 0.1^2)."""
    return torch.randn(n, H, K, V, generator=_gen(seed)) * 0.1


@dataclass(frozen=True)
class Workload:
    """One named workload of the pages' prefill/decode steps."""
    name: str
    kind: str  # "chunk" | "prefill" | "decode"
    dims: dict = field(default_factory=dict)


# The five workloads: a tiny fp32 case, a bf16 prefill, a packed varlen
# prefill that starts from prepare, a GVA prefill and a decode step.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32 B1 T128 H2 K32 V32 M2 BT64", "chunk",
                          dict(B=1, T=128, H=2, HV=2, K=32, V=32, M=2, BT=64,
                               dtype=torch.float32)),
    "prefill_bf16": Workload("prefill bf16 B2 T4096 H16 K128 V128 M2 BT64", "chunk",
                             dict(B=2, T=4096, H=16, HV=16, K=128, V=128, M=2, BT=64,
                                  dtype=torch.bfloat16)),
    "varlen_bf16": Workload("varlen bf16 16 requests U(64,2048) H32 G8 K128 V128 M3 BT64",
                            "prefill",
                            dict(n_seq=16, H=32, G=8, P=128, N=128, M=3, BT=64,
                                 dtype=torch.bfloat16)),
    "gva_bf16": Workload("GVA bf16 B4 T8192 H8 HV32 K128 V256 M2 BT64", "chunk",
                         dict(B=4, T=8192, H=8, HV=32, K=128, V=256, M=2, BT=64,
                              dtype=torch.bfloat16)),
    "decode": Workload("decode n256 S4 M2 H32 G8 P128 N128", "decode",
                       dict(n=256, S=4, M=2, H=32, G=8, P=128, N=128, dtype=torch.bfloat16)),
}
