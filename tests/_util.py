"""Shared helpers for the parity tests (no method arithmetic beyond error metrics)."""
from __future__ import annotations

import torch

import oracle
import synth_inputs as si

# Tolerances: max |x - x_ref| <= tol * RMS(x_ref), separately for o and the final
# state; tol = 2e-3 for bf16/fp16 inputs and 1e-5 for fp32 inputs.
TOL = {torch.bfloat16: 2e-3, torch.float16: 2e-3, torch.float32: 1e-5}

# Gates against the host-libm oracle, in ulp. The kernels' gates are bit-exact
# against the eager composition with CUDA's math library (asserted separately);
# the oracle calls the host's expf/log1pf. With CUDA's documented maximum errors
# (expf 2 ulp, log1pf 1 ulp) and the host's (expf 1 ulp, log1pf 2 ulp), the two
# sides' exp differ by at most 3 ulp and their log1p by at most 3 ulp more:
#   beta = 1/(1 + e^-b): 3 ulp passed through the sum (condition <= 1) plus the
#     add's and the division's rounding on each side: <= 5 ulp;
#   g = -e^A_log softplus(a + dt_bias) = -e^A_log log1p(e^x): 3 ulp (e^A_log) +
#     3 ulp (e^x, through log1p with condition <= 1) + 3 ulp (log1p) + the
#     product's rounding on each side: <= 10 ulp.
GATE_ULP = {"beta": 5, "g": 10}


def rel_err(got, want) -> float:
    want = want.detach().cpu().to(torch.float64)
    got = got.detach().cpu().to(torch.float64)
    rms = want.pow(2).mean().sqrt().item()
    if want.numel() == 0:
        return 0.0
    return (got - want).abs().max().item() / max(rms, 1e-300)


def chunk_case(B, T, H, HV, K, V, M, seed=0, dtype=torch.bfloat16, gated=True, shrink=False):
    """Seeded raw inputs plus oracle-computed gates (identical bits for both sides).

    shrink=True scales q and k by K**-0.5 (then re-rounds to ``dtype``) so that
    runs without the in-kernel L2 norm keep beta*|k|^2 near 1; with raw N(0,1)
    keys the delta rule's transition has eigenvalues far below -1 and the
    recurrence diverges, which no finite-precision path can follow."""
    d = si.chunk_inputs(B, T, H, HV, K, V, M, seed=seed, dtype=dtype)
    q, k = d["q"], d["k"]
    if shrink:
        q = (q.float() * K ** -0.5).to(dtype)
        k = (k.float() * K ** -0.5).to(dtype)
    beta, g = oracle.gate_map(d["b"], d["a"], d["A_log"], d["dt_bias"])
    return q, k, d["v"], beta, (g if gated else None)


def to(dev, *ts):
    return [None if t is None else t.to(dev) for t in ts]
