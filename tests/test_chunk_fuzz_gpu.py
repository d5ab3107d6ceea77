"""Seeded shape sweep of gdp_chunk_fwd (wy_fast page: recompute_w_u_fwd; chunk_o
page: chunk_gated_delta_product_fwd_o, parameters cu_seqlens, num_householder,
GVA with H < HV) against the CPU oracle's fp64 token walk, element by element.

Each case draws its shape from a fixed seed: the tensor-core path (bf16, K = 128,
chunk 64, V in {64, 128, 256}, M in 1..3) or the CUDA-core path (fp32 / fp16 /
bf16 with other K, chunk sizes or M), dense batches or ragged packed sequences
(empty and one-token sequences among them), GVA head ratios, gates on or off,
the in-kernel L2 norm on or off, with or without an initial state. Tolerance as
in the other chunk tests: max |x - x_ref| <= tol * RMS(x_ref), tol 2e-3 for
16-bit inputs and 1e-5 for fp32, for o and for every sequence's final state.
"""
import random

import pytest
import torch

import oracle
import synth_inputs as si
from _util import TOL, chunk_case, rel_err, to

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _draw(seed):
    r = random.Random(seed)
    tc = r.random() < 0.6
    if tc:
        dtype, K, BT = torch.bfloat16, 128, 64
        V = r.choice([64, 128, 256])
        M = r.choice([1, 2, 3])
    else:
        dtype = r.choice([torch.float32, torch.float16, torch.bfloat16])
        K = r.choice([32, 64, 256])
        V = r.choice([16, 32, 48, 64])
        BT = r.choice([16, 32, 64])
        M = r.choice([1, 2, 3, 4])
    H = r.choice([1, 2])
    HV = H * r.choice([1, 2, 4])
    varlen = r.random() < 0.5
    if varlen:
        n = r.randint(1, 6)
        lens = [r.choice([0, 1, r.randint(2, 64), r.randint(65, 400)]) for _ in range(n)]
        if sum(lens) == 0:
            lens[-1] = r.randint(1, 200)
        B, T = 1, sum(lens)
    else:
        lens = None
        B, T = r.randint(1, 3), r.randint(1, 400)
    gated = r.random() < 0.8
    l2 = r.random() < 0.7
    h0 = r.random() < 0.4
    return dict(tc=tc, dtype=dtype, K=K, V=V, BT=BT, M=M, H=H, HV=HV, lens=lens, B=B, T=T,
                gated=gated, l2=l2, h0=h0)


SEEDS = list(range(100, 220))


@pytest.mark.parametrize("seed", SEEDS)
def test_chunk_fwd_shape_sweep(gdp, seed):
    c = _draw(seed)
    B, T, H, HV, K, V, M = c["B"], c["T"], c["H"], c["HV"], c["K"], c["V"], c["M"]
    q, k, v, beta, g = chunk_case(B, T, H, HV, K, V, M, seed=seed, dtype=c["dtype"],
                                  gated=c["gated"], shrink=not c["l2"])
    cu = si.cu_seqlens_of(c["lens"]) if c["lens"] is not None else None
    N = len(c["lens"]) if cu is not None else B
    h0 = (torch.randn(N, HV, K, V, generator=torch.Generator().manual_seed(seed))
          if c["h0"] else None)
    qd, kd, vd, bd, gd, hd, cd = to(DEV, q, k, v, beta, g, h0, cu)
    o, fs = gdp.gdp_chunk_fwd(qd, kd, vd, bd, gd, cu_seqlens=cd, chunk_size=c["BT"],
                              num_householder=M, initial_state=hd, use_qk_l2norm=c["l2"])
    torch.cuda.synchronize()
    path = gdp.gdp_chunk_fwd_stage_offsets(B, T, N, H, HV, K, V, M, c["BT"], c["dtype"])[5]
    assert path == (1 if c["tc"] else 0), (c, path)
    ro, rfs = oracle.walk(q, k, v, beta, g, M, K ** -0.5, h0=h0, cu_seqlens=cu, l2norm=c["l2"])
    tol = TOL[c["dtype"]]
    o = o.cpu()
    assert rel_err(o, ro) <= tol, (c, rel_err(o, ro))
    fs = fs.cpu()
    for s_ in range(N):
        assert rel_err(fs[s_], rfs[s_]) <= tol, (c, s_, rel_err(fs[s_], rfs[s_]))
