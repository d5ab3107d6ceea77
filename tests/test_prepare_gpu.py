"""Parity of the fused prepare kernel (prepare page: gdp_prefill_prepare,
gdp_decode_prepare) against the CPU oracle's fp32 map and the eager PyTorch
composition of the same fp32 operations.

q/k/v and the +0 placements are bit moves: bit-exact against the oracle.
beta and g are bit-exact against the eager GPU composition (the pages'
contract, asserted with torch.equal) and within the libm error bound of the
oracle, whose host expf/log1pf are not CUDA's (GATE_ULP: beta 5, g 10 ulp).
"""
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth_inputs as si
from _util import GATE_ULP

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ulp(a, b):
    ai = a.contiguous().view(torch.int32).to(torch.int64)
    bi = b.contiguous().view(torch.int32).to(torch.int64)
    ai = torch.where(ai < 0, -(ai & 0x7FFFFFFF), ai)
    bi = torch.where(bi < 0, -(bi & 0x7FFFFFFF), bi)
    return (ai - bi).abs()


def _eager_gates(ba, A_log, dt_bias, M, H, decode):
    n, T = ba.shape[:2]
    b = ba[..., :M * H].float().reshape(n, T * M, H)
    a = ba[..., M * H:].float()
    beta = torch.sigmoid(b)
    gt = -torch.exp(A_log.float()) * F.softplus(a + dt_bias.float())
    if decode:
        g = torch.zeros(n, T, M, H, dtype=torch.float32, device=ba.device)
        g[:, :, 0] = gt
        gt = g.reshape(n, T * M, H)
    return beta, gt


def _check(gdp, x, ba, A_log, dt_bias, M, H, G, P, N, decode):
    fn = gdp.gdp_decode_prepare if decode else gdp.gdp_prefill_prepare
    out = fn(x.to(DEV) if not x.is_cuda else x, ba.to(DEV) if not ba.is_cuda else ba,
             A_log.to(DEV), dt_bias.to(DEV), M, H, G, P, N)
    torch.cuda.synchronize()
    ref = oracle.prepare(x.cpu(), ba.cpu(), A_log, dt_bias, M, H, G, P, N, decode=decode)
    names = ("q", "k", "v", "beta", "g")
    for nm, a, b in zip(names[:3], out[:3], ref[:3]):
        assert a.dtype == b.dtype and tuple(a.shape) == tuple(b.shape), nm
        assert torch.equal(a.cpu(), b), f"{nm} differs from the oracle's bit copy"
    eb, eg = _eager_gates(ba.to(DEV), A_log.to(DEV), dt_bias.to(DEV), M, H, decode)
    assert torch.equal(out[3], eb), "beta differs from the eager composition"
    assert torch.equal(out[4], eg), "g differs from the eager composition"
    for nm, a, b in zip(names[3:], out[3:], ref[3:]):
        d = _ulp(a.cpu(), b)
        assert int(d.max()) <= GATE_ULP[nm], f"{nm}: {int(d.max())} ulp from the oracle"
    if decode:
        n, T = x.shape[:2]
        assert torch.count_nonzero(out[0].view(n, T, M, H, N)[:, :, :M - 1]) == 0
        assert torch.count_nonzero(out[4].view(n, T, M, H)[:, :, 1:]) == 0


def test_prefill_prepare_varlen_packed_workload(gdp):
    w = si.WORKLOADS["varlen_bf16"].dims
    T = int(si.varlen_lengths(w["n_seq"], seed=0).sum())
    d = si.prepare_inputs(1, T, w["M"], w["H"], w["G"], w["P"], w["N"], seed=0)
    _check(gdp, d["x"], d["ba"], d["A_log"], d["dt_bias"], w["M"], w["H"], w["G"], w["P"],
           w["N"], decode=False)


def test_decode_prepare_workload(gdp):
    w = si.WORKLOADS["decode"].dims
    d = si.prepare_inputs(w["n"], w["S"], w["M"], w["H"], w["G"], w["P"], w["N"], seed=1)
    _check(gdp, d["x"], d["ba"], d["A_log"], d["dt_bias"], w["M"], w["H"], w["G"], w["P"],
           w["N"], decode=True)


@pytest.mark.parametrize("decode", [False, True])
@pytest.mark.parametrize("M,H,G,P,N,dtype", [
    (3, 6, 3, 24, 16, torch.bfloat16),   # 16-byte vector path
    (2, 4, 2, 3, 5, torch.bfloat16),     # odd head sizes: element path
    (1, 2, 1, 8, 8, torch.float32),
    (2, 4, 4, 5, 4, torch.float32),
    (4, 8, 2, 16, 8, torch.float16),
])
def test_prepare_small_strided(gdp, decode, M, H, G, P, N, dtype):
    n, T = 3, 5
    d = si.prepare_inputs(n, T, M, H, G, P, N, seed=7, dtype=dtype)
    D = d["x"].shape[-1]
    # rows strided inside a wider buffer (a view of a conv output), ba non-contiguous
    big = torch.zeros(n, T + 1, D + 24, dtype=dtype)
    big[:, :T, 8:8 + D] = d["x"]
    x = big.to(DEV)[:, :T, 8:8 + D]
    bbig = torch.zeros(n, T, M * H + H + 5, dtype=dtype)
    bbig[..., 2:2 + M * H + H] = d["ba"]
    ba = bbig.to(DEV)[..., 2:2 + M * H + H]
    assert not x.is_contiguous() and not ba.is_contiguous()
    _check(gdp, x, ba, d["A_log"], d["dt_bias"], M, H, G, P, N, decode)


def test_gate_extremes(gdp):
    """Saturation of softplus above 20 and sigmoid tails, through the kernel."""
    M, H, G, P, N = 1, 8, 1, 8, 8
    vals = torch.tensor([-100., -30., -20., -1e-3, 0., 1e-3, 19.99, 20., 20.01, 25., 88., 1e4])
    T = vals.numel()
    d = si.prepare_inputs(1, T, M, H, G, P, N, seed=2, dtype=torch.float32)
    ba = d["ba"].clone()
    ba[0, :, :M * H] = vals.view(T, 1)
    ba[0, :, M * H:] = vals.view(T, 1)
    _check(gdp, d["x"], ba, d["A_log"], torch.zeros(H), M, H, G, P, N, decode=False)


def test_empty_prefill_is_a_no_op(gdp):
    M, H, G, P, N = 2, 4, 2, 8, 8
    x = torch.empty(1, 0, M * H * P + M * G * N + G * N, dtype=torch.bfloat16, device=DEV)
    ba = torch.empty(1, 0, M * H + H, dtype=torch.bfloat16, device=DEV)
    q, k, v, beta, g = gdp.gdp_prefill_prepare(x, ba, torch.zeros(H, device=DEV),
                                               torch.zeros(H, device=DEV), M, H, G, P, N)
    assert q.numel() == 0 and k.numel() == 0 and beta.numel() == 0


def test_deterministic(gdp):
    M, H, G, P, N = 2, 8, 4, 64, 64
    d = si.prepare_inputs(2, 33, M, H, G, P, N, seed=5)
    args = (d["x"].to(DEV), d["ba"].to(DEV), d["A_log"].to(DEV), d["dt_bias"].to(DEV), M, H, G,
            P, N)
    a = gdp.gdp_prefill_prepare(*args)
    b = gdp.gdp_prefill_prepare(*args)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("decode", [False, True])
@pytest.mark.parametrize("M,H,G,P,N,n,T", [
    (3, 16, 4, 128, 128, 2, 7), (2, 32, 8, 128, 128, 2, 7), (5, 8, 8, 64, 128, 2, 7),
    (2, 32, 8, 128, 128, 100, 16),  # several rows per resident CTA: the ring wraps
    (4, 64, 8, 128, 128, 2, 3),     # 76 KB rows: past the ring, one row at a time
])
def test_prepare_long_rows(gdp, decode, M, H, G, P, N, n, T):
    """Rows of 1.4-5k 16-byte vectors, beyond one pass of the row kernel: the
    shared-memory ring of raw rows (several rows per CTA when there are more
    rows than resident CTAs) and, for rows too long for the ring, the
    row-at-a-time kernel; over strided rows."""
    d = si.prepare_inputs(n, T, M, H, G, P, N, seed=M + H)
    D = d["x"].shape[-1]
    big = torch.zeros(n, T, D + 64, dtype=torch.bfloat16)
    big[:, :, 64:] = d["x"]
    x = big.to(DEV)[:, :, 64:]
    assert not x.is_contiguous()
    _check(gdp, x, d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N, decode)


@pytest.mark.parametrize("seed", list(range(500, 540)))
def test_prepare_shape_sweep(gdp, seed):
    """Seeded shapes: copies M, heads H over groups G, head sizes P and N (16-byte
    vector and element paths), all input dtypes, contiguous or strided rows,
    prefill or decode; row lengths from a few vectors to past the shared-memory
    ring, row counts below and above the resident CTAs."""
    import random
    r = random.Random(seed)
    decode = r.random() < 0.4
    dtype = r.choice([torch.bfloat16, torch.bfloat16, torch.float16, torch.float32])
    M = r.randint(1, 4)
    G = r.choice([1, 2, 4, 8])
    H = G * r.choice([1, 2, 4])
    P = r.choice([3, 5, 8, 16, 24, 64, 128])
    N = r.choice([4, 8, 16, 32, 64, 128])
    n = r.randint(1, 64)
    T = r.randint(1, 16) if decode else r.randint(1, 40)
    d = si.prepare_inputs(n, T, M, H, G, P, N, seed=seed, dtype=dtype)
    x, ba = d["x"], d["ba"]
    if r.random() < 0.5:  # rows inside a wider buffer (a view of a conv output)
        D = x.shape[-1]
        pad = r.choice([8, 16, 40])
        big = torch.zeros(n, T, D + pad, dtype=dtype)
        big[:, :, pad:] = x
        x = big.to(DEV)[:, :, pad:]
    _check(gdp, x, ba, d["A_log"], d["dt_bias"], M, H, G, P, N, decode)
