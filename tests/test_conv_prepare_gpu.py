"""Parity of the short causal conv fused into prepare (gdp_prefill_conv_prepare,
gdp_decode_conv_prepare; the prepare page's module overview places the conv
just before prepare and makes a -1 slot zero its output).

The conv outputs are computed values, so against the CPU oracle (host libm
expf) q/k/v agree to 1 unit in the last place of the activation dtype; against
the eager GPU composition of the same fp32 operations (torch elementwise ops,
CUDA's expf) they are bit-identical. The gates are prepare's and keep its bars
(bit-exact vs eager, within GATE_ULP of the oracle). Conv states are copies of inputs:
bit-exact.
"""
import pytest
import torch

import bench
import oracle
import synth_inputs as si
from _util import GATE_ULP, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ord(t):
    """Monotone integer image of a float tensor's bit patterns (bf16 or fp32)."""
    if t.dtype == torch.bfloat16:
        i = t.contiguous().view(torch.int16).to(torch.int64)
        return torch.where(i < 0, -(i & 0x7FFF), i)
    i = t.contiguous().view(torch.int32).to(torch.int64)
    return torch.where(i < 0, -(i & 0x7FFFFFFF), i)


def _ulps(a, b):
    return int((_ord(a.cpu()) - _ord(b.cpu())).abs().max()) if a.numel() else 0


def _eager_conv(xp, w, b, state=None):
    """The conv as torch elementwise ops on the GPU, in the kernel's operation order
    (z = b; z = z + w_i * x_i; y = z / (1 + exp(-z))), one sequence per batch row."""
    n, T, C = xp.shape
    W = w.shape[1]
    xf = xp.float()
    prev = (torch.zeros(n, W - 1, C, device=xp.device) if state is None
            else state.float().transpose(1, 2))
    full = torch.cat([prev, xf], 1)  # [n, W-1+T, C]
    z = b.float().view(1, 1, C).expand(n, T, C) if b is not None else torch.zeros(n, T, C, device=xp.device)
    for i in range(W):
        z = z + w[:, i].view(1, 1, C) * full[:, i:i + T]
    return (z / (1.0 + torch.exp(-z))).to(xp.dtype)


def _inputs(n, T, M, H, G, P, N, W, seed, dtype=torch.bfloat16):
    d = si.prepare_inputs(n, T, M, H, G, P, N, seed=seed, dtype=dtype)
    C = d["x"].shape[-1]
    gen = torch.Generator().manual_seed(seed + 1)
    w = torch.randn(C, W, generator=gen) * 0.5
    b = torch.randn(C, generator=gen) * 0.1
    return d, w, b


@pytest.mark.parametrize("W", [1, 2, 4])
@pytest.mark.parametrize("M,H,G,P,N", [(2, 4, 2, 64, 64), (3, 8, 2, 128, 128)])
def test_prefill_conv_prepare(gdp, W, M, H, G, P, N):
    n, T = 2, 45
    d, w, b = _inputs(n, T, M, H, G, P, N, W, seed=W + M)
    C = d["x"].shape[-1]
    h0 = torch.randn(n, C, W - 1, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    xp, ba = d["x"].to(DEV), d["ba"].to(DEV)
    args = (d["A_log"].to(DEV), d["dt_bias"].to(DEV), M, H, G, P, N)
    q, k, v, beta, g, st = gdp.gdp_prefill_conv_prepare(xp, w.to(DEV), b.to(DEV), ba, *args,
                                                       conv_state=h0.to(DEV))
    torch.cuda.synchronize()
    # the eager GPU composition, bit for bit
    xc = _eager_conv(xp, w.to(DEV), b.to(DEV), h0.to(DEV))
    ref = bench.eager_prepare(xc, ba, d["A_log"].to(DEV), d["dt_bias"].to(DEV), M, H, G, P, N,
                              False)
    for name, a_, b_ in zip("qkv", (q, k, v), ref[:3]):
        assert torch.equal(a_, b_.contiguous()), name
    assert torch.equal(beta, ref[3]) and torch.equal(g, ref[4])
    # the oracle: conv then prepare on the CPU
    oc, ost = oracle.conv(d["x"], w, b, state=h0)
    rq, rk, rv, rb, rg = oracle.prepare(oc, d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N,
                                        decode=False)
    for a_, b_ in ((q, rq), (k, rk), (v, rv)):
        assert _ulps(a_, b_) <= 1
    assert _ulps(beta, rb) <= GATE_ULP["beta"] and _ulps(g, rg) <= GATE_ULP["g"]
    assert torch.equal(st.cpu(), ost)


def test_prefill_conv_prepare_varlen_strided(gdp):
    M, H, G, P, N, W = 2, 4, 4, 64, 64, 4
    lens = [1, 2, 0, 40, 3, 70]
    cu = si.cu_seqlens_of(lens)
    T = int(cu[-1]) + 6  # rows past the last sequence are not outputs
    d, w, b = _inputs(1, T, M, H, G, P, N, W, seed=7)
    C = d["x"].shape[-1]
    h0 = torch.randn(len(lens), C, W - 1, generator=torch.Generator().manual_seed(8)).to(torch.bfloat16)
    big = torch.zeros(1, T, C + 64, dtype=torch.bfloat16)
    big[:, :, 32:32 + C] = d["x"]
    xp = big.to(DEV)[:, :, 32:32 + C]
    assert not xp.is_contiguous()
    q, k, v, beta, g, st = gdp.gdp_prefill_conv_prepare(
        xp, w.to(DEV), b.to(DEV), d["ba"].to(DEV), d["A_log"].to(DEV), d["dt_bias"].to(DEV), M,
        H, G, P, N, conv_state=h0.to(DEV), cu_seqlens=cu.to(DEV))
    torch.cuda.synchronize()
    oc, ost = oracle.conv(d["x"], w, b, state=h0, cu_seqlens=cu)
    rq, rk, rv, rb, rg = oracle.prepare(oc, d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N,
                                        decode=False)
    n_tok = int(cu[-1])
    assert _ulps(q[:, :n_tok], rq[:, :n_tok]) <= 1
    assert _ulps(k[:, :M * n_tok], rk[:, :M * n_tok]) <= 1
    assert _ulps(v[:, :M * n_tok], rv[:, :M * n_tok]) <= 1
    assert torch.equal(st.cpu(), ost)
    assert torch.equal(st.cpu()[2], h0[2])  # the empty sequence keeps its state


def test_decode_conv_prepare_with_pool_and_padding(gdp):
    w_ = si.WORKLOADS["decode"].dims
    n, S, M, H, G, P, N = 64, w_["S"], w_["M"], w_["H"], w_["G"], w_["P"], w_["N"]
    W, n_slots = 4, 100
    d, w, b = _inputs(n, S, M, H, G, P, N, W, seed=11)
    C = d["x"].shape[-1]
    gen = torch.Generator().manual_seed(12)
    pool = torch.randn(n_slots, C, W - 1, generator=gen).to(torch.bfloat16)
    slots = torch.randperm(n_slots, generator=gen)[:n].to(torch.int32)
    slots[[3, 17, 40]] = -1
    pd = pool.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, k, v, beta, g = gdp.gdp_decode_conv_prepare(
        d["x"].to(DEV), w.to(DEV), b.to(DEV), d["ba"].to(DEV), d["A_log"].to(DEV),
        d["dt_bias"].to(DEV), M, H, G, P, N, pd, slots.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    oc, opool = oracle.conv(d["x"], w, b, state=pool, slot=slots)
    rq, rk, rv, rb, rg = oracle.prepare(oc, d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N,
                                        decode=True)
    for a_, b_ in ((q, rq), (k, rk), (v, rv)):
        assert _ulps(a_, b_) <= 1
    assert _ulps(beta, rb) <= GATE_ULP["beta"] and _ulps(g, rg) <= GATE_ULP["g"]
    assert torch.equal(pd.cpu(), opool)
    for r in (3, 17, 40):  # padding: zero q, k, v
        assert torch.count_nonzero(q[r]) + torch.count_nonzero(k[r]) + torch.count_nonzero(v[r]) == 0
    # a repeated slot is rejected and both requests become padding
    bad = slots.clone()
    bad[5] = bad[6]
    status.zero_()
    q2, k2, v2, _, _ = gdp.gdp_decode_conv_prepare(
        d["x"].to(DEV), w.to(DEV), b.to(DEV), d["ba"].to(DEV), d["A_log"].to(DEV),
        d["dt_bias"].to(DEV), M, H, G, P, N, pool.to(DEV), bad.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert torch.count_nonzero(v2[5]) + torch.count_nonzero(v2[6]) == 0


def test_conv_prepare_then_chunk_fwd_matches_the_oracle(gdp):
    """From pre-conv activations to o: fused conv + prepare, then the chunked forward,
    against the oracle's conv, prepare and fp64 walk."""
    M, H, G, P, N, W, T = 2, 4, 2, 128, 128, 4, 300
    d, w, b = _inputs(1, T, M, H, G, P, N, W, seed=13)
    q, k, v, beta, g, _ = gdp.gdp_prefill_conv_prepare(
        d["x"].to(DEV), w.to(DEV), b.to(DEV), d["ba"].to(DEV), d["A_log"].to(DEV),
        d["dt_bias"].to(DEV), M, H, G, P, N)
    o, fs = gdp.gdp_chunk_fwd(q, k, v, beta, g, chunk_size=64, num_householder=M,
                              use_qk_l2norm=True)
    torch.cuda.synchronize()
    oc, _ = oracle.conv(d["x"], w, b)
    rq, rk, rv, rb, rg = oracle.prepare(oc, d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N,
                                        decode=False)
    ro, rfs = oracle.walk(rq, rk, rv, rb, rg, M, N ** -0.5, l2norm=True)
    assert rel_err(o, ro) <= 2e-3 and rel_err(fs, rfs) <= 2e-3


def test_conv_prepare_fp32(gdp):
    M, H, G, P, N, W = 2, 2, 1, 8, 8, 3
    d, w, b = _inputs(2, 9, M, H, G, P, N, W, seed=14, dtype=torch.float32)
    q, k, v, beta, g, st = gdp.gdp_prefill_conv_prepare(
        d["x"].to(DEV), w.to(DEV), b.to(DEV), d["ba"].to(DEV), d["A_log"].to(DEV),
        d["dt_bias"].to(DEV), M, H, G, P, N)
    torch.cuda.synchronize()
    oc, ost = oracle.conv(d["x"], w, b)
    rq, rk, rv, _, _ = oracle.prepare(oc, d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N,
                                      decode=False)
    for a_, b_ in ((q, rq), (k, rk), (v, rv)):
        assert _ulps(a_, b_) <= 4
    assert torch.equal(st.cpu(), ost)
