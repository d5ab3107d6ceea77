"""Parity of gdp_recurrent_update (decode: the copies walked as a sequence,
prepare page decode bullet) against the oracle's fp64 per-step walk."""
import pytest
import torch

import oracle
import synth_inputs as si
from _util import TOL, chunk_case, rel_err, to

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_decode_workload_prepare_then_update(gdp):
    w = si.WORKLOADS["decode"].dims
    n, S, M, H, G, P, N = w["n"], w["S"], w["M"], w["H"], w["G"], w["P"], w["N"]
    d = si.prepare_inputs(n, S, M, H, G, P, N, seed=1)
    q, k, v, beta, g = gdp.gdp_decode_prepare(d["x"].to(DEV), d["ba"].to(DEV),
                                              d["A_log"].to(DEV), d["dt_bias"].to(DEV), M, H, G,
                                              P, N)
    state = si.decode_state(n, H, N, P).to(DEV)
    s0 = state.cpu()
    o = gdp.gdp_recurrent_update(q, k, v, beta, g, state, use_qk_l2norm=True)
    torch.cuda.synchronize()
    rq, rk, rv, rb, rg = oracle.prepare(d["x"], d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N,
                                        decode=True)
    ro, rs = oracle.recurrent(rq, rk, rv, rb, rg, s0, N ** -0.5, l2norm=True)
    assert rel_err(o, ro) <= 2e-3
    assert rel_err(state, rs) <= 2e-3


@pytest.mark.parametrize("n,L,H,HV,K,V,dtype,l2", [
    (3, 5, 2, 2, 32, 16, torch.float32, True),
    (2, 8, 1, 4, 64, 128, torch.float32, False),     # GVA
    (4, 3, 2, 2, 256, 136, torch.bfloat16, True),    # several CTAs along V, ragged slice
    (2, 4, 2, 2, 128, 128, torch.float16, True),
    (3, 11, 2, 4, 128, 72, torch.bfloat16, True),    # K = 128 kernel: ragged slice, two batches
    (40, 4, 4, 8, 128, 128, torch.bfloat16, True),   # more items than resident CTAs
    (2, 3, 1, 2, 128, 136, torch.float32, False),    # K = 128 kernel: three slices, fp32
])
def test_recurrent_small(gdp, n, L, H, HV, K, V, dtype, l2):
    gen = torch.Generator().manual_seed(n * L + K)
    # without the L2 norm, raw N(0,1) keys make the delta rule diverge; scale them
    sc = 1.0 if l2 else K ** -0.5
    q = (torch.randn(n, L, H, K, generator=gen) * sc).to(dtype)
    k = (torch.randn(n, L, H, K, generator=gen) * sc).to(dtype)
    v = torch.randn(n, L, HV, V, generator=gen).to(dtype)
    beta = torch.rand(n, L, HV, generator=gen)
    g = -torch.rand(n, L, HV, generator=gen)
    state = torch.randn(n, HV, K, V, generator=gen) * 0.1
    ro, rs = oracle.recurrent(q, k, v, beta, g, state, K ** -0.5, l2norm=l2)
    sd = state.to(DEV)
    o = gdp.gdp_recurrent_update(*to(DEV, q, k, v, beta, g), sd, use_qk_l2norm=l2)
    torch.cuda.synchronize()
    assert rel_err(o, ro) <= TOL[dtype]
    assert rel_err(sd, rs) <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_recurrent_extreme_decays_and_zero_queries(gdp, dtype):
    """K = 128 kernel: decays strong enough that the running product of a call's
    decays leaves the fp32 range (g = -200 underflows e^g to 0; runs of -30 cross
    2^-40 several times), g = 0 steps, and all-zero query rows (their o rows are
    exact zeros), over two staged batches of steps."""
    n, L, H, HV, K, V = 3, 13, 2, 4, 128, 72
    gen = torch.Generator().manual_seed(11)
    q = torch.randn(n, L, H, K, generator=gen).to(dtype)
    q[:, 0::2] = 0          # every other step has no query (the decode copy layout)
    q[1, 5] = 0
    k = torch.randn(n, L, H, K, generator=gen).to(dtype)
    v = torch.randn(n, L, HV, V, generator=gen).to(dtype)
    beta = torch.rand(n, L, HV, generator=gen)
    g = -torch.rand(n, L, HV, generator=gen)
    g[0, :, :] = -30.0
    g[1, 3, :] = -200.0
    g[1, 7:, 1] = -45.0
    g[2, :, 2] = 0.0
    state = torch.randn(n, HV, K, V, generator=gen) * 0.1
    ro, rs = oracle.recurrent(q, k, v, beta, g, state, K ** -0.5, l2norm=True)
    sd = state.to(DEV)
    o = gdp.gdp_recurrent_update(*to(DEV, q, k, v, beta, g), sd, use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert rel_err(o, ro) <= TOL[dtype]
    assert rel_err(sd, rs) <= TOL[dtype]
    zero_rows = (q.float().abs().sum(-1) == 0)            # [n, L, H]
    hv_to_h = torch.arange(HV) // (HV // H)
    oz = o.cpu()[zero_rows[:, :, hv_to_h]]
    assert torch.count_nonzero(oz) == 0


@pytest.mark.parametrize("K", [64, 128])
def test_recurrent_matches_chunked_prefill(gdp, K):
    """Walking a prefill's copies one step at a time (q on the last copy, g on the
    first) gives the chunked forward's outputs and final state."""
    B, T, H, HV, V, M = 2, 40, 2, 2, 64, 3
    q, k, v, beta, g = chunk_case(B, T, H, HV, K, V, M, seed=2)
    qd, kd, vd, bd, gd = to(DEV, q, k, v, beta, g)
    o, fs = gdp.gdp_chunk_fwd(qd, kd, vd, bd, gd, chunk_size=64, num_householder=M,
                              use_qk_l2norm=True)
    qp = torch.zeros(B, T * M, H, K, dtype=q.dtype, device=DEV)
    qp.view(B, T, M, H, K)[:, :, M - 1] = qd
    gp = torch.zeros(B, T * M, HV, device=DEV)
    gp.view(B, T, M, HV)[:, :, 0] = gd
    state = torch.zeros(B, HV, K, V, device=DEV)
    od = gdp.gdp_recurrent_update(qp, kd, vd, bd, gp, state, use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert rel_err(od.view(B, T, M, HV, V)[:, :, M - 1], o) <= 1e-4
    assert rel_err(state, fs) <= 1e-4


def test_graph_capture_replay(gdp):
    """Static shapes, no host sync: the decode step captures into a CUDA graph."""
    w = si.WORKLOADS["decode"].dims
    n, S, M, H, G, P, N = 16, w["S"], w["M"], w["H"], w["G"], w["P"], w["N"]
    d = si.prepare_inputs(n, S, M, H, G, P, N, seed=3)
    x, ba = d["x"].to(DEV), d["ba"].to(DEV)
    A_log, dt_bias = d["A_log"].to(DEV), d["dt_bias"].to(DEV)
    s_init = si.decode_state(n, H, N, P).to(DEV)
    outs = gdp.gdp_decode_prepare(x, ba, A_log, dt_bias, M, H, G, P, N)
    state = s_init.clone()
    o = torch.empty(n, S * M, H, P, device=DEV)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # warm up
        gdp.gdp_decode_prepare(x, ba, A_log, dt_bias, M, H, G, P, N, out=outs)
        gdp.gdp_recurrent_update(*outs, state, use_qk_l2norm=True, out=o)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdp.gdp_decode_prepare(x, ba, A_log, dt_bias, M, H, G, P, N, out=outs)
        gdp.gdp_recurrent_update(*outs, state, use_qk_l2norm=True, out=o)
    state.copy_(s_init)
    graph.replay()
    torch.cuda.synchronize()
    o_graph, s_graph = o.clone(), state.clone()
    state.copy_(s_init)
    gdp.gdp_decode_prepare(x, ba, A_log, dt_bias, M, H, G, P, N, out=outs)
    o2 = gdp.gdp_recurrent_update(*outs, state, use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert torch.equal(o_graph, o2) and torch.equal(s_graph, state)


def _slot_reference(q, k, v, beta, g, pool, slots, scale, l2):
    """The oracle's per-step walk applied to the pool entries the slots name; padding
    requests (slot -1) produce zero rows and leave the pool alone."""
    new_pool = pool.clone().double()
    o = torch.zeros(q.shape[0], q.shape[1], v.shape[2], v.shape[3], dtype=torch.float64)
    live = [r for r in range(q.shape[0]) if int(slots[r]) >= 0]
    if live:
        idx = torch.tensor([int(slots[r]) for r in live])
        lr = torch.tensor(live)
        ro, rs = oracle.recurrent(q[lr], k[lr], v[lr], beta[lr], g[lr], pool[idx], scale,
                                  l2norm=l2)
        o[lr] = ro
        new_pool[idx] = rs
    return o, new_pool


@pytest.mark.parametrize("K,V,dtype", [(128, 128, torch.bfloat16), (64, 48, torch.float32)])
def test_recurrent_slots_with_padding(gdp, K, V, dtype):
    n, L, H, HV, n_slots = 24, 4, 2, 4, 40
    gen = torch.Generator().manual_seed(K + V)
    q = torch.randn(n, L, H, K, generator=gen).to(dtype)
    k = torch.randn(n, L, H, K, generator=gen).to(dtype)
    v = torch.randn(n, L, HV, V, generator=gen).to(dtype)
    beta = torch.rand(n, L, HV, generator=gen)
    g = -torch.rand(n, L, HV, generator=gen)
    pool = torch.randn(n_slots, HV, K, V, generator=gen) * 0.1
    perm = torch.randperm(n_slots, generator=gen)[:n].to(torch.int32)
    perm[[2, 7, 8, 20]] = -1  # padding requests
    ro, rpool = _slot_reference(q, k, v, beta, g, pool, perm, K ** -0.5, True)
    pd = pool.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gdp.gdp_recurrent_update_slots(*to(DEV, q, k, v, beta, g), pd, perm.to(DEV),
                                       use_qk_l2norm=True, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rel_err(o, ro) <= TOL[dtype]
    assert rel_err(pd, rpool) <= TOL[dtype]
    untouched = sorted(set(range(n_slots)) - {int(s) for s in perm if int(s) >= 0})
    assert torch.equal(pd.cpu()[untouched], pool[untouched])  # bitwise: never written
    pad = perm < 0
    assert torch.count_nonzero(o.cpu()[pad]) == 0


def test_recurrent_slots_identity_equals_dense_call(gdp):
    """slot[r] = r over a pool of n entries is the dense call, bit for bit."""
    n, L, H, HV, K, V = 8, 4, 2, 2, 128, 128
    gen = torch.Generator().manual_seed(7)
    q, k = (torch.randn(n, L, H, K, generator=gen).to(torch.bfloat16) for _ in range(2))
    v = torch.randn(n, L, HV, V, generator=gen).to(torch.bfloat16)
    beta, g = torch.rand(n, L, HV, generator=gen), -torch.rand(n, L, HV, generator=gen)
    s0 = torch.randn(n, HV, K, V, generator=gen) * 0.1
    a, b = s0.to(DEV), s0.to(DEV)
    ins = to(DEV, q, k, v, beta, g)
    o1 = gdp.gdp_recurrent_update(*ins, a, use_qk_l2norm=True)
    o2 = gdp.gdp_recurrent_update_slots(*ins, b, torch.arange(n, dtype=torch.int32, device=DEV),
                                        use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(a, b)


def test_recurrent_slots_request_order_does_not_matter(gdp):
    """The same requests in a permuted order, each keeping its pool entry, give
    every request's o rows and pool entry bit for bit."""
    n, L, H, HV, K, V, n_slots = 12, 4, 2, 4, 128, 128, 20
    gen = torch.Generator().manual_seed(17)
    q, k = (torch.randn(n, L, H, K, generator=gen).to(torch.bfloat16) for _ in range(2))
    v = torch.randn(n, L, HV, V, generator=gen).to(torch.bfloat16)
    beta, g = torch.rand(n, L, HV, generator=gen), -torch.rand(n, L, HV, generator=gen)
    pool = torch.randn(n_slots, HV, K, V, generator=gen) * 0.1
    slots = torch.randperm(n_slots, generator=gen)[:n].to(torch.int32)
    slots[3] = -1
    perm = torch.randperm(n, generator=gen)
    a, b = pool.to(DEV), pool.to(DEV)
    o1 = gdp.gdp_recurrent_update_slots(*to(DEV, q, k, v, beta, g), a, slots.to(DEV),
                                        use_qk_l2norm=True)
    o2 = gdp.gdp_recurrent_update_slots(*to(DEV, q[perm], k[perm], v[perm], beta[perm], g[perm]), b,
                                        slots[perm].to(DEV), use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert torch.equal(o2.cpu(), o1.cpu()[perm])
    assert torch.equal(a, b)


@pytest.mark.parametrize("bad", ["repeated", "out_of_range"])
def test_recurrent_slots_rejects_bad_slots_on_device(gdp, bad):
    n, L, H, HV, K, V, n_slots = 6, 2, 2, 2, 128, 64, 8
    gen = torch.Generator().manual_seed(9)
    q, k = (torch.randn(n, L, H, K, generator=gen).to(torch.bfloat16) for _ in range(2))
    v = torch.randn(n, L, HV, V, generator=gen).to(torch.bfloat16)
    beta, g = torch.rand(n, L, HV, generator=gen), -torch.rand(n, L, HV, generator=gen)
    pool = torch.randn(n_slots, HV, K, V, generator=gen) * 0.1
    slots = torch.tensor([0, 3, 5, 1, 6, 2], dtype=torch.int32)
    if bad == "repeated":
        slots[4] = 3  # requests 1 and 4 both name entry 3
        rejected = [1, 4]
    else:
        slots[2] = n_slots  # past the pool
        rejected = [2]
    ref_slots = slots.clone()
    ref_slots[rejected] = -1
    ro, rpool = _slot_reference(q, k, v, beta, g, pool, ref_slots, K ** -0.5, True)
    pd = pool.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gdp.gdp_recurrent_update_slots(*to(DEV, q, k, v, beta, g), pd, slots.to(DEV),
                                       use_qk_l2norm=True, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert torch.count_nonzero(o.cpu()[rejected]) == 0
    assert rel_err(o, ro) <= 2e-3 and rel_err(pd, rpool) <= 2e-3


def test_recurrent_slots_graph_replay_with_new_slots(gdp):
    """Captured once, replayed after the slot table changes in place."""
    n, L, H, HV, K, V, n_slots = 8, 4, 2, 4, 128, 128, 16
    gen = torch.Generator().manual_seed(10)
    q, k = (torch.randn(n, L, H, K, generator=gen).to(torch.bfloat16) for _ in range(2))
    v = torch.randn(n, L, HV, V, generator=gen).to(torch.bfloat16)
    beta, g = torch.rand(n, L, HV, generator=gen), -torch.rand(n, L, HV, generator=gen)
    pool0 = torch.randn(n_slots, HV, K, V, generator=gen) * 0.1
    ins = to(DEV, q, k, v, beta, g)
    pd = pool0.to(DEV)
    slots = torch.arange(n, dtype=torch.int32, device=DEV)
    o = torch.empty(n, L, HV, V, device=DEV)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        gdp.gdp_recurrent_update_slots(*ins, pd, slots, use_qk_l2norm=True, out=o)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdp.gdp_recurrent_update_slots(*ins, pd, slots, use_qk_l2norm=True, out=o)
    new = torch.tensor([9, -1, 3, 15, 0, -1, 12, 4], dtype=torch.int32)
    slots.copy_(new.to(DEV))
    pd.copy_(pool0.to(DEV))
    graph.replay()
    torch.cuda.synchronize()
    ro, rpool = _slot_reference(q, k, v, beta, g, pool0, new, K ** -0.5, True)
    assert rel_err(o, ro) <= 2e-3 and rel_err(pd, rpool) <= 2e-3


def _draw_decode(seed):
    import random
    r = random.Random(seed)
    H = r.choice([1, 2])
    return dict(n=r.randint(1, 40), L=r.randint(1, 20), H=H, HV=H * r.choice([1, 2, 4]),
                K=r.choice([32, 64, 128, 128, 256]),
                V=r.choice([8, 16, 40, 64, 72, 128, 136, 200, 256]),
                dtype=r.choice([torch.float32, torch.float16, torch.bfloat16]),
                l2=r.random() < 0.7, slots=r.random() < 0.4, strong=r.random() < 0.3)


@pytest.mark.parametrize("seed", list(range(300, 360)))
def test_recurrent_shape_sweep(gdp, seed):
    """Seeded shapes for the decode update, dense or through a slot pool with
    padding requests: both kernels (K = 128 and the others), ragged value
    slices, one or two staged step batches, GVA ratios, all input dtypes, the
    L2 norm on or off, and some calls with decays far below the fp32 range."""
    c = _draw_decode(seed)
    n, L, H, HV, K, V, dtype, l2 = (c[x] for x in ("n", "L", "H", "HV", "K", "V", "dtype", "l2"))
    gen = torch.Generator().manual_seed(seed)
    sc = 1.0 if l2 else K ** -0.5
    q = (torch.randn(n, L, H, K, generator=gen) * sc).to(dtype)
    k = (torch.randn(n, L, H, K, generator=gen) * sc).to(dtype)
    v = torch.randn(n, L, HV, V, generator=gen).to(dtype)
    beta = torch.rand(n, L, HV, generator=gen)
    g = -torch.rand(n, L, HV, generator=gen) * (40.0 if c["strong"] else 1.0)
    if c["slots"]:
        n_slots = n + 5
        pool = torch.randn(n_slots, HV, K, V, generator=gen) * 0.1
        slots = torch.randperm(n_slots, generator=gen)[:n].to(torch.int32)
        slots[torch.rand(n, generator=gen) < 0.15] = -1
        ro, rpool = _slot_reference(q, k, v, beta, g, pool, slots, K ** -0.5, l2)
        pd = pool.to(DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        o = gdp.gdp_recurrent_update_slots(*to(DEV, q, k, v, beta, g), pd, slots.to(DEV),
                                           use_qk_l2norm=l2, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert rel_err(o, ro) <= TOL[dtype], (c, rel_err(o, ro))
        assert rel_err(pd, rpool) <= TOL[dtype], (c, rel_err(pd, rpool))
        untouched = sorted(set(range(n_slots)) - {int(s) for s in slots if int(s) >= 0})
        assert torch.equal(pd.cpu()[untouched], pool[untouched])
    else:
        state = torch.randn(n, HV, K, V, generator=gen) * 0.1
        ro, rs = oracle.recurrent(q, k, v, beta, g, state, K ** -0.5, l2norm=l2)
        sd = state.to(DEV)
        o = gdp.gdp_recurrent_update(*to(DEV, q, k, v, beta, g), sd, use_qk_l2norm=l2)
        torch.cuda.synchronize()
        assert rel_err(o, ro) <= TOL[dtype], (c, rel_err(o, ro))
        assert rel_err(sd, rs) <= TOL[dtype], (c, rel_err(sd, rs))
