"""Parity of gdp_chunk_fwd (wy_fast page: recompute_w_u_fwd; chunk_o page:
chunk_gated_delta_product_fwd_o) against the CPU oracle's fp64 token walk,
element by element, plus stage-by-stage checks against the oracle's chunked
WY restatement.

Tolerance: max |x - x_ref| <= tol * RMS(x_ref) for o and for the final state,
tol = 2e-3 for bf16/fp16 inputs and 1e-5 for fp32 inputs. The oracle reads
the same quantised inputs (and the same fp32 gates) as the GPU.
"""
import pytest
import torch

import oracle
import synth_inputs as si
from _util import TOL, chunk_case, rel_err, to

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(gdp, q, k, v, beta, g, M, BT, l2, h0=None, cu=None):
    qd, kd, vd, bd, gd, hd, cd = to(DEV, q, k, v, beta, g, h0, cu)
    o, fs = gdp.gdp_chunk_fwd(qd, kd, vd, bd, gd, cu_seqlens=cd, chunk_size=BT,
                              num_householder=M, initial_state=hd, use_qk_l2norm=l2)
    torch.cuda.synchronize()
    return o.cpu(), fs.cpu()


CASES = [
    # B, T, H, HV, K, V, M, BT, dtype, l2norm, gated, h0
    (1, 128, 2, 2, 32, 32, 2, 64, torch.float32, True, True, False),   # tiny fp32 workload
    (2, 200, 2, 2, 64, 64, 2, 64, torch.bfloat16, True, True, False),
    (1, 150, 2, 2, 32, 48, 3, 64, torch.bfloat16, True, True, True),   # chunks split tokens
    (1, 77, 1, 1, 64, 32, 1, 32, torch.float32, False, True, True),
    (2, 90, 2, 6, 32, 48, 2, 64, torch.bfloat16, True, True, False),   # GVA
    (1, 70, 2, 2, 32, 32, 2, 16, torch.float32, True, False, True),    # ungated
    (1, 100, 2, 2, 64, 64, 4, 64, torch.float16, True, True, False),
    (1, 300, 2, 2, 128, 128, 2, 64, torch.bfloat16, True, True, True),
    (1, 260, 2, 4, 128, 256, 2, 64, torch.bfloat16, True, True, False),
    (2, 330, 2, 2, 128, 64, 2, 64, torch.bfloat16, True, True, True),  # tensor-core path, V = 64
    (1, 131, 2, 2, 128, 128, 3, 64, torch.bfloat16, False, True, False),
    (1, 65, 1, 1, 256, 64, 1, 64, torch.float32, True, True, False),
    (1, 200, 2, 2, 128, 128, 2, 64, torch.bfloat16, True, False, True),  # tensor-core, ungated
    (1, 150, 2, 2, 128, 64, 3, 64, torch.bfloat16, True, False, False),  # tensor-core, ungated
    (1, 600, 2, 2, 128, 128, 1, 64, torch.bfloat16, True, True, True),   # tensor-core, M = 1
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_chunk_fwd_matches_walk(gdp, case):
    B, T, H, HV, K, V, M, BT, dtype, l2, gated, with_h0 = case
    q, k, v, beta, g = chunk_case(B, T, H, HV, K, V, M, seed=T + K, dtype=dtype, gated=gated,
                                  shrink=not l2)
    h0 = torch.randn(B, HV, K, V, generator=torch.Generator().manual_seed(3)) if with_h0 else None
    o, fs = _run(gdp, q, k, v, beta, g, M, BT, l2, h0=h0)
    ro, rfs = oracle.walk(q, k, v, beta, g, M, K ** -0.5, h0=h0, l2norm=l2)
    tol = TOL[dtype]
    assert rel_err(o, ro) <= tol, rel_err(o, ro)
    assert rel_err(fs, rfs) <= tol, rel_err(fs, rfs)


@pytest.mark.parametrize("K,V,M", [(32, 32, 2), (128, 128, 2), (128, 128, 3), (128, 64, 2)])
def test_varlen_with_ragged_and_empty_sequences(gdp, K, V, M):
    lens = [1, 63, 64, 65, 130, 0, 7, 200]
    cu = si.cu_seqlens_of(lens)
    T = int(cu[-1]) + 5  # padding tokens after the last sequence are untouched
    q, k, v, beta, g = chunk_case(1, T, 2, 2, K, V, M, seed=11)
    h0 = torch.randn(len(lens), 2, K, V, generator=torch.Generator().manual_seed(4))
    o, fs = _run(gdp, q, k, v, beta, g, M, 64, True, h0=h0, cu=cu)
    ro, rfs = oracle.walk(q, k, v, beta, g, M, K ** -0.5, cu_seqlens=cu, h0=h0, l2norm=True)
    n = int(cu[-1])
    assert rel_err(o[:, :n], ro[:, :n]) <= 2e-3
    assert rel_err(fs, rfs) <= 2e-3
    # empty sequence: final state is its initial state
    assert torch.equal(fs[5], h0[5])


@pytest.mark.parametrize("M", [2, 3])
def test_varlen_many_sequences(gdp, M):
    """More sequences than the chunk-table kernel keeps in shared memory (1024):
    the table fill for the ones past it takes its other branch. Short ragged
    lengths, empty ones among them, on the tensor-core path."""
    gen = torch.Generator().manual_seed(21)
    lens = torch.randint(0, 5, (1100,), generator=gen).tolist()
    lens[1050] = 70  # one sequence past the shared records spans two 64-token chunks
    cu = si.cu_seqlens_of(lens)
    T = int(cu[-1])
    q, k, v, beta, g = chunk_case(1, T, 1, 1, 128, 128, M, seed=22)
    o, fs = _run(gdp, q, k, v, beta, g, M, 64, True, cu=cu)
    ro, rfs = oracle.walk(q, k, v, beta, g, M, 128 ** -0.5, cu_seqlens=cu, l2norm=True)
    assert rel_err(o, ro) <= 2e-3
    assert rel_err(fs, rfs) <= 2e-3


def test_varlen_equals_separate_calls(gdp):
    lens = [70, 129, 5]
    cu = si.cu_seqlens_of(lens)
    T = int(cu[-1])
    q, k, v, beta, g = chunk_case(1, T, 2, 2, 64, 64, 2, seed=5)
    o, fs = _run(gdp, q, k, v, beta, g, 2, 64, True, cu=cu)
    for i in range(len(lens)):
        t0, t1 = int(cu[i]), int(cu[i + 1])
        oi, fi = _run(gdp, q[:, t0:t1], k[:, 2 * t0:2 * t1], v[:, 2 * t0:2 * t1],
                      beta[:, 2 * t0:2 * t1], g[:, t0:t1], 2, 64, True)
        assert rel_err(o[:, t0:t1], oi) <= 1e-5
        assert rel_err(fs[i:i + 1], fi) <= 1e-5


def test_gva_equals_repeated_heads(gdp):
    q, k, v, beta, g = chunk_case(1, 140, 2, 8, 64, 64, 2, seed=6)
    o, fs = _run(gdp, q, k, v, beta, g, 2, 64, True)
    o2, fs2 = _run(gdp, q.repeat_interleave(4, 2), k.repeat_interleave(4, 2), v, beta, g, 2, 64,
                   True)
    assert rel_err(o, o2) <= 1e-5 and rel_err(fs, fs2) <= 1e-5


def test_deterministic_and_causal(gdp):
    q, k, v, beta, g = chunk_case(1, 160, 2, 2, 128, 128, 2, seed=8)
    o1, f1 = _run(gdp, q, k, v, beta, g, 2, 64, True)
    o2, f2 = _run(gdp, q, k, v, beta, g, 2, 64, True)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    t = 100  # perturb token t and everything after; outputs before t must not move
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[:, t:] = -q2[:, t:]
    k2[:, 2 * t:] = k2[:, 2 * t:].flip(-1)
    v2[:, 2 * t:] *= 3
    o3, _ = _run(gdp, q2, k2, v2, beta, g, 2, 64, True)
    assert rel_err(o3[:, :t], o1[:, :t]) <= 1e-6
    assert rel_err(o3[:, t:], o1[:, t:]) > 1e-2


def test_continuation_through_initial_state(gdp):
    q, k, v, beta, g = chunk_case(1, 200, 2, 2, 64, 64, 2, seed=9)
    o, fs = _run(gdp, q, k, v, beta, g, 2, 64, True)
    oa, fa = _run(gdp, q[:, :77], k[:, :154], v[:, :154], beta[:, :154], g[:, :77], 2, 64, True)
    ob, fb = _run(gdp, q[:, 77:], k[:, 154:], v[:, 154:], beta[:, 154:], g[:, 77:], 2, 64, True,
                  h0=fa)
    assert rel_err(torch.cat([oa, ob], 1), o) <= 2e-3
    assert rel_err(fb, fs) <= 2e-3


@pytest.mark.parametrize("M", [1, 2, 3])
def test_continuation_at_a_chunk_boundary_is_exact(gdp, M):
    """Tensor-core path: a sequence split at a token-chunk boundary (128 tokens)
    and continued through initial_state gives the single call's outputs and
    final state bit for bit (the state crosses the split in fp32, and every WY
    block and output chunk of the second call is one of the single call's)."""
    T, T1 = 320, 128
    q, k, v, beta, g = chunk_case(1, T, 2, 4, 128, 128, M, seed=47)
    o, fs = _run(gdp, q, k, v, beta, g, M, 64, True)
    E1 = T1 * M
    oa, fa = _run(gdp, q[:, :T1], k[:, :E1], v[:, :E1], beta[:, :E1], g[:, :T1], M, 64, True)
    ob, fb = _run(gdp, q[:, T1:], k[:, E1:], v[:, E1:], beta[:, E1:], g[:, T1:], M, 64, True,
                  h0=fa)
    assert torch.equal(torch.cat([oa, ob], 1), o)
    assert torch.equal(fb, fs)


def test_empty_inputs(gdp):
    q, k, v, beta, g = chunk_case(1, 0, 2, 2, 32, 32, 2, seed=1, dtype=torch.float32)
    o, fs = _run(gdp, q, k, v, beta, g, 2, 64, False)
    assert o.numel() == 0 and torch.count_nonzero(fs) == 0
    cu = torch.zeros(1, dtype=torch.int32)  # no sequences at all
    q, k, v, beta, g = chunk_case(1, 4, 2, 2, 32, 32, 2, seed=1, dtype=torch.float32)
    qd, kd, vd, bd, gd, cd = to(DEV, q, k, v, beta, g, cu)
    o, fs = gdp.gdp_chunk_fwd(qd, kd, vd, bd, gd, cu_seqlens=cd, num_householder=2)
    assert fs.numel() == 0


@pytest.mark.parametrize("K,V,M,dtype", [(32, 32, 2, torch.float32), (128, 128, 2, torch.bfloat16),
                                         (128, 128, 3, torch.bfloat16)])
@pytest.mark.parametrize("cu_list", [[0, 6, 4], [1, 5, 9], [0, 5, 400]],
                         ids=["decreasing", "nonzero_start", "past_end"])
def test_bad_seqlens_reported_on_device(gdp, K, V, M, dtype, cu_list):
    """A bad offset list sets the status word; o keeps its canaries and the final
    state is the initial state. The workspace starts as garbage (0xA5 bytes), so
    nothing may depend on a previous call's tables."""
    T = 300
    q, k, v, beta, g = chunk_case(1, T, 2, 2, K, V, M, seed=1, dtype=dtype)
    cu = torch.tensor(cu_list, dtype=torch.int32)
    h0 = torch.randn(2, 2, K, V, generator=torch.Generator().manual_seed(2))
    qd, kd, vd, bd, gd, cd, hd = to(DEV, q, k, v, beta, g, cu, h0)
    need = gdp.gdp_chunk_fwd_workspace_size(1, T, 2, 2, 2, K, V, M, 64, dtype)
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device=DEV)
    o = torch.full((1, T, 2, V), float("nan"), device=DEV)
    fs = torch.full((2, 2, K, V), float("nan"), device=DEV)
    gdp.gdp_chunk_fwd(qd, kd, vd, bd, gd, cu_seqlens=cd, num_householder=M, initial_state=hd,
                      use_qk_l2norm=True, workspace=ws, out=(o, fs))
    assert gdp.gdp_read_status(ws) == 1
    assert torch.isnan(o).all()
    assert torch.equal(fs.cpu(), h0)


# ---------------------------------------------------------------------------------
# stage-by-stage parity against the chunked WY restatement
# ---------------------------------------------------------------------------------
@pytest.mark.parametrize("K,V,M,dtype", [(32, 48, 3, torch.float32), (128, 128, 2, torch.bfloat16)])
def test_stages_match_chunked_restatement(gdp, K, V, M, dtype):
    B, T, H, HV, BT = 1, 150, 2, 2, 64
    q, k, v, beta, g = chunk_case(B, T, H, HV, K, V, M, seed=21, dtype=dtype)
    qd, kd, vd, bd, gd = to(DEV, q, k, v, beta, g)
    need = gdp.gdp_chunk_fwd_workspace_size(B, T, B, H, HV, K, V, M, BT, dtype)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    gdp.gdp_chunk_fwd(qd, kd, vd, bd, gd, chunk_size=BT, num_householder=M, use_qk_l2norm=True,
                      workspace=ws)
    torch.cuda.synchronize()
    off = gdp.gdp_chunk_fwd_stage_offsets(B, T, B, H, HV, K, V, M, BT, dtype)
    Te = B * T * M
    NONE = (1 << 64) - 1
    WY = off[6]  # WY block length of the selected path (A, w, u live on these blocks)

    def view(i, shape):
        return ws[off[i]:off[i] + 4 * int(torch.tensor(shape).prod())].view(torch.float32).view(
            *shape).cpu().double()

    for hv in range(HV):
        f = lambda x: x.double().numpy()
        ref = oracle.chunked_stream(f(q[0, :, hv]), f(k[0, :, hv]), f(v[0, :, hv]),
                                    f(beta[0, :, hv]), f(g[0, :, hv]), M, BT, K ** -0.5,
                                    l2norm=True)
        wyref = ref if WY == BT else oracle.chunked_stream(
            f(q[0, :, hv]), f(k[0, :, hv]), f(v[0, :, hv]), f(beta[0, :, hv]), f(g[0, :, hv]),
            M, WY, K ** -0.5, l2norm=True)
        if off[0] != NONE:
            A = view(0, (Te, HV, WY))[:, hv]
            for c, Ac in enumerate(wyref["A"]):
                n = Ac.shape[0]
                assert rel_err(A[c * WY:c * WY + n, :n], torch.from_numpy(Ac)) <= 1e-5
        for name, idx, width in (("w", 1, K), ("u", 2, V), ("v_new", 3, V)):
            if off[idx] != NONE:
                got = view(idx, (Te, HV, width))[:, hv]
                want = (wyref if name != "v_new" else ref)[name]
                assert rel_err(got, torch.from_numpy(want)) <= 1e-4, name
        if off[4] != NONE:
            hs = view(4, (-(-T // BT), HV, K, V))[:, hv]
            for c in range(hs.shape[0]):
                want = torch.from_numpy(ref["h_chunks"][c * M])
                if want.abs().max() > 0:
                    assert rel_err(hs[c], want) <= 1e-4


# ---------------------------------------------------------------------------------
# full-size workloads, launched as the benchmark launches them, compared element
# by element with the oracle's fp64 walk of every (sequence, value head) unit
# (OpenMP over the units on the host cores)
# ---------------------------------------------------------------------------------
def _check_all(o, fs, q, k, v, beta, g, M, l2=True, cu=None):
    ro, rfs = oracle.walk(q, k, v, beta, g, M, q.shape[3] ** -0.5, cu_seqlens=cu, l2norm=l2)
    n = o.shape[1] if cu is None else int(cu[-1])
    assert rel_err(o[:, :n], ro[:, :n]) <= 2e-3, rel_err(o[:, :n], ro[:, :n])
    assert rel_err(fs, rfs) <= 2e-3, rel_err(fs, rfs)
    # per-unit bound as well: a bad unit cannot hide behind the global RMS
    for s_ in range(fs.shape[0]):
        for hv in range(fs.shape[1]):
            assert rel_err(fs[s_, hv], rfs[s_, hv]) <= 2e-3, (s_, hv)


def test_prefill_bf16_workload(gdp):
    w = si.WORKLOADS["prefill_bf16"].dims
    q, k, v, beta, g = chunk_case(w["B"], w["T"], w["H"], w["HV"], w["K"], w["V"], w["M"], seed=0)
    o, fs = _run(gdp, q, k, v, beta, g, w["M"], w["BT"], True)
    assert torch.isfinite(o).all()
    _check_all(o, fs, q, k, v, beta, g, w["M"])


@pytest.mark.parametrize("T,H,HV,V", [(4096, 8, 8, 128), (2100, 2, 8, 256)])
def test_persistent_wy_loop_many_items_per_cta(gdp, T, H, HV, V):
    """M=2, K=128: 520 (V = 128) or 264 (V = 256, GVA, a partial last block per
    head) (128-position block, head) items, more than the persistent WY grid, so
    every CTA runs the next-item loads (for V = 256 also the second value round
    through the k buffer), the buffer reuse and the next item's decay prefix
    more than once."""
    q, k, v, beta, g = chunk_case(1, T, H, HV, 128, V, 2, seed=12)
    o, fs = _run(gdp, q, k, v, beta, g, 2, 64, True)
    _check_all(o, fs, q, k, v, beta, g, 2)


@pytest.mark.parametrize("M,V", [(1, 128), (3, 128), (3, 256)])
def test_persistent_output_loop_many_items_per_cta(gdp, M, V):
    """Odd M, K=128, ragged sequences (one empty, one of a single token): 360
    (V = 128) or 720 (V = 256) (token chunk, value head, 64-column slice) items
    for the persistent output kernel, padding chunks among them, so every CTA
    skips padding, alternates its two TMEM column sets and runs the next-item
    loads, products and norms more than once."""
    lens = [700, 0, 1, 1199, 600]
    cu = si.cu_seqlens_of(lens)
    q, k, v, beta, g = chunk_case(1, sum(lens), 2, 4, 128, V, M, seed=15)
    o, fs = _run(gdp, q, k, v, beta, g, M, 64, True, cu=cu)
    _check_all(o, fs, q, k, v, beta, g, M, cu=cu)


@pytest.mark.parametrize("M", [1, 2, 3])
def test_packed_equal_lengths_equal_dense_batch(gdp, M):
    """B equal-length sequences packed through cu_seqlens give the dense batch's
    outputs bit for bit: the device tables (closed form for the dense batch, the
    offset scan for the packed one) and the scan's launch order (grid order
    against longest first) change nothing in any sequence's arithmetic."""
    B, T, H, HV = 3, 333, 2, 4
    q, k, v, beta, g = chunk_case(B, T, H, HV, 128, 128, M, seed=41)
    h0 = torch.randn(B, HV, 128, 128, generator=torch.Generator().manual_seed(5))
    o_d, fs_d = _run(gdp, q, k, v, beta, g, M, 64, True, h0=h0)
    flat = lambda x: x.reshape(1, -1, *x.shape[2:])
    cu = torch.arange(0, B * T + 1, T, dtype=torch.int32)
    o_p, fs_p = _run(gdp, flat(q), flat(k), flat(v), flat(beta), flat(g), M, 64, True, h0=h0, cu=cu)
    assert torch.equal(o_p.reshape(o_d.shape), o_d)
    assert torch.equal(fs_p, fs_d)


@pytest.mark.parametrize("M", [1, 2, 3])
def test_gva_equals_repeated_key_heads(gdp, M):
    """HV = 4 H value heads reading key/query head hv / 4 give, bit for bit, the
    outputs of the same call with the key and query heads repeated to H = HV
    (wy_fast page, GVA parameters: the kernels only index the key head)."""
    B, T, H, HV, V = 2, 300, 2, 8, 256
    q, k, v, beta, g = chunk_case(B, T, H, HV, 128, V, M, seed=43)
    o_g, fs_g = _run(gdp, q, k, v, beta, g, M, 64, True)
    rep = lambda x: x.repeat_interleave(HV // H, dim=2)
    o_r, fs_r = _run(gdp, rep(q), rep(k), v, beta, g, M, 64, True)
    assert torch.equal(o_g, o_r)
    assert torch.equal(fs_g, fs_r)


@pytest.mark.parametrize("M", [2, 3])
def test_long_single_sequence(gdp, M):
    """One 32768-token sequence (65536 or 98304 expanded positions): a state chain
    of 512 (M = 2, 128-position blocks) or 1536 (M = 3, 64-position steps) steps
    and token / position coordinates far from zero, element by element."""
    q, k, v, beta, g = chunk_case(1, 32768, 1, 1, 128, 128, M, seed=31)
    o, fs = _run(gdp, q, k, v, beta, g, M, 64, True)
    _check_all(o, fs, q, k, v, beta, g, M)


@pytest.mark.parametrize("M", [2, 3])
def test_tensor_core_ungated(gdp, M):
    """g = None on the bf16 tensor-core path (no decay anywhere)."""
    q, k, v, beta, _ = chunk_case(1, 900, 2, 4, 128, 128, M, seed=13)
    o, fs = _run(gdp, q, k, v, beta, None, M, 64, True)
    _check_all(o, fs, q, k, v, beta, None, M)


def test_gva_bf16_workload(gdp):
    w = si.WORKLOADS["gva_bf16"].dims
    q, k, v, beta, g = chunk_case(w["B"], w["T"], w["H"], w["HV"], w["K"], w["V"], w["M"], seed=0)
    o, fs = _run(gdp, q, k, v, beta, g, w["M"], w["BT"], True)
    assert torch.isfinite(o).all()
    for b in range(w["B"]):  # one batch row at a time bounds the oracle's fp64 copies
        sl = slice(b, b + 1)
        _check_all(o[sl], fs[sl], q[sl], k[sl], v[sl], beta[sl], g[sl], w["M"])


def test_varlen_workload_from_prepare(gdp):
    w = si.WORKLOADS["varlen_bf16"].dims
    lens = si.varlen_lengths(w["n_seq"], seed=0)
    cu = si.cu_seqlens_of(lens)
    T = int(cu[-1])
    M, H, G, P, N = w["M"], w["H"], w["G"], w["P"], w["N"]
    d = si.prepare_inputs(1, T, M, H, G, P, N, seed=0)
    q, k, v, beta, g = gdp.gdp_prefill_prepare(d["x"].to(DEV), d["ba"].to(DEV),
                                               d["A_log"].to(DEV), d["dt_bias"].to(DEV), M, H,
                                               G, P, N)
    o, fs = gdp.gdp_chunk_fwd(q, k, v, beta, g, cu_seqlens=cu.to(DEV), chunk_size=w["BT"],
                              num_householder=M, use_qk_l2norm=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all()
    # the oracle walks its own prepare of the same raw inputs
    rq, rk, rv, rb, rg = oracle.prepare(d["x"], d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N,
                                        decode=False)
    _check_all(o.cpu(), fs.cpu(), rq, rk, rv, rb, rg, M, cu=cu)


def test_bounded_wait_runs_out_and_reports_timeout(gdp):
    """Device-side failure path without a GPU fault: the test hook leaves one
    tensor-core commit out of the WY kernel's first CTA and shortens the wait
    budget to 50 ms, so that CTA's bounded wait runs out. The call must return,
    the workspace status word must read GDP_ERR_DEVICE_TIMEOUT, and the next
    normal call must be correct."""
    import time
    B, T, H, HV, K, V, M = 1, 300, 2, 2, 128, 128, 2
    q, k, v, beta, g = chunk_case(B, T, H, HV, K, V, M, seed=14)
    qd, kd, vd, bd, gd = to(DEV, q, k, v, beta, g)
    need = gdp.gdp_chunk_fwd_workspace_size(B, T, B, H, HV, K, V, M, 64, torch.bfloat16)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    try:
        gdp.gdp_debug_wait_fault(True, 0.05)
        t0 = time.time()
        gdp.gdp_chunk_fwd(qd, kd, vd, bd, gd, chunk_size=64, num_householder=M,
                          use_qk_l2norm=True, workspace=ws)
        status = gdp.gdp_read_status(ws)  # synchronises
        elapsed = time.time() - t0
    finally:
        gdp.gdp_debug_wait_fault(False, 0.0)
    assert status == 4, status  # GDP_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0, elapsed
    ws2 = torch.zeros_like(ws)
    o, fs = gdp.gdp_chunk_fwd(qd, kd, vd, bd, gd, chunk_size=64, num_householder=M,
                              use_qk_l2norm=True, workspace=ws2)
    assert gdp.gdp_read_status(ws2) == 0
    ro, rfs = oracle.walk(q, k, v, beta, g, M, K ** -0.5, l2norm=True)
    assert rel_err(o, ro) <= 2e-3 and rel_err(fs, rfs) <= 2e-3
