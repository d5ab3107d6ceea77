"""Pins for the CPU oracle: each test ties it to something other than itself.

Sources: the prepare page (softplus definition, gate formulas, copy placement
for decode and prefill), the chunk_o page (queries on the unexpanded stream,
keys/values on the expanded one, summed over the copies) and the wy_fast page
(WY factors from the inverted transition block), plus the mathematics of the
gated delta rule. None of these tests touches a GPU.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si

RNG = np.random.default_rng(1234)


def _rand_case(B=1, T=6, H=2, HV=2, K=4, V=3, M=2, seed=0, gated=True):
    r = np.random.default_rng(seed)
    q = torch.from_numpy(r.standard_normal((B, T, H, K)))
    k = torch.from_numpy(r.standard_normal((B, T * M, H, K)))
    v = torch.from_numpy(r.standard_normal((B, T * M, HV, V)))
    beta = torch.from_numpy(r.uniform(0.05, 0.95, (B, T * M, HV)))
    g = torch.from_numpy(-r.uniform(0.0, 1.0, (B, T, HV))) if gated else None
    return q, k, v, beta, g


def _unit(x):
    return x / np.linalg.norm(x)


# ----------------------------------------------------------------------------------
# 1. Per-token product form (DeltaProduct: one token's transition is the product of
#    its M generalised Householder factors; decay on the first copy, query read
#    after the last) -- an explicit-matrix formula, not the oracle's rank-1 loop.
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 2, 3])
def test_walk_matches_per_token_product_form(M):
    B, T, H, HV, K, V = 1, 5, 1, 2, 4, 3
    q, k, v, beta, g = _rand_case(B, T, H, HV, K, V, M, seed=M)
    h0 = torch.from_numpy(RNG.standard_normal((1, HV, K, V)))
    scale = 0.7
    o, hT = oracle.walk(q, k, v, beta, g, M, scale, h0=h0)
    for hv in range(HV):
        S = h0[0, hv].numpy().T.copy()  # V x K
        for t in range(T):
            Hs = [np.eye(K) - beta[0, t * M + j, hv].item()
                  * np.outer(k[0, t * M + j, 0].numpy(), k[0, t * M + j, 0].numpy())
                  for j in range(M)]
            prod_all = np.eye(K)
            for j in range(M):
                prod_all = prod_all @ Hs[j]
            inj = np.zeros((V, K))
            for j in range(M):
                tail = np.eye(K)
                for l in range(j + 1, M):
                    tail = tail @ Hs[l]
                inj += beta[0, t * M + j, hv].item() * np.outer(
                    v[0, t * M + j, hv].numpy(), k[0, t * M + j, 0].numpy()) @ tail
            S = math.exp(g[0, t, hv].item()) * S @ prod_all + inj
            np.testing.assert_allclose(o[0, t, hv].numpy(), scale * S @ q[0, t, 0].numpy(),
                                       rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(hT[0, hv].numpy(), S.T, rtol=1e-12, atol=1e-12)


def test_scalar_case_is_a_decayed_moving_average():
    """K = V = 1, k = 1: S_T = sum_t beta_t v_t prod_{s>t} e^{g_s}(1 - beta_s)
    (closed-form sum of the scalar gated delta rule, M = 1)."""
    T = 9
    r = np.random.default_rng(7)
    beta = r.uniform(0.1, 0.9, T)
    g = -r.uniform(0.0, 0.5, T)
    v = r.standard_normal(T)
    q = torch.ones(1, T, 1, 1, dtype=torch.float64)
    k = torch.ones(1, T, 1, 1, dtype=torch.float64)
    o, hT = oracle.walk(q, k, torch.from_numpy(v).view(1, T, 1, 1),
                        torch.from_numpy(beta).view(1, T, 1),
                        torch.from_numpy(g).view(1, T, 1), 1, 1.0)
    for t_end in range(T):
        want = 0.0
        for t in range(t_end + 1):
            fac = 1.0
            for s in range(t + 1, t_end + 1):
                fac *= math.exp(g[s]) * (1.0 - beta[s])
            want += beta[t] * v[t] * fac
        assert abs(o[0, t_end, 0, 0].item() - want) < 1e-13
    assert abs(hT[0, 0, 0, 0].item() - o[0, T - 1, 0, 0].item()) < 1e-15


# ----------------------------------------------------------------------------------
# 2.-8. Invariants of the recurrence
# ----------------------------------------------------------------------------------
def test_zero_beta_zero_decay_leaves_state_unchanged():
    q, k, v, beta, g = _rand_case(T=7, M=3, seed=3)
    beta.zero_()
    g.zero_()
    h0 = torch.from_numpy(RNG.standard_normal((1, 2, 4, 3)))
    o, hT = oracle.walk(q, k, v, beta, g, 3, 0.5, h0=h0)
    np.testing.assert_allclose(hT.numpy(), h0.numpy(), rtol=0, atol=1e-15)
    for hv in range(2):
        want = 0.5 * q[0, :, hv].numpy() @ h0[0, hv].numpy()  # scale * S0 q, S0 = h0^T (H == HV)
        np.testing.assert_allclose(o[0, :, hv].numpy(), want, atol=1e-14)


def test_unit_key_beta_one_memorises_value():
    """beta = 1, |k| = 1: after the step S k = v exactly, whatever S and g were."""
    K, V = 5, 4
    S0 = RNG.standard_normal((V, K))
    kk = _unit(RNG.standard_normal(K))
    vv = RNG.standard_normal(V)
    q = torch.from_numpy(kk).view(1, 1, 1, K)
    o, hT = oracle.walk(q, q.clone(), torch.from_numpy(vv).view(1, 1, 1, V),
                        torch.ones(1, 1, 1, dtype=torch.float64),
                        torch.full((1, 1, 1), -0.3, dtype=torch.float64), 1, 1.0,
                        h0=torch.from_numpy(S0.T.copy()).view(1, 1, K, V))
    np.testing.assert_allclose(o[0, 0, 0].numpy(), vv, atol=1e-13)
    np.testing.assert_allclose(hT[0, 0].numpy().T @ kk, vv, atol=1e-13)


def test_orthonormal_keys_give_linear_attention_sum():
    """Orthonormal keys, beta = 1, g = 0, S0 = 0 -> S = sum_t v_t k_t^T."""
    K, V, T = 6, 3, 6
    Q, _ = np.linalg.qr(RNG.standard_normal((K, K)))
    keys = Q.T  # rows orthonormal
    vals = RNG.standard_normal((T, V))
    k = torch.from_numpy(keys).view(1, T, 1, K)
    qq = torch.from_numpy(RNG.standard_normal((1, T, 1, K)))
    o, hT = oracle.walk(qq, k, torch.from_numpy(vals).view(1, T, 1, V),
                        torch.ones(1, T, 1, dtype=torch.float64),
                        torch.zeros(1, T, 1, dtype=torch.float64), 1, 1.0)
    S = sum(np.outer(vals[t], keys[t]) for t in range(T))
    np.testing.assert_allclose(hT[0, 0].numpy(), S.T, atol=1e-13)


def test_linear_in_values_and_initial_state():
    q, k, v, beta, g = _rand_case(T=5, M=2, seed=11)
    v2 = torch.from_numpy(RNG.standard_normal(v.shape))
    h0a = torch.from_numpy(RNG.standard_normal((1, 2, 4, 3)))
    h0b = torch.from_numpy(RNG.standard_normal((1, 2, 4, 3)))
    a, b = 0.7, -1.3
    o1, s1 = oracle.walk(q, k, v, beta, g, 2, 1.0, h0=h0a)
    o2, s2 = oracle.walk(q, k, v2, beta, g, 2, 1.0, h0=h0b)
    o3, s3 = oracle.walk(q, k, a * v + b * v2, beta, g, 2, 1.0, h0=a * h0a + b * h0b)
    np.testing.assert_allclose(o3.numpy(), a * o1.numpy() + b * o2.numpy(), atol=1e-12)
    np.testing.assert_allclose(s3.numpy(), a * s1.numpy() + b * s2.numpy(), atol=1e-12)


def test_large_negative_decay_resets_state():
    """g_t -> -inf wipes the state before token t's copies."""
    q, k, v, beta, g = _rand_case(T=8, M=2, seed=5)
    g[0, 4] = -1e4
    o, hT = oracle.walk(q, k, v, beta, g, 2, 1.0,
                        h0=torch.from_numpy(RNG.standard_normal((1, 2, 4, 3))))
    o_tail, h_tail = oracle.walk(q[:, 4:], k[:, 8:], v[:, 8:], beta[:, 8:], g[:, 4:], 2, 1.0)
    np.testing.assert_allclose(o[:, 4:].numpy(), o_tail.numpy(), atol=1e-12)
    np.testing.assert_allclose(hT.numpy(), h_tail.numpy(), atol=1e-12)


def test_reflections_preserve_norm_and_square_to_identity():
    """beta = 2, |k| = 1 is a Householder reflection: orthogonal (Frobenius norm
    kept when v = 0, g = 0), and two equal reflections cancel."""
    K, V, M = 5, 4, 2
    kk = _unit(RNG.standard_normal(K))
    other = _unit(RNG.standard_normal(K))
    S0 = RNG.standard_normal((V, K))
    h0 = torch.from_numpy(S0.T.copy()).view(1, 1, K, V)
    z = lambda *s: torch.zeros(*s, dtype=torch.float64)
    k_same = torch.from_numpy(np.stack([kk, kk])).view(1, M, 1, K)
    _, hT = oracle.walk(z(1, 1, 1, K), k_same, z(1, M, 1, V),
                        torch.full((1, M, 1), 2.0, dtype=torch.float64), z(1, 1, 1), M, 1.0,
                        h0=h0)
    np.testing.assert_allclose(hT[0, 0].numpy(), S0.T, atol=1e-13)
    k_diff = torch.from_numpy(np.stack([kk, other])).view(1, M, 1, K)
    _, hT2 = oracle.walk(z(1, 1, 1, K), k_diff, z(1, M, 1, V),
                         torch.full((1, M, 1), 2.0, dtype=torch.float64), z(1, 1, 1), M, 1.0,
                         h0=h0)
    assert abs(np.linalg.norm(hT2.numpy()) - np.linalg.norm(S0)) < 1e-12


def test_l2norm_flag_is_scale_invariant():
    q, k, v, beta, g = _rand_case(T=6, M=2, seed=9)
    c = torch.from_numpy(RNG.uniform(0.5, 3.0, (1, 6 * 2, 2, 1)))
    cq = torch.from_numpy(RNG.uniform(0.5, 3.0, (1, 6, 2, 1)))
    o1, s1 = oracle.walk(q, k, v, beta, g, 2, 1.0, l2norm=True)
    o2, s2 = oracle.walk(q * cq, k * c, v, beta, g, 2, 1.0, l2norm=True)
    # the 1e-6 inside the sqrt breaks exact invariance by O(1e-6 / |x|^2)
    np.testing.assert_allclose(o1.numpy(), o2.numpy(), atol=1e-5)
    np.testing.assert_allclose(s1.numpy(), s2.numpy(), atol=1e-5)
    o1b, _ = oracle.walk(q, k, v, beta, g, 2, 1.0, l2norm=False)
    assert np.abs(o1b.numpy() - o1.numpy()).max() > 1e-2  # the flag does act
    # with unit-norm inputs the flag changes nothing beyond the 1e-6 epsilon
    qn = q / q.norm(dim=-1, keepdim=True)
    kn = k / k.norm(dim=-1, keepdim=True)
    o3, _ = oracle.walk(qn, kn, v, beta, g, 2, 1.0, l2norm=True)
    o4, _ = oracle.walk(qn, kn, v, beta, g, 2, 1.0, l2norm=False)
    np.testing.assert_allclose(o3.numpy(), o4.numpy(), atol=1e-5)


# ----------------------------------------------------------------------------------
# 9. Decompositions: varlen = separate sequences, GVA = repeated heads,
#    continuation through the final state, decode walk = prefill walk.
# ----------------------------------------------------------------------------------
def test_varlen_equals_separate_sequences():
    lens = [3, 1, 5, 0, 4]
    cu = si.cu_seqlens_of(lens)
    T = int(cu[-1])
    q, k, v, beta, g = _rand_case(B=1, T=T, M=2, seed=21)
    h0 = torch.from_numpy(RNG.standard_normal((len(lens), 2, 4, 3)))
    o, hT = oracle.walk(q, k, v, beta, g, 2, 0.9, cu_seqlens=cu, h0=h0, l2norm=True)
    for i, (t0, t1) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())):
        oi, hi = oracle.walk(q[:, t0:t1], k[:, 2 * t0:2 * t1], v[:, 2 * t0:2 * t1],
                             beta[:, 2 * t0:2 * t1], g[:, t0:t1], 2, 0.9, h0=h0[i:i + 1],
                             l2norm=True)
        np.testing.assert_allclose(o[:, t0:t1].numpy(), oi.numpy(), atol=1e-13)
        np.testing.assert_allclose(hT[i].numpy(), hi[0].numpy(), atol=1e-13)


def test_gva_equals_repeated_key_heads():
    B, T, H, HV, K, V, M = 2, 5, 2, 6, 4, 3, 2
    q, k, v, beta, g = _rand_case(B, T, H, HV, K, V, M, seed=4)
    o, hT = oracle.walk(q, k, v, beta, g, M, 1.0)
    rep = HV // H
    o2, h2 = oracle.walk(q.repeat_interleave(rep, dim=2), k.repeat_interleave(rep, dim=2),
                         v, beta, g, M, 1.0)
    np.testing.assert_allclose(o.numpy(), o2.numpy(), atol=1e-14)
    np.testing.assert_allclose(hT.numpy(), h2.numpy(), atol=1e-14)


def test_continuation_through_final_state():
    q, k, v, beta, g = _rand_case(T=9, M=3, seed=8)
    o, hT = oracle.walk(q, k, v, beta, g, 3, 1.0)
    oa, ha = oracle.walk(q[:, :4], k[:, :12], v[:, :12], beta[:, :12], g[:, :4], 3, 1.0)
    ob, hb = oracle.walk(q[:, 4:], k[:, 12:], v[:, 12:], beta[:, 12:], g[:, 4:], 3, 1.0, h0=ha)
    np.testing.assert_allclose(o.numpy(), torch.cat([oa, ob], 1).numpy(), atol=1e-13)
    np.testing.assert_allclose(hT.numpy(), hb.numpy(), atol=1e-13)


def test_decode_walk_equals_prefill_walk_on_placed_copies():
    """Placing q on the last copy and g on the first (prepare page, decode bullet)
    and stepping every copy gives the prefill walk's outputs at the last copies."""
    B, T, H, HV, K, V, M = 2, 4, 2, 2, 4, 3, 3
    q, k, v, beta, g = _rand_case(B, T, H, HV, K, V, M, seed=13)
    h0 = torch.from_numpy(RNG.standard_normal((B, HV, K, V)))
    o, hT = oracle.walk(q, k, v, beta, g, M, 0.8, h0=h0, l2norm=True)
    qd = torch.zeros(B, T * M, H, K, dtype=torch.float64)
    qd[:, M - 1::M] = q
    gd = torch.zeros(B, T * M, HV, dtype=torch.float64)
    gd[:, 0::M] = g
    od, sd = oracle.recurrent(qd, k, v, beta, gd, h0, 0.8, l2norm=True)
    np.testing.assert_allclose(od[:, M - 1::M].numpy(), o.numpy(), atol=1e-13)
    np.testing.assert_allclose(sd.numpy(), hT.numpy(), atol=1e-13)
    assert torch.count_nonzero(od.view(B, T, M, HV, V)[:, :, :M - 1]) == 0


# ----------------------------------------------------------------------------------
# Chunked WY form (second algorithm) == token walk, for every chunk size
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("M,BT,T", [(1, 8, 40), (2, 16, 40), (3, 16, 50), (3, 7, 37),
                                    (2, 64, 64), (2, 1, 9), (3, 3, 10), (2, 100, 30),
                                    (1, 64, 0)])
def test_chunked_matches_walk(M, BT, T):
    K, V = 5, 4
    q, k, v, beta, g = _rand_case(1, T, 1, 1, K, V, M, seed=M * 100 + BT)
    h0 = torch.from_numpy(RNG.standard_normal((1, 1, K, V)))
    o, hT = oracle.walk(q, k, v, beta, g, M, 0.6, h0=h0, l2norm=True)
    res = oracle.chunked_stream(q[0, :, 0].numpy(), k[0, :, 0].numpy(), v[0, :, 0].numpy(),
                                beta[0, :, 0].numpy(), g[0, :, 0].numpy(), M, BT, 0.6,
                                h0=h0[0, 0].numpy(), l2norm=True)
    np.testing.assert_allclose(res["o"], o[0, :, 0].numpy(), atol=1e-11)
    np.testing.assert_allclose(res["h_final"], hT[0, 0].numpy(), atol=1e-11)


def test_solve_tril_inverse_and_wy_stage_identities():
    q, k, v, beta, g = _rand_case(1, 32, 1, 1, 6, 5, 2, seed=2)
    res = oracle.chunked_stream(q[0, :, 0].numpy(), k[0, :, 0].numpy(), v[0, :, 0].numpy(),
                                beta[0, :, 0].numpy(), g[0, :, 0].numpy(), 2, 16, 1.0)
    for Lm, A in zip(res["L"], res["A"]):
        n = Lm.shape[0]
        assert np.allclose(np.triu(Lm), 0.0)           # strictly lower
        assert np.allclose(np.diag(A), 1.0) and np.allclose(np.triu(A, 1), 0.0)
        np.testing.assert_allclose(A @ (np.eye(n) + Lm), np.eye(n), atol=1e-12)
        np.testing.assert_allclose(np.linalg.inv(np.eye(n) + Lm), A, atol=1e-12)
    # v_new is the per-position delta beta_p (v_p - e^{g_p} S_{p-1} k_p): chunk-size free
    r1 = oracle.chunked_stream(q[0, :, 0].numpy(), k[0, :, 0].numpy(), v[0, :, 0].numpy(),
                               beta[0, :, 0].numpy(), g[0, :, 0].numpy(), 2, 5, 1.0)
    np.testing.assert_allclose(r1["v_new"], res["v_new"], atol=1e-12)


# ----------------------------------------------------------------------------------
# Prepare map (fp32)
# ----------------------------------------------------------------------------------
def _f32_ulp_diff(a, b):
    ai = a.contiguous().view(torch.int32).to(torch.int64)
    bi = b.contiguous().view(torch.int32).to(torch.int64)
    ai = torch.where(ai < 0, -(ai & 0x7FFFFFFF), ai)
    bi = torch.where(bi < 0, -(bi & 0x7FFFFFFF), bi)
    return (ai - bi).abs()


def test_softplus_page_values():
    """Golden values from the prepare page's softplus section (identity above 20,
    log1p keeps the far-negative tail), stored in tests/golden/softplus_page.txt."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "softplus_page.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    for x_s, kind, want_s in rows:
        x = float(x_s)
        a = torch.tensor([[x]], dtype=torch.float32)  # a + dt_bias with dt_bias = 0
        _, g = oracle.gate_map(torch.zeros(1, 1), a, torch.zeros(1), torch.zeros(1))
        sp = -g.item()  # g = -exp(0) * softplus(x)
        if kind == "identity":
            assert sp == np.float32(float(want_s))
        else:  # "exp": softplus(x) ~ e^x in the far-negative tail, to a few ulp
            want = np.float32(math.exp(x))
            assert want > 0 and abs(sp - want) <= 4 * np.spacing(want)


def test_gates_against_library_routines():
    b = torch.linspace(-30, 30, 4001, dtype=torch.float32).view(-1, 1)
    a = torch.linspace(-40, 40, 4001, dtype=torch.float32).view(-1, 1)
    beta, g = oracle.gate_map(b, a, torch.tensor([0.3]), torch.tensor([0.0]))
    from scipy.special import expit
    want_beta = torch.from_numpy(expit(b.view(-1).double().numpy()))
    assert torch.all(_f32_ulp_diff(beta.view(-1), want_beta.float()) <= 4)
    sp = [x if x > 20 else math.log1p(math.exp(x)) for x in a.view(-1).tolist()]
    want_g = torch.tensor([-math.exp(float(np.float32(0.3))) * s for s in sp]).float()
    assert torch.all(_f32_ulp_diff(g.view(-1), want_g) <= 4)
    b0, _ = oracle.gate_map(torch.zeros(1, 1), torch.zeros(1, 1), torch.zeros(1), torch.zeros(1))
    assert b0.item() == 0.5  # sigmoid(0) exactly
    assert torch.all(g <= 0) and torch.all((beta > 0) & (beta < 1) | (b.abs() > 16))


def _tiny_prepare(M, H, G, P, N, n=2, T=3, dtype=torch.float32, strided=True):
    D = M * H * P + M * G * N + G * N
    # every element distinct: its own flat index (exact in fp32)
    base = torch.arange(n * T * D, dtype=torch.float32).view(n, T, D)
    if strided:
        big = torch.zeros(n, T, D + 8, dtype=dtype)
        big[..., :D] = base.to(dtype)
        x = big[..., :D]
    else:
        x = base.to(dtype)
    r = np.random.default_rng(3)
    ba_full = torch.from_numpy(r.standard_normal((n, T, M * H + H + 3))).to(dtype)
    ba = ba_full[..., :M * H + H]
    A_log = torch.from_numpy(r.uniform(0, math.log(16), H)).float()
    dt_bias = torch.from_numpy(r.normal(0, 0.5, H)).float()
    return x, ba, A_log, dt_bias


@pytest.mark.parametrize("M,H,G", [(1, 2, 1), (2, 4, 2), (3, 4, 4), (2, 6, 3)])
def test_prepare_decode_and_prefill_agree(M, H, G):
    P, N = 3, 2
    x, ba, A_log, dt_bias = _tiny_prepare(M, H, G, P, N)
    qd, kd, vd, bd, gd = oracle.prepare(x, ba, A_log, dt_bias, M, H, G, P, N, decode=True)
    qp, kp, vp, bp, gp = oracle.prepare(x, ba, A_log, dt_bias, M, H, G, P, N, decode=False)
    n, T = x.shape[:2]
    assert torch.equal(kd, kp) and torch.equal(vd, vp) and torch.equal(bd, bp)
    assert torch.equal(qd[:, M - 1::M], qp) and torch.equal(gd[:, 0::M], gp)
    for j in range(M - 1):
        assert torch.count_nonzero(qd[:, j::M]) == 0
    for j in range(1, M):
        assert torch.count_nonzero(gd[:, j::M]) == 0
    # the gates equal the standalone gate map
    bb, gg = oracle.gate_map(ba[..., :M * H].float().reshape(n, T * M, H), ba[..., M * H:].float(),
                             A_log, dt_bias)
    assert torch.equal(bb, bp) and torch.equal(gg, gp)


@pytest.mark.parametrize("M,H,G", [(2, 4, 2), (3, 6, 3)])
def test_prepare_copies_are_a_bijection_of_the_blocks(M, H, G):
    """value output is the value block of every row, each element once; every
    key/query group row appears H/G times; nothing else is copied."""
    P, N = 4, 2
    x, ba, A_log, dt_bias = _tiny_prepare(M, H, G, P, N)
    q, k, v, _, _ = oracle.prepare(x, ba, A_log, dt_bias, M, H, G, P, N, decode=False)
    n, T, D = x.shape
    vb = x[..., :M * H * P]
    assert torch.equal(torch.sort(v.flatten()).values, torch.sort(vb.flatten()).values)
    kb = x[..., M * H * P:M * H * P + M * G * N]
    hpg = H // G
    assert torch.equal(torch.sort(k.flatten()).values,
                       torch.sort(kb.flatten().repeat_interleave(1).repeat(hpg)).values)
    qb = x[..., M * H * P + M * G * N:]
    assert torch.equal(torch.sort(q.flatten()).values, torch.sort(qb.flatten().repeat(hpg)).values)
    # heads sharing a group hold identical rows; heads in different groups do not
    for h in range(H):
        assert torch.equal(k[:, :, h], k[:, :, (h // hpg) * hpg])
    if G > 1:
        assert not torch.equal(k[:, :, 0], k[:, :, hpg])
    # per expanded row, the value is one contiguous run of the token's value block
    for t in range(T):
        for j in range(M):
            assert torch.equal(v[0, t * M + j].flatten(), vb[0, t, j * H * P:(j + 1) * H * P])


def test_prepare_bf16_copies_are_bit_moves():
    M, H, G, P, N = 2, 4, 2, 8, 8
    d = si.prepare_inputs(2, 5, M, H, G, P, N, seed=3)
    q, k, v, beta, g = oracle.prepare(d["x"], d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N,
                                      decode=False)
    assert q.dtype == torch.bfloat16 and k.dtype == torch.bfloat16 and v.dtype == torch.bfloat16
    assert beta.dtype == torch.float32 and g.dtype == torch.float32
    assert torch.equal(v.view(2, 5, -1), d["x"][..., :M * H * P])


# ---------------------------------------------------------------------------------
# the short causal conv before prepare (oracle.conv): pins against library
# routines and the conv's invariants
# ---------------------------------------------------------------------------------
def _conv_inputs(n, T, C, W, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, T, C, generator=g).to(dtype)
    w = torch.randn(C, W, generator=g) * 0.5
    b = torch.randn(C, generator=g) * 0.1
    return x, w, b


def test_conv_width_one_is_silu():
    x, _, _ = _conv_inputs(2, 9, 16, 1, 1)
    y, st = oracle.conv(x, torch.ones(16, 1), None)
    ref = torch.nn.functional.silu(x)  # library SiLU
    assert st.shape == (2, 16, 0)
    assert (y - ref).abs().max() <= 4e-7 * ref.abs().max()


@pytest.mark.parametrize("W", [2, 3, 4])
def test_conv_matches_numpy_correlation(W):
    """z = b + sum_i w[i] x[t-(W-1)+i] with zeros before the sequence is a valid
    cross-correlation of the zero-padded input with the taps (numpy's routine)."""
    n, T, C = 2, 11, 6
    x, w, b = _conv_inputs(n, T, C, W, W)
    y, _ = oracle.conv(x, w, b)
    xd = x.double().numpy()
    for r in range(n):
        for c in range(C):
            xpad = np.concatenate([np.zeros(W - 1), xd[r, :, c]])
            z = np.correlate(xpad, w[c].double().numpy(), "valid") + float(b[c])
            ref = z / (1.0 + np.exp(-z))
            assert np.abs(y[r, :, c].double().numpy() - ref).max() <= 2e-6 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("tap", [0, 1, 3])
def test_conv_one_hot_tap_shifts_and_reads_the_state_oldest_first(tap):
    """With w = e_tap and no bias, y[t] = silu(xin[t - 3 + tap]); positions before
    the sequence come from the state, entry W-1+t (oldest first)."""
    W, T, C = 4, 6, 5
    x, _, _ = _conv_inputs(1, T, C, W, 10 + tap)
    state = torch.randn(1, C, W - 1, generator=torch.Generator().manual_seed(3))
    w = torch.zeros(C, W)
    w[:, tap] = 1.0
    y, st = oracle.conv(x, w, None, state=state)
    full = torch.cat([state[0].t(), x[0]], 0)  # [W-1+T, C]: state entries, then tokens
    want = torch.nn.functional.silu(full[tap:tap + T])
    assert (y[0] - want).abs().max() <= 4e-7 * want.abs().max()
    assert torch.equal(st[0], full[-(W - 1):].t())  # last W-1 inputs, oldest first


def test_conv_chained_calls_equal_one_call_and_varlen_equals_separate():
    W, C = 4, 8
    x, w, b = _conv_inputs(1, 20, C, W, 21, dtype=torch.bfloat16)
    y, st = oracle.conv(x, w, b)
    y1, s1 = oracle.conv(x[:, :2], w, b)            # shorter than W - 1
    y2, s2 = oracle.conv(x[:, 2:13], w, b, state=s1)
    y3, s3 = oracle.conv(x[:, 13:], w, b, state=s2)
    assert torch.equal(torch.cat([y1, y2, y3], 1), y) and torch.equal(s3, st)
    cu = torch.tensor([0, 2, 2, 13, 20], dtype=torch.int32)  # with an empty sequence
    h0 = torch.randn(4, C, W - 1).to(torch.bfloat16)
    yv, sv = oracle.conv(x, w, b, state=h0, cu_seqlens=cu)
    for i in range(4):
        t0, t1 = int(cu[i]), int(cu[i + 1])
        yi, si = oracle.conv(x[:, t0:t1], w, b, state=h0[i:i + 1])
        assert torch.equal(yv[:, t0:t1], yi) and torch.equal(sv[i], si[0])
    assert torch.equal(sv[1], h0[1])  # empty sequence keeps its state


def test_conv_decode_pool_padding_and_continuation():
    W, C, n, S, n_slots = 3, 8, 4, 2, 6
    x, w, b = _conv_inputs(n, 5 + S, C, W, 31, dtype=torch.bfloat16)
    # continuation: prefill of 5 tokens, then a decode step of S from its state
    yp, sp = oracle.conv(x[:, :5], w, b)
    pool = torch.zeros(n_slots, C, W - 1, dtype=torch.bfloat16)
    slots = torch.tensor([4, -1, 0, 2], dtype=torch.int32)
    for r in range(n):
        if slots[r] >= 0:
            pool[slots[r]] = sp[r]
    yd, new_pool = oracle.conv(x[:, 5:], w, b, state=pool, slot=slots)
    yfull, sfull = oracle.conv(x, w, b)
    for r in (0, 2, 3):
        assert torch.equal(yd[r], yfull[r, 5:]) and torch.equal(new_pool[slots[r]], sfull[r])
    assert torch.count_nonzero(yd[1]) == 0
    untouched = [1, 3, 5]
    assert torch.equal(new_pool[untouched], pool[untouched])
    # a slot named twice makes both requests padding
    yd2, pool2 = oracle.conv(x[:, 5:], w, b, state=pool, slot=torch.tensor([4, 4, 0, 2],
                                                                         dtype=torch.int32))
    assert torch.count_nonzero(yd2[:2]) == 0 and torch.equal(pool2[4], pool[4])
