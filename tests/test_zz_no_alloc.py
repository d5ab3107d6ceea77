"""gdp_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate
device memory (fixed memory budgets, allocator callbacks, loops that must not
reach cudaMalloc). It uses the library's own fixed device scratch array instead
of a caller workspace and runs the same deterministic kernels, so its results
must equal gdp_chunk_fwd's bit for bit.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

import synth_inputs as si
from _util import chunk_case, to

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc_raw(gdp, q, k, v, beta, g, o, fs, M, BT, l2, h0=None, cu=None):
    """Call the C entry point directly with preallocated outputs."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = B if cu is None else cu.numel() - 1
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return gdp.load().gdp_chunk_fwd_noalloc(P(q), P(k), P(v), P(beta), P(g), P(h0), P(cu), N, B,
                                            T, H, HV, K, V, M, BT, float(K ** -0.5), int(l2), 0,
                                            P(o), P(fs), stream)


def _twice_equal(gdp, q, k, v, beta, g, M, h0=None, cu=None):
    BT = 64
    ref_o, ref_fs = gdp.gdp_chunk_fwd(q, k, v, beta, g, cu_seqlens=cu, chunk_size=BT,
                                      num_householder=M, initial_state=h0, use_qk_l2norm=True)
    o = torch.empty_like(ref_o)
    fs = torch.empty_like(ref_fs)
    n = ref_o.shape[1] if cu is None else int(cu[-1])
    for _ in range(2):  # two calls in a row share (and reuse) the scratch array
        o.fill_(float("nan"))
        fs.fill_(float("nan"))
        assert _noalloc_raw(gdp, q, k, v, beta, g, o, fs, M, BT, True, h0=h0, cu=cu) == 0
        torch.cuda.synchronize()
        assert torch.equal(o[:, :n], ref_o[:, :n])
        assert torch.equal(fs, ref_fs)


@pytest.mark.parametrize("T,K,V,M", [(300, 128, 128, 2), (150, 64, 32, 3), (260, 128, 128, 3)])
def test_noalloc_matches_workspace_entry_point_twice(gdp, T, K, V, M):
    q, k, v, beta, g = to(DEV, *chunk_case(1, T, 2, 2, K, V, M, seed=31))
    _twice_equal(gdp, q, k, v, beta, g, M)


def test_noalloc_varlen_with_initial_state_twice(gdp):
    lens = [1, 63, 130, 0, 200]
    cu = si.cu_seqlens_of(lens)
    T = int(cu[-1]) + 3
    q, k, v, beta, g = chunk_case(1, T, 2, 2, 128, 128, 2, seed=32)
    h0 = torch.randn(len(lens), 2, 128, 128, generator=torch.Generator().manual_seed(5))
    _twice_equal(gdp, *to(DEV, q, k, v, beta, g), 2, h0=h0.to(DEV), cu=cu.to(DEV))


def test_noalloc_gva_twice(gdp):
    q, k, v, beta, g = to(DEV, *chunk_case(2, 140, 2, 8, 128, 64, 2, seed=33))
    _twice_equal(gdp, q, k, v, beta, g, 2)


def test_noalloc_bad_seqlens_after_a_valid_call(gdp):
    """A valid call fills the scratch with tables of large sequences; a following
    call with a bad offset list on a smaller problem must not reuse them: o keeps
    its canaries and the final state is the initial state."""
    M, K, V = 2, 128, 128
    q, k, v, beta, g = to(DEV, *chunk_case(1, 600, 2, 2, K, V, M, seed=34))
    o = torch.empty(1, 600, 2, V, device=DEV)
    fs = torch.empty(1, 2, K, V, device=DEV)
    assert _noalloc_raw(gdp, q, k, v, beta, g, o, fs, M, 64, True) == 0
    T = 100
    q2, k2, v2, beta2, g2 = to(DEV, *chunk_case(1, T, 2, 2, K, V, M, seed=35))
    cu = torch.tensor([0, 60, 30], dtype=torch.int32, device=DEV)  # decreasing
    h0 = torch.randn(2, 2, K, V, generator=torch.Generator().manual_seed(6)).to(DEV)
    o2 = torch.full((1, T, 2, V), float("nan"), device=DEV)
    fs2 = torch.full((2, 2, K, V), float("nan"), device=DEV)
    assert _noalloc_raw(gdp, q2, k2, v2, beta2, g2, o2, fs2, M, 64, True, h0=h0, cu=cu) == 0
    torch.cuda.synchronize()
    assert torch.isnan(o2).all()
    assert torch.equal(fs2, h0)


def test_noalloc_rejects_problems_larger_than_its_scratch(gdp):
    B, T, H, HV, K, V, M = 1, 8192, 16, 16, 128, 128, 2
    need = gdp.gdp_chunk_fwd_workspace_size(B, T, B, H, HV, K, V, M, 64, torch.bfloat16)
    assert need > 32 << 20
    q = torch.zeros(B, T, H, K, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(B, T * M, H, K, dtype=torch.bfloat16, device=DEV)
    v = torch.zeros(B, T * M, HV, V, dtype=torch.bfloat16, device=DEV)
    beta = torch.zeros(B, T * M, HV, device=DEV)
    o = torch.empty(B, T, HV, V, device=DEV)
    fs = torch.empty(B, HV, K, V, device=DEV)
    assert _noalloc_raw(gdp, q, k, v, beta, None, o, fs, M, 64, False) == 5  # GDP_ERR_WORKSPACE
