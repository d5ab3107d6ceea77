"""gdp_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate
device memory (fixed memory budgets, allocator callbacks, loops that must not
reach cudaMalloc). It uses the library's own fixed device scratch array instead
of a caller workspace; its results must match gdp_chunk_fwd's.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

from _util import chunk_case, rel_err, to

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc_raw(gdp, q, k, v, beta, g, o, fs, M, BT, l2):
    """Call the C entry point directly with preallocated outputs."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return gdp.load().gdp_chunk_fwd_noalloc(P(q), P(k), P(v), P(beta), P(g), None, None, B, B, T,
                                            H, HV, K, V, M, BT, float(K ** -0.5), int(l2), 0,
                                            P(o), P(fs), stream)


@pytest.mark.parametrize("T,K,V,M", [(300, 128, 128, 2), (150, 64, 32, 3)])
def test_noalloc_matches_workspace_entry_point_twice(gdp, T, K, V, M):
    B, H, HV, BT = 1, 2, 2, 64
    q, k, v, beta, g = to(DEV, *chunk_case(B, T, H, HV, K, V, M, seed=31))
    ref_o, ref_fs = gdp.gdp_chunk_fwd(q, k, v, beta, g, chunk_size=BT, num_householder=M,
                                      use_qk_l2norm=True)
    o = torch.empty_like(ref_o)
    fs = torch.empty_like(ref_fs)
    for _ in range(2):  # two calls in a row share (and reuse) the scratch array
        o.fill_(float("nan"))
        fs.fill_(float("nan"))
        assert _noalloc_raw(gdp, q, k, v, beta, g, o, fs, M, BT, True) == 0
        torch.cuda.synchronize()
        assert rel_err(o, ref_o) <= 2e-3
        assert rel_err(fs, ref_fs) <= 2e-3


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
