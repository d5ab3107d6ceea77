"""Host-side checks of the bench's eager prepare comparator (no GPU).

The bench times the fused prepare kernel against an eager PyTorch composition
of the same step and checks the two agree bit for bit on the GPU. Here the
same composition runs on CPU tensors against the oracle's prepare map: the
copies (split, group expansion, copy folding, +0 placements) must be
bit-identical, and the gates within a few ulp (torch's CPU exp/log1p are not
the host libm the oracle calls).
"""
import pytest
import torch

import bench
import oracle
import synth_inputs as si
from _util import GATE_ULP


def _ulp(a, b):
    ai = a.contiguous().view(torch.int32).to(torch.int64)
    bi = b.contiguous().view(torch.int32).to(torch.int64)
    ai = torch.where(ai < 0, -(ai & 0x7FFFFFFF), ai)
    bi = torch.where(bi < 0, -(bi & 0x7FFFFFFF), bi)
    return (ai - bi).abs()


@pytest.mark.parametrize("decode", [False, True])
@pytest.mark.parametrize("n,T,M,H,G,P,N", [(2, 7, 2, 4, 2, 16, 8), (1, 5, 3, 6, 3, 8, 16)])
def test_eager_prepare_matches_the_oracle(decode, n, T, M, H, G, P, N):
    d = si.prepare_inputs(n, T, M, H, G, P, N, seed=n + T + M)
    got = bench.eager_prepare(d["x"], d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N, decode)
    ref = oracle.prepare(d["x"], d["ba"], d["A_log"], d["dt_bias"], M, H, G, P, N, decode=decode)
    for name, a, b in zip(("q", "k", "v"), got[:3], ref[:3]):
        assert a.dtype == b.dtype and tuple(a.shape) == tuple(b.shape), name
        assert torch.equal(a.contiguous(), b), name
    for name, a, b in zip(("beta", "g"), got[3:], ref[3:]):
        assert a.dtype == torch.float32 and tuple(a.shape) == tuple(b.shape), name
        assert int(_ulp(a, b).max()) <= GATE_ULP[name], name
