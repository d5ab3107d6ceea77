"""C-ABI boundary checks that need no GPU: the library loads, exports every
symbol the header declares, and rejects invalid arguments before launching."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import linear_attention_ssm_gdp_gb300 as gdp
    if not os.path.exists(gdp.LIB_PATH):
        from linear_attention_ssm_gdp_gb300 import _build
        _build.build()
    return gdp


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(gdp_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_path(lib):
    names = _declared()
    for want in ("gdp_prefill_prepare", "gdp_decode_prepare", "gdp_chunk_fwd",
                 "gdp_chunk_fwd_workspace_size", "gdp_recurrent_update", "gdp_read_status"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(so, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings_and_version(lib):
    so = lib.load()
    for s in range(6):
        assert so.gdp_status_string(s)
    assert lib.gdp_version() >= 100


def _chunk(so, **kw):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, beta=1 << 20, g=None, h0=None, cu=None, N=2, B=2,
             T=64, H=2, HV=2, K=32, V=32, M=2, BT=64, scale=1.0, l2=0, dt=0, o=1 << 20,
             fs=None, ws=1 << 20, ws_bytes=1 << 40)
    a.update(kw)
    P = ctypes.c_void_p
    return so.gdp_chunk_fwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["beta"]), P(a["g"]),
                            P(a["h0"]), P(a["cu"]), a["N"], a["B"], a["T"], a["H"], a["HV"],
                            a["K"], a["V"], a["M"], a["BT"], a["scale"], a["l2"], a["dt"],
                            P(a["o"]), P(a["fs"]), P(a["ws"]), a["ws_bytes"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(H=3, HV=4), 1),            # HV % H != 0
    (dict(BT=48), 2),                # chunk size not built
    (dict(K=512), 2),                # K too large
    (dict(M=0), 1),
    (dict(B=0), 1),
    (dict(q=None), 1),               # null input
    (dict(o=None), 1),               # null output
    (dict(cu=1 << 20, B=2), 1),      # cu_seqlens needs B == 1
    (dict(N=3), 1),                  # without cu_seqlens N_seq must equal B
    (dict(ws_bytes=1000), 5),        # workspace too small
    (dict(ws=(1 << 20) + 8), 5),     # workspace misaligned
    (dict(dt=7), 2),                 # unknown dtype
    (dict(B=1, T=1 << 28, N=1, HV=8, H=2), 2),      # positions x heads past 32-bit coordinates
    (dict(cu=1 << 20, B=1, T=64, N=1 << 27, HV=64, H=2, K=256), 2),  # state rows past 32 bits
])
def test_chunk_fwd_rejects_before_launch(lib, kw, status):
    assert _chunk(lib.load(), **kw) == status


def test_workspace_size_query(lib):
    so = lib.load()
    ws = so.gdp_chunk_fwd_workspace_size
    assert ws(2, 4096, 2, 16, 16, 128, 128, 2, 64, 0) > 0
    assert ws(2, 4096, 2, 16, 16, 128, 128, 2, 48, 0) == 0
    assert ws(2, 4096, 2, 3, 16, 128, 128, 2, 64, 0) == 0
    assert ws(1, 8192, 4, 16, 16, 128, 128, 2, 64, 0) >= ws(1, 4096, 4, 16, 16, 128, 128, 2, 64, 0)
    off = lib.gdp_chunk_fwd_stage_offsets(1, 100, 1, 2, 2, 32, 32, 2, 64, torch.float32)
    assert off[5] in (0, 1)


def test_path_selection_and_fused_output(lib):
    """Which path a problem takes, and whether the chunk output is computed inside
    the scan (the tensor-core path for two Householder copies), as the stage-offset
    query reports it; host arithmetic only."""
    NONE = (1 << 64) - 1
    q = lambda *a: lib.gdp_chunk_fwd_stage_offsets(*a)
    bf, f32 = torch.bfloat16, torch.float32
    tc2 = q(2, 4096, 2, 16, 16, 128, 128, 2, 64, bf)    # bf16, K = 128, M = 2
    assert tc2[5] == 1 and tc2[7] == 1 and tc2[6] == 128
    assert tc2[3] == NONE and tc2[4] == NONE           # v_new and states never stored
    tc3 = q(1, 512, 1, 4, 4, 128, 128, 3, 64, bf)      # odd M: separate output kernel
    assert tc3[5] == 1 and tc3[7] == 0 and tc3[6] == 64
    gen = q(1, 128, 1, 2, 2, 32, 32, 2, 64, f32)       # fp32: generic path
    assert gen[5] == 0 and gen[7] == 0 and gen[3] != NONE and gen[4] != NONE


def _prep(fn, **kw):
    a = dict(x=1 << 20, x_sn=0, x_st=0, ba=1 << 20, ba_sn=0, ba_st=0, A=1 << 20, dtb=1 << 20,
             n=1, T=4, M=2, H=4, G=2, P=8, N=8, dt=0, q=1 << 20, k=1 << 20, v=1 << 20,
             beta=1 << 20, g=1 << 20)
    a.update(kw)
    D = a["M"] * a["H"] * a["P"] + a["M"] * a["G"] * a["N"] + a["G"] * a["N"]
    if a["x_st"] == 0:
        a["x_st"] = D
    if a["ba_st"] == 0:
        a["ba_st"] = a["M"] * a["H"] + a["H"]
    P = ctypes.c_void_p
    return fn(P(a["x"]), a["x_sn"], a["x_st"], P(a["ba"]), a["ba_sn"], a["ba_st"], P(a["A"]),
              P(a["dtb"]), a["n"], a["T"], a["M"], a["H"], a["G"], a["P"], a["N"], a["dt"],
              P(a["q"]), P(a["k"]), P(a["v"]), P(a["beta"]), P(a["g"]), None)


@pytest.mark.parametrize("kw,status", [
    (dict(H=4, G=3), 1),      # H % G != 0
    (dict(x=None), 1),
    (dict(g=None), 1),
    (dict(x_st=10), 1),       # row stride shorter than a row
    (dict(M=0), 1),
    (dict(dt=9), 2),
])
def test_prepare_rejects_before_launch(lib, kw, status):
    so = lib.load()
    assert _prep(so.gdp_prefill_prepare, **kw) == status
    assert _prep(so.gdp_decode_prepare, **kw) == status


def test_decode_prepare_draft_limit(lib):
    so = lib.load()
    assert _prep(so.gdp_decode_prepare, T=17) == 1
    assert _prep(so.gdp_decode_prepare, T=0) == 1


def test_empty_problems_are_no_ops(lib):
    so = lib.load()
    assert _prep(so.gdp_prefill_prepare, T=0, x=None, q=None) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(K=48), 2), (dict(V=12), 2), (dict(H=3, HV=4), 1), (dict(state=None), 1),
    (dict(state=(1 << 20) + 4), 1),
])
def test_recurrent_rejects_before_launch(lib, kw, status):
    a = dict(n=2, L=4, H=2, HV=2, K=32, V=32, state=1 << 20)
    a.update(kw)
    P = ctypes.c_void_p
    so = lib.load()
    st = so.gdp_recurrent_update(P(1 << 20), P(1 << 20), P(1 << 20), P(1 << 20), P(1 << 20),
                                 P(a["state"]), a["n"], a["L"], a["H"], a["HV"], a["K"],
                                 a["V"], 1.0, 0, 0, P(1 << 20), None)
    assert st == status


@pytest.mark.parametrize("kw,status", [
    (dict(K=48), 2), (dict(slot=None), 1), (dict(n_slots=-1), 1), (dict(pool=None), 1),
    (dict(pool=(1 << 20) + 4), 1), (dict(H=3, HV=4), 1),
])
def test_recurrent_slots_rejects_before_launch(lib, kw, status):
    a = dict(n=2, L=4, H=2, HV=2, K=32, V=32, pool=1 << 20, slot=1 << 20, n_slots=4)
    a.update(kw)
    P = ctypes.c_void_p
    so = lib.load()
    st = so.gdp_recurrent_update_slots(P(1 << 20), P(1 << 20), P(1 << 20), P(1 << 20),
                                       P(1 << 20), P(a["pool"]), P(a["slot"]), a["n_slots"],
                                       a["n"], a["L"], a["H"], a["HV"], a["K"], a["V"], 1.0, 0,
                                       0, P(1 << 20), None, None)
    assert st == status
