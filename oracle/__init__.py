"""CPU oracle for the Gated Delta Product (GDP) forward pass.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. It shares no code with the
CUDA library (``linear_attention_ssm_gdp_gb300``) and never imports it.

Two independent restatements of what the pages compute:

* ``gdp_oracle.c`` (compiled with gcc, loaded with ctypes): the fp32 prepare map
  (prepare page: module overview, ``softplus``, ``gdp_prepare_kernel``,
  ``gdp_decode_prepare``, ``gdp_prefill_prepare``) and the fp64 token walk of
  the gated delta rule over the Householder-expanded stream.
* ``chunked_stream`` below: the chunked WY form in fp64 numpy (wy_fast page:
  "Recompute the w and u factors of the WY representation", A from
  ``solve_tril``; chunk_o page: state at chunk boundaries from ``chunk_h`` plus
  causal within-chunk attention summed over the copies). It exposes every
  intermediate (L, A, w, u, v_new, h) for stage-by-stage checks.

Pins that tie these to the pages and the mathematics live in
``tests/test_oracle_pins.py``. Functions whose parity is pinned only by
invariants (not by a value the pages print) are listed there; the layout
reading of the prepare split (copy-major value/key blocks, contiguous
group-to-head map) has no worked example on the pages: parity unpinned
beyond the decode/prefill cross-checks and the bijection checks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdp_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DT = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}


def build(force: bool = False) -> str:
    """Compile gdp_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_gate_map.argtypes = [P, I64, P, I64, I, P, P, P, P]
            lib.oracle_prepare.argtypes = [P, I64, I64, P, I64, I64, P, P] + [I] * 9 + [P] * 5
            lib.oracle_gdp_walk.argtypes = [P] * 7 + [I] * 8 + [D, I, I, P, P]
            lib.oracle_gdp_recurrent.argtypes = [P] * 6 + [I] * 6 + [D, I, I, P]
            lib.oracle_conv.argtypes = ([P, I64, I64, P, P, I, P, P, P, I, P, I] + [I] * 5 + [P])
            lib.oracle_max_threads.argtypes = []
            for f in ("oracle_gate_map", "oracle_prepare", "oracle_gdp_walk", "oracle_conv",
                      "oracle_gdp_recurrent", "oracle_max_threads"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


# --------------------------------------------------------------------------------------
# prepare (fp32 map)
# --------------------------------------------------------------------------------------

def gate_map(b: torch.Tensor, a: torch.Tensor, A_log: torch.Tensor, dt_bias: torch.Tensor):
    """beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias), fp32 (prepare page).

    ``b`` [..., H] and ``a`` [..., H] are read as fp32; returns (beta, g) fp32 with
    their shapes.
    """
    H = b.shape[-1]
    bf = b.detach().to(torch.float32).contiguous().cpu()
    af = a.detach().to(torch.float32).contiguous().cpu()
    Al = A_log.detach().to(torch.float32).contiguous().cpu()
    db = dt_bias.detach().to(torch.float32).contiguous().cpu()
    beta = torch.empty_like(bf)
    g = torch.empty_like(af)
    rc = _load().oracle_gate_map(_ptr(bf), bf.numel() // H, _ptr(af), af.numel() // H, H,
                                 _ptr(Al), _ptr(db), _ptr(beta), _ptr(g))
    if rc:
        raise ValueError("oracle_gate_map: bad arguments")
    return beta, g


def prepare(x: torch.Tensor, ba: torch.Tensor, A_log: torch.Tensor, dt_bias: torch.Tensor,
            M: int, H: int, G: int, P: int, N: int, decode: bool):
    """The prepare map on CPU. Returns (q, k, v, beta, g) with the pages' layouts."""
    assert x.dtype == ba.dtype and x.dtype in _DT
    n, T, D = x.shape
    assert D == M * H * P + M * G * N + G * N and ba.shape == (n, T, M * H + H)
    assert x.stride(-1) == 1 and ba.stride(-1) == 1
    x = x.cpu()
    ba = ba.cpu()
    Al = A_log.detach().to(torch.float32).contiguous().cpu()
    db = dt_bias.detach().to(torch.float32).contiguous().cpu()
    L = T * M
    q = torch.empty((n, L if decode else T, H, N), dtype=x.dtype)
    k = torch.empty((n, L, H, N), dtype=x.dtype)
    v = torch.empty((n, L, H, P), dtype=x.dtype)
    beta = torch.empty((n, L, H), dtype=torch.float32)
    g = torch.empty((n, L if decode else T, H), dtype=torch.float32)
    rc = _load().oracle_prepare(
        ctypes.c_void_p(x.data_ptr()), x.stride(0), x.stride(1),
        ctypes.c_void_p(ba.data_ptr()), ba.stride(0), ba.stride(1), _ptr(Al), _ptr(db),
        n, T, M, H, G, P, N, _DT[x.dtype], 1 if decode else 0,
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g))
    if rc:
        raise ValueError("oracle_prepare: bad arguments")
    return q, k, v, beta, g


def conv(xp: torch.Tensor, w: torch.Tensor, b, state=None, cu_seqlens=None, slot=None):
    """The short causal conv + SiLU before prepare (depthwise, width W = w.shape[1]),
    fp32 one operation at a time, output in xp's dtype (bf16 or fp32).

    Prefill (slot None): state [N, C, W-1] or None; returns (x [n,T,C], new_state
    [N, C, W-1]). Decode (slot int32 [n]): state is the pool [n_slots, C, W-1];
    returns (x, new_pool) with padding requests (slot -1, out of range, repeated)
    zero and their entries untouched.
    """
    assert xp.dtype in (torch.bfloat16, torch.float32) and xp.stride(-1) == 1
    n, T, C = xp.shape
    W = w.shape[1]
    xc = xp.cpu()
    wf = w.detach().to(torch.float32).contiguous().cpu()
    bf = None if b is None else b.detach().to(torch.float32).contiguous().cpu()
    out = torch.zeros((n, T, C), dtype=xp.dtype)
    decode = slot is not None
    if decode:
        pool = state.detach().cpu().contiguous().clone()
        sl = slot.detach().cpu().to(torch.int32).contiguous()
        rc = _load().oracle_conv(ctypes.c_void_p(xc.data_ptr()), xc.stride(0), xc.stride(1),
                                 _ptr(wf), _ptr(bf), W, _ptr(pool), _ptr(pool), None, n,
                                 _ptr(sl), pool.shape[0], n, T, C, _DT[xp.dtype], 1, _ptr(out))
        if rc:
            raise ValueError("oracle_conv: bad arguments")
        return out, pool
    cu = None if cu_seqlens is None else cu_seqlens.detach().cpu().to(torch.int32).contiguous()
    N = n if cu is None else cu.numel() - 1
    st_in = None if state is None else state.detach().cpu().contiguous()
    st_out = torch.zeros((N, C, max(W - 1, 0)), dtype=xp.dtype)
    rc = _load().oracle_conv(ctypes.c_void_p(xc.data_ptr()), xc.stride(0), xc.stride(1),
                             _ptr(wf), _ptr(bf), W, _ptr(st_in), _ptr(st_out), _ptr(cu), N, None,
                             0, n, T, C, _DT[xp.dtype], 0, _ptr(out))
    if rc:
        raise ValueError("oracle_conv: bad arguments")
    return out, st_out


# --------------------------------------------------------------------------------------
# fp64 token walk (the recurrence itself)
# --------------------------------------------------------------------------------------

def _d(t):
    return None if t is None else t.detach().cpu().to(torch.float64).contiguous()


def walk(q, k, v, beta, g, M: int, scale: float, cu_seqlens=None, h0=None,
         l2norm: bool = False, nthreads: int = 0):
    """fp64 gated-delta walk over the expanded stream.

    q [B,T,H,K], k [B,T*M,H,K], v [B,T*M,HV,V], beta [B,T*M,HV],
    g [B,T,HV] (natural-log decay per token, or None), h0 [S,HV,K,V] or None,
    cu_seqlens [N+1] int (B must be 1) or None.
    Returns (o [B,T,HV,V], final_state [S,HV,K,V]) as float64 tensors.
    """
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    assert k.shape == (B, T * M, H, K) and v.shape[:2] == (B, T * M)
    qd, kd, vd, bd, gd, hd = _d(q), _d(k), _d(v), _d(beta), _d(g), _d(h0)
    cu = None
    nseq = B
    if cu_seqlens is not None:
        cu = cu_seqlens.detach().cpu().to(torch.int32).contiguous()
        nseq = cu.numel() - 1
    o = torch.zeros((B, T, HV, V), dtype=torch.float64)
    hT = torch.zeros((nseq, HV, K, V), dtype=torch.float64)
    rc = _load().oracle_gdp_walk(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(bd), _ptr(gd), _ptr(hd),
                                 _ptr(cu), nseq, B, T, H, HV, K, V, M, float(scale),
                                 1 if l2norm else 0, int(nthreads), _ptr(o), _ptr(hT))
    if rc:
        raise ValueError("oracle_gdp_walk: bad arguments")
    return o, hT


def recurrent(q, k, v, beta, g, state, scale: float, l2norm: bool = False, nthreads: int = 0):
    """fp64 per-step walk (decode): inputs [n,L,...] with q/g already placed on copies.

    Returns (o [n,L,HV,V], new_state [n,HV,K,V]) as float64 tensors.
    """
    n, L, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    st = _d(state).clone()
    o = torch.zeros((n, L, HV, V), dtype=torch.float64)
    # keep every converted input alive for the duration of the C call
    qd, kd, vd, bd, gd = _d(q), _d(k), _d(v), _d(beta), _d(g)
    rc = _load().oracle_gdp_recurrent(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(bd), _ptr(gd), _ptr(st),
                                      n, L, H, HV, K, V, float(scale), 1 if l2norm else 0,
                                      int(nthreads), _ptr(o))
    if rc:
        raise ValueError("oracle_gdp_recurrent: bad arguments")
    return o, st


# --------------------------------------------------------------------------------------
# fp64 chunked WY restatement (one sequence, one value head)
# --------------------------------------------------------------------------------------

def _l2(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + 1e-6)


def chunked_stream(q, k, v, beta, g, M: int, BT: int, scale: float, h0=None,
                   l2norm: bool = False):
    """Chunked form of the same recurrence for one (sequence, value head), fp64.

    q [T,K] (token stream), k [T*M,K], v [T*M,V], beta [T*M], g [T] natural-log
    decay per token (or None). WY stages run on chunks of BT expanded positions;
    the output runs on chunks of BT tokens and reads the state at expanded
    position c*BT*M, which is the start of expanded chunk c*M.

    Per expanded chunk with start state h (K x V) and Gam the inclusive cumsum
    of the per-position decay (g_t on a token's first copy, 0 on the others):
        L[p,i] = beta_p exp(Gam_p - Gam_i) k_p.k_i  (i < p), else 0
        A      = (I + L)^-1                      (solve_tril)
        w      = A (beta exp(Gam) k),  u = A (beta v)   (recompute_w_u)
        v_new  = u - w h                          (corrected values)
        h'     = exp(Gam_last) h + (k exp(Gam_last - Gam))^T v_new   (chunk_h)
    Per token chunk with start state hc and Gt the token-stream cumsum:
        o_t = scale (exp(Gt_t) q_t.hc + sum_{s<=t} sum_j exp(Gt_t - Gt_s)(q_t.k_{s,j}) v_new_{s,j})
    Returns a dict of numpy arrays: L, A (per chunk), w, u, v_new (per position),
    h_chunks (state at each expanded chunk start), o [T,V], h_final [K,V].
    """
    from scipy.linalg import solve_triangular

    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, K = q.shape
    Le, V = v.shape
    assert Le == T * M and k.shape == (Le, K) and beta.shape == (Le,)
    if l2norm:
        q = _l2(q)
        k = _l2(k)
    ge = np.zeros(Le)
    if g is not None:
        ge[0::M] = np.asarray(g, dtype=np.float64)
    h = np.zeros((K, V)) if h0 is None else np.array(h0, dtype=np.float64)
    Ls, As, hs = [], [], []
    w = np.zeros((Le, K))
    u = np.zeros((Le, V))
    v_new = np.zeros((Le, V))
    for e0 in range(0, Le, BT):
        e1 = min(e0 + BT, Le)
        n = e1 - e0
        kc, vc, bc = k[e0:e1], v[e0:e1], beta[e0:e1]
        gam = np.cumsum(ge[e0:e1])
        Lm = np.zeros((n, n))
        for p in range(n):
            for i in range(p):
                Lm[p, i] = bc[p] * np.exp(gam[p] - gam[i]) * (kc[p] @ kc[i])
        A = solve_triangular(np.eye(n) + Lm, np.eye(n), lower=True, unit_diagonal=True)
        wc = A @ (bc[:, None] * np.exp(gam)[:, None] * kc)
        uc = A @ (bc[:, None] * vc)
        hs.append(h.copy())
        vn = uc - wc @ h
        h = np.exp(gam[-1]) * h + (kc * np.exp(gam[-1] - gam)[:, None]).T @ vn
        Ls.append(Lm)
        As.append(A)
        w[e0:e1], u[e0:e1], v_new[e0:e1] = wc, uc, vn
    h_final = h
    if Le == 0:
        hs.append(h.copy())
    o = np.zeros((T, V))
    gt = np.zeros(T) if g is None else np.asarray(g, dtype=np.float64)
    for t0 in range(0, T, BT):
        t1 = min(t0 + BT, T)
        hc = hs[(t0 * M) // BT]
        Gt = np.cumsum(gt[t0:t1])
        for t in range(t0, t1):
            acc = np.exp(Gt[t - t0]) * (q[t] @ hc)
            for s in range(t0, t + 1):
                dec = np.exp(Gt[t - t0] - Gt[s - t0])
                for j in range(M):
                    acc = acc + dec * (q[t] @ k[s * M + j]) * v_new[s * M + j]
            o[t] = scale * acc
    return {"L": Ls, "A": As, "w": w, "u": u, "v_new": v_new, "h_chunks": hs, "o": o,
            "h_final": h_final}
