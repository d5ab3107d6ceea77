"""Gated Delta Product (GDP) forward pass for NVIDIA GB300 (sm_103a).

Thin ctypes binding over ``libgdp.so`` (C ABI in ``include/gdp.h``). The
Python functions carry the C names and only marshal arguments: they allocate
outputs and workspace with PyTorch (device memory and streams are all PyTorch
is used for), pass raw device pointers and the current CUDA stream, and raise
on a non-OK status. Every step of the computation runs in the library's CUDA
kernels; there is no CPU path. ``load()`` raises if the library has not been
built (``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "load", "GDPError", "gdp_prefill_prepare", "gdp_decode_prepare", "gdp_chunk_fwd",
    "gdp_chunk_fwd_workspace_size", "gdp_chunk_fwd_stage_offsets", "gdp_recurrent_update",
    "gdp_read_status", "gdp_version", "gdp_set_stage_events", "gdp_chunk_fwd_noalloc",
    "gdp_recurrent_update_slots", "gdp_debug_wait_fault", "gdp_prefill_conv_prepare",
    "gdp_decode_conv_prepare",
    "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgdp.so")

GDP_OK, GDP_ERR_INVALID_ARG, GDP_ERR_UNSUPPORTED, GDP_ERR_CUDA = 0, 1, 2, 3
GDP_ERR_DEVICE_TIMEOUT, GDP_ERR_WORKSPACE = 4, 5
_DTYPE = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}

_lock = threading.Lock()
_lib = None


class GDPError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libgdp.so once; raises if it is missing (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() first")
            lib = ctypes.CDLL(LIB_PATH)
            P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
            prep = [P, I64, I64, P, I64, I64, P, P] + [I] * 7 + [I] + [P] * 5 + [P]
            lib.gdp_prefill_prepare.argtypes = prep
            lib.gdp_decode_prepare.argtypes = prep
            lib.gdp_prefill_conv_prepare.argtypes = ([P, I64, I64, P, P, I, P, P, P, I, P, I64, I64,
                                                      P, P] + [I] * 8 + [P] * 6)
            lib.gdp_decode_conv_prepare.argtypes = ([P, I64, I64, P, P, I, P, P, I, P, I64, I64, P,
                                                     P] + [I] * 8 + [P] * 7)
            lib.gdp_chunk_fwd_workspace_size.argtypes = [I] * 9 + [I]
            lib.gdp_chunk_fwd_workspace_size.restype = SZ
            lib.gdp_chunk_fwd_stage_offsets.argtypes = [I] * 9 + [I, P]
            lib.gdp_chunk_fwd.argtypes = ([P] * 7 + [I] * 9 + [F, I, I] + [P, P, P, SZ, P])
            lib.gdp_recurrent_update.argtypes = [P] * 6 + [I] * 6 + [F, I, I, P, P]
            lib.gdp_recurrent_update_slots.argtypes = ([P] * 7 + [I] * 7 + [F, I, I, P, P, P])
            lib.gdp_chunk_fwd_noalloc.argtypes = [P] * 7 + [I] * 9 + [F, I, I] + [P, P, P]
            lib.gdp_chunk_fwd_noalloc.restype = I
            lib.gdp_read_status.argtypes = [P, P]
            lib.gdp_debug_wait_fault.argtypes = [I, ctypes.c_double]
            lib.gdp_debug_wait_fault.restype = I
            lib.gdp_set_stage_events.argtypes = [P, I]
            lib.gdp_set_stage_events.restype = I
            lib.gdp_status_string.argtypes = [I]
            lib.gdp_status_string.restype = ctypes.c_char_p
            lib.gdp_version.argtypes = []
            for f in ("gdp_prefill_prepare", "gdp_decode_prepare", "gdp_chunk_fwd",
                      "gdp_prefill_conv_prepare", "gdp_decode_conv_prepare",
                      "gdp_recurrent_update", "gdp_recurrent_update_slots", "gdp_read_status",
                      "gdp_chunk_fwd_stage_offsets",
                      "gdp_version"):
                getattr(lib, f).restype = I
            _lib = lib
    return _lib


def _check(fn: str, status: int):
    if status != GDP_OK:
        raise GDPError(fn, status, load().gdp_status_string(status).decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libgdp works on CUDA tensors only")


def gdp_version() -> int:
    return int(load().gdp_version())


# ----------------------------------------------------------------------------------
# prepare
# ----------------------------------------------------------------------------------

def _prepare(name, x, ba, A_log, dt_bias, M, H, G, P, N, decode, out=None):
    _need_cuda(x, ba, A_log, dt_bias)
    if x.dtype not in _DTYPE or ba.dtype != x.dtype:
        raise ValueError("x and ba must share a dtype in {bf16, fp16, fp32}")
    if x.dim() != 3 or ba.dim() != 3 or x.stride(-1) != 1 or ba.stride(-1) != 1:
        raise ValueError("x and ba must be [n, T, D] with a contiguous last dimension")
    n, T, D = x.shape
    if D != M * H * P + M * G * N + G * N or tuple(ba.shape) != (n, T, M * H + H):
        raise ValueError("x/ba last dimensions do not match M, H, G, P, N")
    A_log = A_log.to(torch.float32).contiguous()
    dt_bias = dt_bias.to(torch.float32).contiguous()
    L = T * M
    dev = x.device
    if out is None:
        q = torch.empty((n, L if decode else T, H, N), dtype=x.dtype, device=dev)
        k = torch.empty((n, L, H, N), dtype=x.dtype, device=dev)
        v = torch.empty((n, L, H, P), dtype=x.dtype, device=dev)
        beta = torch.empty((n, L, H), dtype=torch.float32, device=dev)
        g = torch.empty((n, L if decode else T, H), dtype=torch.float32, device=dev)
    else:
        q, k, v, beta, g = out
    fn = getattr(load(), name)
    st = fn(_p(x), x.stride(0), x.stride(1), _p(ba), ba.stride(0), ba.stride(1), _p(A_log),
            _p(dt_bias), n, T, M, H, G, P, N, _DTYPE[x.dtype], _p(q), _p(k), _p(v), _p(beta),
            _p(g), _stream(dev))
    _check(name, st)
    return q, k, v, beta, g


def gdp_prefill_prepare(x, ba, A_log, dt_bias, num_householder: int, num_heads: int,
                        num_groups: int, head_dim: int, state_dim: int, out=None):
    """Split/expand/gate a prefill step: returns (q [n,T,H,N], k [n,T*M,H,N],
    v [n,T*M,H,P], beta [n,T*M,H] fp32, g [n,T,H] fp32)."""
    return _prepare("gdp_prefill_prepare", x, ba, A_log, dt_bias, num_householder, num_heads,
                    num_groups, head_dim, state_dim, False, out)


def gdp_decode_prepare(x, ba, A_log, dt_bias, num_householder: int, num_heads: int,
                       num_groups: int, head_dim: int, state_dim: int, out=None):
    """Split/expand/gate a decode step (q on the last copy, g on the first):
    returns (q, k [n,S*M,H,N], v [n,S*M,H,P], beta, g [n,S*M,H] fp32)."""
    return _prepare("gdp_decode_prepare", x, ba, A_log, dt_bias, num_householder, num_heads,
                    num_groups, head_dim, state_dim, True, out)


# ----------------------------------------------------------------------------------
# chunked forward
# ----------------------------------------------------------------------------------

def gdp_chunk_fwd_workspace_size(B, T, N_seq, H, HV, K, V, M, chunk_size, dtype) -> int:
    return int(load().gdp_chunk_fwd_workspace_size(B, T, N_seq, H, HV, K, V, M, chunk_size,
                                                   _DTYPE[dtype]))


def gdp_chunk_fwd_stage_offsets(B, T, N_seq, H, HV, K, V, M, chunk_size, dtype):
    out = (ctypes.c_size_t * 8)()
    _check("gdp_chunk_fwd_stage_offsets",
           load().gdp_chunk_fwd_stage_offsets(B, T, N_seq, H, HV, K, V, M, chunk_size,
                                              _DTYPE[dtype], out))
    return list(out)


def gdp_chunk_fwd(q, k, v, beta, g=None, cu_seqlens=None, chunk_size: int = 64,
                  num_householder: int = 1, scale: float | None = None, initial_state=None,
                  use_qk_l2norm: bool = False, output_final_state: bool = True, workspace=None,
                  out=None):
    """Chunked GDP forward: returns (o [B,T,HV,V] fp32, final_state [N,HV,K,V] fp32 or None).

    q [B,T,H,K], k [B,T*M,H,K], v [B,T*M,HV,V] (bf16/fp16/fp32), beta [B,T*M,HV]
    fp32, g [B,T,HV] fp32 natural-log decay per token (None: ungated),
    cu_seqlens [N+1] int32 on the device (B must be 1), initial_state [N,HV,K,V]
    fp32. ``scale`` defaults to K**-0.5. ``workspace``: optional uint8 device
    tensor of at least gdp_chunk_fwd_workspace_size() bytes.
    """
    _need_cuda(q, k, v, beta, g, cu_seqlens, initial_state)
    M = int(num_householder)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if tuple(k.shape) != (B, T * M, H, K) or tuple(v.shape[:2]) != (B, T * M):
        raise ValueError("k/v must be [B, T*M, ...]")
    if tuple(beta.shape) != (B, T * M, HV) or (g is not None and tuple(g.shape) != (B, T, HV)):
        raise ValueError("beta must be [B,T*M,HV] and g [B,T,HV]")
    for t in (q, k, v, beta, g, initial_state):
        if t is not None and not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    if beta.dtype != torch.float32 or (g is not None and g.dtype != torch.float32):
        raise ValueError("beta and g must be fp32")
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in _DTYPE:
        raise ValueError("q, k, v must share a dtype in {bf16, fp16, fp32}")
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    if initial_state is not None and (tuple(initial_state.shape) != (N, HV, K, V)
                                      or initial_state.dtype != torch.float32):
        raise ValueError("initial_state must be fp32 [N, HV, K, V]")
    if scale is None:
        scale = K ** -0.5
    dev = q.device
    need = gdp_chunk_fwd_workspace_size(B, T, N, H, HV, K, V, M, chunk_size, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    if out is None:
        o = torch.empty((B, T, HV, V), dtype=torch.float32, device=dev)
        fs = (torch.empty((N, HV, K, V), dtype=torch.float32, device=dev)
              if output_final_state else None)
    else:
        o, fs = out
    st = load().gdp_chunk_fwd(_p(q), _p(k), _p(v), _p(beta), _p(g), _p(initial_state),
                              _p(cu_seqlens), N, B, T, H, HV, K, V, M, int(chunk_size),
                              float(scale), 1 if use_qk_l2norm else 0, _DTYPE[q.dtype], _p(o),
                              _p(fs), _p(workspace), workspace.numel(), _stream(dev))
    _check("gdp_chunk_fwd", st)
    return o, fs


GDP_STAGE_EVENTS = 5


def gdp_set_stage_events(events):
    """Profiling hook: record ``events`` (5 torch.cuda.Event, or None to switch
    off) at the stage boundaries of every later gdp_chunk_fwd call: entry, after
    the chunk tables, after the WY stage, after the state recurrence, after the
    output stage."""
    lib = load()
    if events is None:
        _check("gdp_set_stage_events", lib.gdp_set_stage_events(None, 0))
        return
    for e in events:
        e.record()  # forces the lazy creation of the CUDA event
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check("gdp_set_stage_events", lib.gdp_set_stage_events(arr, len(events)))


def gdp_chunk_fwd_noalloc(q, k, v, beta, g=None, cu_seqlens=None, chunk_size: int = 64,
                          num_householder: int = 1, scale: float | None = None,
                          initial_state=None, use_qk_l2norm: bool = False,
                          output_final_state: bool = True, out=None):
    """gdp_chunk_fwd without a caller workspace: the library's fixed 32 MiB device
    scratch array is used instead, for callers that cannot allocate device memory
    (fixed memory budgets, allocator callbacks, loops that must not reach
    cudaMalloc). Outputs are still allocated here unless ``out`` is given; pass
    ``out`` to allocate nothing. Larger problems raise GDPError (workspace).
    Calls sharing the array must not overlap on the GPU."""
    _need_cuda(q, k, v, beta, g, cu_seqlens, initial_state)
    M = int(num_householder)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    if out is None:
        o = torch.empty((B, T, HV, V), dtype=torch.float32, device=q.device)
        fs = (torch.empty((N, HV, K, V), dtype=torch.float32, device=q.device)
              if output_final_state else None)
    else:
        o, fs = out
    st = load().gdp_chunk_fwd_noalloc(_p(q), _p(k), _p(v), _p(beta), _p(g), _p(initial_state),
                                      _p(cu_seqlens), N, B, T, H, HV, K, V, M, int(chunk_size),
                                      float(scale), 1 if use_qk_l2norm else 0, _DTYPE[q.dtype],
                                      _p(o), _p(fs), _stream(q.device))
    _check("gdp_chunk_fwd_noalloc", st)
    return o, fs


def gdp_read_status(workspace) -> int:
    """Synchronise and read the device status word of a chunk_fwd workspace."""
    return int(load().gdp_read_status(_p(workspace), _stream(workspace.device)))


# ----------------------------------------------------------------------------------
# decode recurrent update
# ----------------------------------------------------------------------------------

def gdp_recurrent_update(q, k, v, beta, g, state, scale: float | None = None,
                         use_qk_l2norm: bool = False, out=None):
    """Recurrent update over L = S*M steps per request; ``state`` [n,HV,K,V] fp32 is
    updated in place. Returns o [n,L,HV,V] fp32 (one row per step)."""
    _need_cuda(q, k, v, beta, g, state)
    n, L, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if tuple(k.shape) != (n, L, H, K) or tuple(v.shape[:2]) != (n, L):
        raise ValueError("q, k must be [n,L,H,K] and v [n,L,HV,V]")
    if tuple(beta.shape) != (n, L, HV) or tuple(g.shape) != (n, L, HV):
        raise ValueError("beta and g must be [n,L,HV]")
    if tuple(state.shape) != (n, HV, K, V) or state.dtype != torch.float32:
        raise ValueError("state must be fp32 [n,HV,K,V]")
    for t in (q, k, v, beta, g, state):
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    if scale is None:
        scale = K ** -0.5
    o = out if out is not None else torch.empty((n, L, HV, V), dtype=torch.float32,
                                                device=q.device)
    st = load().gdp_recurrent_update(_p(q), _p(k), _p(v), _p(beta), _p(g), _p(state), n, L, H,
                                     HV, K, V, float(scale), 1 if use_qk_l2norm else 0,
                                     _DTYPE[q.dtype], _p(o), _stream(q.device))
    _check("gdp_recurrent_update", st)
    return o


def gdp_recurrent_update_slots(q, k, v, beta, g, state_pool, state_slot, scale=None,
                               use_qk_l2norm: bool = False, status=None, out=None):
    """Recurrent update of a decode batch whose states live in a pool: request r
    updates ``state_pool[state_slot[r]]`` in place (``state_slot`` int32 [n] on the
    device; -1 marks a padding request, whose o rows are zero and which touches no
    state). ``status`` (optional int32 device tensor, one element) is set to 1 when
    a slot is out of range or repeated; those requests are skipped. Returns o."""
    _need_cuda(q, k, v, beta, g, state_pool, state_slot, status)
    n, L, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if tuple(k.shape) != (n, L, H, K) or tuple(v.shape[:2]) != (n, L):
        raise ValueError("q, k must be [n,L,H,K] and v [n,L,HV,V]")
    if tuple(beta.shape) != (n, L, HV) or tuple(g.shape) != (n, L, HV):
        raise ValueError("beta and g must be [n,L,HV]")
    if (state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (HV, K, V)
            or state_pool.dtype != torch.float32):
        raise ValueError("state_pool must be fp32 [n_slots,HV,K,V]")
    if tuple(state_slot.shape) != (n,) or state_slot.dtype != torch.int32:
        raise ValueError("state_slot must be int32 [n]")
    if status is not None and (status.dtype != torch.int32 or status.numel() < 1):
        raise ValueError("status must be an int32 device tensor")
    for t in (q, k, v, beta, g, state_pool, state_slot):
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    if scale is None:
        scale = K ** -0.5
    o = out if out is not None else torch.empty((n, L, HV, V), dtype=torch.float32,
                                                device=q.device)
    st = load().gdp_recurrent_update_slots(
        _p(q), _p(k), _p(v), _p(beta), _p(g), _p(state_pool), _p(state_slot),
        state_pool.shape[0], n, L, H, HV, K, V, float(scale), 1 if use_qk_l2norm else 0,
        _DTYPE[q.dtype], _p(o), _p(status), _stream(q.device))
    _check("gdp_recurrent_update_slots", st)
    return o


def gdp_debug_wait_fault(arm: bool, budget_seconds: float = 0.0):
    """Test hook (off by default): arm a one-shot missing tensor-core commit in the
    next 128-position WY launch so that one bounded device wait runs out, and/or set
    the wait budget (<= 0: the default 2 s)."""
    _check("gdp_debug_wait_fault", load().gdp_debug_wait_fault(1 if arm else 0,
                                                                float(budget_seconds)))


def _conv_common(xp, conv_w, conv_b, ba, A_log, dt_bias, M, H, G, P, N):
    _need_cuda(xp, conv_w, conv_b, ba, A_log, dt_bias)
    if xp.dtype not in _DTYPE or ba.dtype != xp.dtype:
        raise ValueError("xp and ba must share a dtype in {bf16, fp16, fp32}")
    if xp.dim() != 3 or ba.dim() != 3 or xp.stride(-1) != 1 or ba.stride(-1) != 1:
        raise ValueError("xp and ba must be [n, T, D] with a contiguous last dimension")
    n, T, C = xp.shape
    if C != M * H * P + M * G * N + G * N or tuple(ba.shape) != (n, T, M * H + H):
        raise ValueError("xp/ba last dimensions do not match M, H, G, P, N")
    if conv_w.dim() != 2 or conv_w.shape[0] != C:
        raise ValueError("conv_w must be [C, W]")
    W = conv_w.shape[1]
    conv_w = conv_w.to(torch.float32).contiguous()
    conv_b = None if conv_b is None else conv_b.to(torch.float32).contiguous()
    return n, T, C, W, conv_w, conv_b, A_log.to(torch.float32).contiguous(), \
        dt_bias.to(torch.float32).contiguous()


def gdp_prefill_conv_prepare(xp, conv_w, conv_b, ba, A_log, dt_bias, num_householder: int,
                             num_heads: int, num_groups: int, head_dim: int, state_dim: int,
                             conv_state=None, cu_seqlens=None, return_conv_state=True,
                             out=None):
    """Short causal conv (+ SiLU) fused with the prefill prepare. Returns
    (q, k, v, beta, g, conv_state_out or None); conv_state_out [N, C, W-1]."""
    M, H, G, P, N = num_householder, num_heads, num_groups, head_dim, state_dim
    n, T, C, W, conv_w, conv_b, A_log, dt_bias = _conv_common(xp, conv_w, conv_b, ba, A_log,
                                                              dt_bias, M, H, G, P, N)
    NS = n if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    if conv_state is not None and (tuple(conv_state.shape) != (NS, C, W - 1)
                                   or conv_state.dtype != xp.dtype
                                   or not conv_state.is_contiguous()):
        raise ValueError("conv_state must be [N, C, W-1] in xp's dtype")
    dev = xp.device
    if out is None:
        out = (torch.empty((n, T, H, N), dtype=xp.dtype, device=dev),
               torch.empty((n, T * M, H, N), dtype=xp.dtype, device=dev),
               torch.empty((n, T * M, H, P), dtype=xp.dtype, device=dev),
               torch.empty((n, T * M, H), dtype=torch.float32, device=dev),
               torch.empty((n, T, H), dtype=torch.float32, device=dev))
    q, k, v, beta, g = out
    st_out = (torch.empty((NS, C, W - 1), dtype=xp.dtype, device=dev)
              if return_conv_state else None)
    st = load().gdp_prefill_conv_prepare(
        _p(xp), xp.stride(0), xp.stride(1), _p(conv_w), _p(conv_b), W, _p(conv_state),
        _p(st_out), _p(cu_seqlens), NS, _p(ba), ba.stride(0), ba.stride(1), _p(A_log),
        _p(dt_bias), n, T, M, H, G, P, N, _DTYPE[xp.dtype], _p(q), _p(k), _p(v), _p(beta),
        _p(g), _stream(dev))
    _check("gdp_prefill_conv_prepare", st)
    return q, k, v, beta, g, st_out


def gdp_decode_conv_prepare(xp, conv_w, conv_b, ba, A_log, dt_bias, num_householder: int,
                            num_heads: int, num_groups: int, head_dim: int, state_dim: int,
                            conv_state_pool, conv_slot, status=None, out=None):
    """Short causal conv (+ SiLU) fused with the decode prepare; conv states live in
    ``conv_state_pool`` [n_slots, C, W-1] (updated in place), ``conv_slot`` int32 [n]
    names each request's entry (-1: padding, zero q/k/v). Returns (q, k, v, beta, g)."""
    M, H, G, P, N = num_householder, num_heads, num_groups, head_dim, state_dim
    n, S, C, W, conv_w, conv_b, A_log, dt_bias = _conv_common(xp, conv_w, conv_b, ba, A_log,
                                                              dt_bias, M, H, G, P, N)
    _need_cuda(conv_state_pool, conv_slot, status)
    if (conv_state_pool.dim() != 3 or tuple(conv_state_pool.shape[1:]) != (C, W - 1)
            or conv_state_pool.dtype != xp.dtype or not conv_state_pool.is_contiguous()):
        raise ValueError("conv_state_pool must be [n_slots, C, W-1] in xp's dtype")
    if tuple(conv_slot.shape) != (n,) or conv_slot.dtype != torch.int32:
        raise ValueError("conv_slot must be int32 [n]")
    dev = xp.device
    L = S * M
    if out is None:
        out = (torch.empty((n, L, H, N), dtype=xp.dtype, device=dev),
               torch.empty((n, L, H, N), dtype=xp.dtype, device=dev),
               torch.empty((n, L, H, P), dtype=xp.dtype, device=dev),
               torch.empty((n, L, H), dtype=torch.float32, device=dev),
               torch.empty((n, L, H), dtype=torch.float32, device=dev))
    q, k, v, beta, g = out
    st = load().gdp_decode_conv_prepare(
        _p(xp), xp.stride(0), xp.stride(1), _p(conv_w), _p(conv_b), W, _p(conv_state_pool),
        _p(conv_slot), conv_state_pool.shape[0], _p(ba), ba.stride(0), ba.stride(1), _p(A_log),
        _p(dt_bias), n, S, M, H, G, P, N, _DTYPE[xp.dtype], _p(q), _p(k), _p(v), _p(beta),
        _p(g), _p(status), _stream(dev))
    _check("gdp_decode_conv_prepare", st)
    return q, k, v, beta, g
