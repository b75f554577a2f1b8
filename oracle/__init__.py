"""fp64 CPU oracle for the Kimi Delta Attention (KDA) forward pass.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``gated_delta_rule_30_gb300``) and never imports it.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, OpenMP over
(sequence, head) pairs); this module only compiles it with gcc, marshals
arguments through ctypes and reshapes results.  ``brute.py`` holds an
independent numpy brute force used to pin the C code.

What is computed (reading of "Flashkda Delta Attention", section "Core Kernel
API", and "MoonshotAI/FlashKDA", section "Kernel API and Constraints"; the
pages print no formula, so the plain gated-delta-rule reading is taken, see
``kda_oracle.c``):

    la_t = max(-exp(A_log[h]) * softplus(g_t + dt_bias[h]), lower_bound)
    S_t  = (I - beta_t k_t k_t^T) Diag(exp(la_t)) S_{t-1} + beta_t k_t v_t^T
    o_t  = scale * S_t^T q_t

State layout is [N, H, K, V] with S[c][j] (key channel c, value channel j).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_fp = ctypes.POINTER(ctypes.c_float)


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into libkda_oracle.so (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        L.kda_oracle_l2norm.restype = None
        L.kda_oracle_l2norm.argtypes = [_dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_double]
        L.kda_oracle_log_decay.restype = ctypes.c_double
        L.kda_oracle_log_decay.argtypes = [ctypes.c_double] * 4
        L.kda_oracle_gate.restype = ctypes.c_int
        L.kda_oracle_gate.argtypes = [_dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _dp, _dp,
                                      ctypes.c_double, _dp]
        L.kda_oracle_fwd_f64.restype = ctypes.c_int
        L.kda_oracle_fwd_f64.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_double, _dp, _dp,
                                         ctypes.c_double, _dp, _dp, _dp, _i64p, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_double, ctypes.c_int]
        L.kda_oracle_fwd_bf16.restype = ctypes.c_int
        L.kda_oracle_fwd_bf16.argtypes = [_u16p, _u16p, _u16p, _u16p, _u16p, ctypes.c_double, _fp,
                                          _fp, ctypes.c_double, ctypes.c_void_p, ctypes.c_int, _dp,
                                          _dp, _i64p, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
        L.kda_oracle_bwd_f64.restype = ctypes.c_int
        L.kda_oracle_bwd_f64.argtypes = ([_dp] * 5 + [ctypes.c_double, _dp, _dp, ctypes.c_double]
                                         + [_dp] * 3 + [_i64p] + [ctypes.c_int64] * 4
                                         + [_dp] * 8 + [ctypes.c_int])
        L.kda_oracle_chunk.restype = ctypes.c_int
        L.kda_oracle_chunk.argtypes = [_dp, ctypes.c_int64, _dp, ctypes.c_int64, _dp,
                                       ctypes.c_int64, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int64, _dp, _dp, _dp, _dp, _dp,
                                       _dp, _dp]
        L.kda_oracle_fwd_chunked.restype = ctypes.c_int
        L.kda_oracle_fwd_chunked.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_double, _dp, _dp,
                                             ctypes.c_double, _dp, _dp, _dp, _i64p,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int64]
        _lib = L
    return _lib


# ----------------------------------------------------------------------------- helpers

def _is_torch(x) -> bool:
    return type(x).__module__.startswith("torch")


def _f64(x) -> np.ndarray:
    """Any tensor/array -> contiguous float64 numpy (bf16/fp32 upcast is exact)."""
    if x is None:
        return None
    if _is_torch(x):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, typ=_dp):
    return None if a is None else a.ctypes.data_as(typ)


def _flatten_tokens(x, last):
    """[B, T, H, D] or [NT, H, D] -> [NT, H, D]; [B, T, H] or [NT, H] -> [NT, H]."""
    shp = tuple(x.shape)
    if last:
        return x.reshape((-1,) + shp[-2:])
    return x.reshape((-1, shp[-1]))


def _cu(cu_seqlens, B, T):
    if cu_seqlens is None:
        return np.arange(B + 1, dtype=np.int64) * T
    c = cu_seqlens
    if _is_torch(c):
        c = c.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(c, dtype=np.int64))


def _bt(q):
    shp = tuple(q.shape)
    if len(shp) == 4:
        return shp[0], shp[1]
    return 1, shp[0]


# ----------------------------------------------------------------------------- API

def log_decay(g, A_log, dt_bias, lower_bound):
    """la for g laid out [..., H, K]; returns float64 array of g's shape."""
    g64 = _f64(g)
    shp = g64.shape
    H, K = shp[-2], shp[-1]
    gf = np.ascontiguousarray(g64.reshape(-1, H, K))
    la = np.empty_like(gf)
    a = _f64(A_log).reshape(H)
    d = _f64(dt_bias).reshape(H, K)
    rc = lib().kda_oracle_gate(_ptr(gf), gf.shape[0], H, K, _ptr(a), _ptr(d), float(lower_bound),
                               _ptr(la))
    if rc:
        raise ValueError(f"kda_oracle_gate failed ({rc})")
    return la.reshape(shp)


L2NORM_EPS = 1e-6  # eps of the query/key normalisation (x / sqrt(|x|^2 + eps))


def l2norm(x, eps=L2NORM_EPS):
    """float64 copy of x [..., D] with every row scaled to x / sqrt(sum x^2 + eps)."""
    a = np.array(_f64(x), dtype=np.float64, order="C", copy=True)
    D = a.shape[-1]
    lib().kda_oracle_l2norm(_ptr(a), int(a.size // D), D, float(eps))
    return a


def l2norm_bwd(x, dxhat, eps=L2NORM_EPS):
    """Gradient with respect to x of sum(dxhat * l2norm(x)), row by row in float64:
    with n = sqrt(sum x^2 + eps) and xhat = x / n, dx = (dxhat - xhat (xhat . dxhat)) / n."""
    a = _f64(x)
    d = np.asarray(dxhat, dtype=np.float64).reshape(a.shape)
    n = np.sqrt(np.sum(a * a, axis=-1, keepdims=True) + eps)
    xh = a / n
    return (d - xh * np.sum(xh * d, axis=-1, keepdims=True)) / n


def recurrent(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None,
              cu_seqlens=None, erase=1.0, nthreads=0, qk_l2norm=False):
    """Token-by-token recurrence (the definition).

    q, k, g: [B, T, H, K] (or [NT, H, K]); v: [..., H, V]; beta: [B, T, H];
    A_log: [H]; dt_bias: [H, K]; initial_state: [N, H, K, V] or None;
    cu_seqlens: [N + 1] or None (then N = B).  Torch bf16 activations are read
    as bf16 bit patterns and upcast exactly inside the C code; anything else is
    converted to float64 first.  qk_l2norm: normalise every (token, head) row of
    q and k first (``l2norm``, in fp64).  Returns (out float64 shaped like v,
    final_state float64 [N, H, K, V]).
    """
    if qk_l2norm:
        q, k = l2norm(q), l2norm(k)
    B, T = _bt(q)
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    H, K = q.shape[-2], q.shape[-1]
    V = v.shape[-1]
    NT = int(np.prod(q.shape[:-2]))
    out = np.empty((NT, H, V), dtype=np.float64)
    hT = np.empty((N, H, K, V), dtype=np.float64)
    L = lib()
    typed = (erase == 1.0 and all(_is_torch(x) and str(x.dtype) == "torch.bfloat16"
                                  for x in (q, k, v, g, beta)))
    if typed:
        import torch

        def bits(x):
            return np.ascontiguousarray(x.detach().to("cpu").contiguous().view(torch.int16)
                                        .numpy().view(np.uint16))

        qb, kb, vb, gb, bb = (bits(x) for x in (q, k, v, g, beta))
        a32 = np.ascontiguousarray(A_log.detach().to("cpu").to(torch.float32).numpy())
        d32 = np.ascontiguousarray(dt_bias.detach().to("cpu").to(torch.float32).numpy())
        h0p, h0k, keep = None, 0, None
        if initial_state is not None:
            if initial_state.dtype == torch.bfloat16:
                keep = bits(initial_state)
                h0k = 1
            else:
                keep = np.ascontiguousarray(initial_state.detach().to("cpu").to(torch.float32)
                                            .numpy())
                h0k = 2
            h0p = keep.ctypes.data_as(ctypes.c_void_p)
        rc = L.kda_oracle_fwd_bf16(_ptr(qb, _u16p), _ptr(kb, _u16p), _ptr(vb, _u16p),
                                   _ptr(gb, _u16p), _ptr(bb, _u16p), float(scale), _ptr(a32, _fp),
                                   _ptr(d32, _fp), float(lower_bound), h0p, h0k, _ptr(out),
                                   _ptr(hT), _ptr(cu, _i64p), N, H, K, V, int(nthreads))
    else:
        qf, kf, vf, gf = (_f64(x) for x in (q, k, v, g))
        bf = _f64(beta)
        h0 = _f64(initial_state)
        rc = L.kda_oracle_fwd_f64(_ptr(qf), _ptr(kf), _ptr(vf), _ptr(gf), _ptr(bf), float(scale),
                                  _ptr(_f64(A_log)), _ptr(_f64(dt_bias)), float(lower_bound),
                                  _ptr(h0), _ptr(out), _ptr(hT), _ptr(cu, _i64p), N, H, K, V,
                                  float(erase), int(nthreads))
    if rc:
        raise ValueError(f"kda_oracle_fwd failed ({rc})")
    return out.reshape(tuple(v.shape[:-1]) + (V,)), hT


def recurrent_bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout,
                  initial_state=None, dfinal_state=None, cu_seqlens=None, nthreads=0,
                  qk_l2norm=False):
    """Reverse mode of ``recurrent`` (fp64): gradients of
    L = sum(dout * out) + sum(dfinal_state * final_state).

    Shapes as for ``recurrent``; dout is shaped like v, dfinal_state like the
    state [N, H, K, V] (None: no final-state term).  Returns a dict with dq, dk,
    dv, dg, dbeta (shaped like the inputs), dA_log [H], ddt_bias [H, K] and dh0
    [N, H, K, V], all float64.

    qk_l2norm: the gradients of ``recurrent(..., qk_l2norm=True)``.  The
    recurrence sees x_hat = x / n with n = sqrt(sum x^2 + eps) for every row of q
    and k; by the chain rule through that map, dx = (dx_hat - x_hat (x_hat .
    dx_hat)) / n, row by row (``l2norm_bwd``).
    """
    if qk_l2norm:
        qn, kn = l2norm(q), l2norm(k)
        res = recurrent_bwd(qn, kn, v, g, beta, scale, A_log, dt_bias, lower_bound, dout,
                            initial_state=initial_state, dfinal_state=dfinal_state,
                            cu_seqlens=cu_seqlens, nthreads=nthreads)
        res["dq"] = l2norm_bwd(q, res["dq"])
        res["dk"] = l2norm_bwd(k, res["dk"])
        return res
    B, T = _bt(q)
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    H, K = q.shape[-2], q.shape[-1]
    V = v.shape[-1]
    qf, kf, vf, gf, bf = (_f64(x) for x in (q, k, v, g, beta))
    h0 = _f64(initial_state)
    do = _f64(dout)
    dhT = _f64(dfinal_state)
    res = {"dq": np.empty_like(qf), "dk": np.empty_like(kf), "dv": np.empty_like(vf),
           "dg": np.empty_like(gf), "dbeta": np.empty_like(bf), "dA_log": np.empty(H),
           "ddt_bias": np.empty((H, K)), "dh0": np.empty((N, H, K, V))}
    rc = lib().kda_oracle_bwd_f64(_ptr(qf), _ptr(kf), _ptr(vf), _ptr(gf), _ptr(bf), float(scale),
                                  _ptr(_f64(A_log)), _ptr(_f64(dt_bias)), float(lower_bound),
                                  _ptr(h0), _ptr(do), _ptr(dhT), _ptr(cu, _i64p), N, H, K, V,
                                  *(_ptr(res[n]) for n in ("dq", "dk", "dv", "dg", "dbeta",
                                                           "dA_log", "ddt_bias", "dh0")),
                                  int(nthreads))
    if rc:
        raise ValueError(f"kda_oracle_bwd_f64 failed ({rc})")
    return res


def chunked(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None,
            cu_seqlens=None, chunk=64):
    """Chunkwise form chained over the sequences (fp64, elementwise exponentials)."""
    B, T = _bt(q)
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    H, K = q.shape[-2], q.shape[-1]
    V = v.shape[-1]
    qf, kf, vf, gf, bf = (_f64(x) for x in (q, k, v, g, beta))
    h0 = _f64(initial_state)
    NT = int(np.prod(q.shape[:-2]))
    out = np.empty((NT, H, V), dtype=np.float64)
    hT = np.empty((N, H, K, V), dtype=np.float64)
    rc = lib().kda_oracle_fwd_chunked(_ptr(qf), _ptr(kf), _ptr(vf), _ptr(gf), _ptr(bf),
                                      float(scale), _ptr(_f64(A_log)), _ptr(_f64(dt_bias)),
                                      float(lower_bound), _ptr(h0), _ptr(out), _ptr(hT),
                                      _ptr(cu, _i64p), N, H, K, V, int(chunk))
    if rc:
        raise ValueError(f"kda_oracle_fwd_chunked failed ({rc})")
    return out.reshape(tuple(v.shape[:-1]) + (V,)), hT


def chunk_stage(q, k, v, la, beta):
    """Intermediates of one chunk of one head.

    q, k: [c, K]; v: [c, V]; la: [c, K] log-decays; beta: [c].
    Returns dict with G [c,K], A [c,c], Aqk [c,c], T [c,c], W [c,K], U [c,V], gamma [K].
    """
    qf, kf, vf, lf, bf = (_f64(x) for x in (q, k, v, la, beta))
    c, K = qf.shape
    V = vf.shape[1]
    res = {"G": np.empty((c, K)), "A": np.empty((c, c)), "Aqk": np.empty((c, c)),
           "T": np.empty((c, c)), "W": np.empty((c, K)), "U": np.empty((c, V)),
           "gamma": np.empty((K,))}
    rc = lib().kda_oracle_chunk(_ptr(qf), K, _ptr(kf), K, _ptr(vf), V, _ptr(lf), _ptr(bf), 1, c,
                                K, V, *(_ptr(res[n]) for n in ("G", "A", "Aqk", "T", "W", "U",
                                                               "gamma")))
    if rc:
        raise ValueError(f"kda_oracle_chunk failed ({rc})")
    return res
