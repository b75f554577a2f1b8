"""Helpers shared by the GPU tests: run the CUDA path, compare with the oracle,
and decode the per-chunk records the chunk kernel writes into the workspace.

The record layout decoded here is the one documented in
``gated_delta_rule_30_gb300/csrc/kda_internal.h``.
"""
from __future__ import annotations

import numpy as np
import torch

RTOL_FRO = 5e-3   # relative Frobenius error bound on bf16 outputs and final states
ATOL_MAX = 3e-2   # max-abs error bound

REC_WQ, REC_KT, REC_AQ, REC_AQL, REC_UT, REC_GAM, REC_BYTES = (0, 32768, 49152, 57344, 65536,
                                                              81920, 82432)


def to_dev(p, device="cuda"):
    d = dict(p)
    for key in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state", "cu_seqlens"):
        if d.get(key) is not None:
            d[key] = d[key].to(device).contiguous()
    return d


def run_gpu(p, final_dtype="same", workspace=None, via_alloc=False):
    """Run the CUDA path on a problem dict from ``inputs.make`` (tensors on CPU).

    final_dtype: "same" (the initial state's dtype, or none), None, torch.float32 or torch.bfloat16.
    Returns (out [B,T,H,V] bf16 CPU, final_state CPU or None).
    """
    import gated_delta_rule_30_gb300 as kda
    d = to_dev(p)
    out = torch.empty_like(d["v"])
    if final_dtype == "same":
        final_dtype = None if d["initial_state"] is None else d["initial_state"].dtype
    hT = None
    if final_dtype is not None:
        H, K, V = d["q"].shape[2], d["q"].shape[3], d["v"].shape[3]
        hT = torch.full((p["N"], H, K, V), float("nan"), dtype=final_dtype, device="cuda")
    fn = kda.fwd_alloc if via_alloc else kda.fwd
    kw = {} if via_alloc else {"workspace": workspace}
    fn(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"], d["dt_bias"],
       d["lower_bound"], initial_state=d["initial_state"], final_state=hT,
       cu_seqlens=d["cu_seqlens"], **kw)
    kda.device_status()
    torch.cuda.synchronize()
    return out.cpu(), (None if hT is None else hT.cpu())


def run_oracle(oracle_mod, p, heads=None):
    """Oracle outputs (float64) for all heads, or for the listed heads only."""
    args = [p["q"], p["k"], p["v"], p["g"], p["beta"]]
    A_log, dt_bias, h0 = p["A_log"], p["dt_bias"], p["initial_state"]
    if heads is not None:
        hs = torch.tensor(heads)
        args = [x.index_select(2, hs).contiguous() for x in args]
        A_log = A_log.index_select(0, hs).contiguous()
        dt_bias = dt_bias.index_select(0, hs).contiguous()
        h0 = None if h0 is None else h0.index_select(1, hs).contiguous()
    return oracle_mod.recurrent(*args, p["scale"], A_log, dt_bias, p["lower_bound"],
                                initial_state=h0, cu_seqlens=p["cu_seqlens"])


def errors(gpu, ref):
    g = np.asarray(gpu.to(torch.float64) if isinstance(gpu, torch.Tensor) else gpu, np.float64)
    r = np.asarray(ref, np.float64)
    diff = g - r
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(diff) / (nr if nr > 0 else 1.0)
    return float(rel), float(np.abs(diff).max() if diff.size else 0.0)


def assert_close(gpu, ref, what, rtol=RTOL_FRO, atol=ATOL_MAX):
    rel, mx = errors(gpu, ref)
    assert np.isfinite(rel) and rel <= rtol and mx <= atol, \
        f"{what}: rel_fro={rel:.3e} (<= {rtol}), max_abs={mx:.3e} (<= {atol})"
    return rel, mx


# ----------------------------------------------------------------------------- record decoding

def _align256(x):
    return (x + 255) & ~255


def workspace_layout(N, max_chunks):
    off_chunk = 256
    off_info = off_chunk + _align256((N + 1) * 4)
    off_rec = off_info + _align256(max_chunks * 8)
    return off_chunk, off_info, off_rec


def read_schedule(ws, N, max_chunks):
    off_chunk, off_info, off_rec = workspace_layout(N, max_chunks)
    raw = ws.cpu().numpy()
    flags = raw[:4].view(np.int32)[0]
    chunk_off = raw[off_chunk:off_chunk + 4 * (N + 1)].view(np.int32).copy()
    n = int(chunk_off[-1])
    info = raw[off_info:off_info + 8 * n].view(np.int32).reshape(n, 2).copy()
    return int(flags), chunk_off, info, off_rec


def _bf16(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _mn_off(mn, k, lbo, sbo):
    return (mn // 8) * lbo + (k // 8) * sbo + (k % 8) * 16 + (mn % 8) * 2


def _k_off(r, k, lbo, sbo):
    return (r // 8) * sbo + (k // 8) * lbo + (r % 8) * 16 + (k % 8) * 2


def decode_record(rec_bytes):
    """rec_bytes: uint8 numpy array of REC_BYTES.  Returns dict of float64 arrays."""
    u16 = rec_bytes.view(np.uint16)
    m = np.arange(128)[:, None]
    k = np.arange(128)[None, :]
    wq = _bf16(u16[(REC_WQ + _mn_off(m, k, 2048, 128)) // 2])
    ch = np.arange(128)[:, None]
    t = np.arange(64)[None, :]
    kt = _bf16(u16[(REC_KT + _k_off(ch, t, 128, 1024)) // 2])   # [ch][t]
    i = np.arange(64)[:, None]
    j = np.arange(64)[None, :]
    aq = _bf16(u16[(REC_AQ + _k_off(i, j, 128, 1024)) // 2]) \
        + _bf16(u16[(REC_AQL + _k_off(i, j, 128, 1024)) // 2])  # hi + lo, [i][j]
    ut = _bf16(u16[REC_UT // 2: REC_UT // 2 + 128 * 64].reshape(128, 64))
    gam = rec_bytes[REC_GAM:REC_GAM + 512].view(np.float32).astype(np.float64)
    return {"W": wq[:64], "Qhat": wq[64:], "Ktil": kt.T, "Aqk": aq, "U": ut.T, "gamma": gam}
