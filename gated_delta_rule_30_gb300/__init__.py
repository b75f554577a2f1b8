"""GB300 (sm_103a) Kimi Delta Attention forward pass (and its backward pass).

Thin Python binding over the C ABI in ``include/kda.h`` (``libkda.so``, built
in-tree by ``gated_delta_rule_30_gb300.build``).  This module only marshals
arguments: it checks tensor shapes/dtypes/devices, passes raw device pointers
and the current CUDA stream, and turns status codes into exceptions.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and a missing library raises.

``fwd`` follows the call printed in "Flashkda Delta Attention", section "Core
Kernel API":

    fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
        initial_state=None, final_state=None, cu_seqlens=None)

``bwd`` returns the gradients of that operation (``kda_bwd``).
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["fwd", "chunk_kda", "bwd", "bwd_workspace_size", "lib", "library_path", "workspace_size", "device_status",
           "KDAError",
           "selftest_tcgen05", "set_recurrence_kernel", "set_stage_events", "last_path",
           "set_wait_limit_ns"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libkda.so")
_lib = None

KDA_OK = 0
FWD_QK_L2NORM = 1  # kda_fwd_ex flag (also a kda_bwd flag)
BWD_LOW_MEMORY = 2  # kda_bwd flag
_STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARGUMENT", 2: "KDA_ERR_UNSUPPORTED",
           3: "KDA_ERR_CUDA", 4: "KDA_ERR_TIMEOUT", 5: "KDA_ERR_DEVICE_INPUT"}
DTYPE_NONE, DTYPE_BF16, DTYPE_FP32 = 0, 1, 2


class KDAError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{_STATUS.get(code, code)}: {message}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def lib():
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()' or "
                "python gated_delta_rule_30_gb300/build.py)")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        fwd_args = [vp, vp, vp, vp, vp, f32, vp, vp, vp, f32, vp, ctypes.c_int, vp, ctypes.c_int,
                    vp, i32, i32, i32, i32, i32, i32]
        L.kda_fwd.restype = ctypes.c_int
        L.kda_fwd.argtypes = fwd_args + [vp]
        L.kda_fwd_ws.restype = ctypes.c_int
        L.kda_fwd_ws.argtypes = fwd_args + [vp, ctypes.c_size_t, vp]
        L.kda_fwd_ex.restype = ctypes.c_int
        L.kda_fwd_ex.argtypes = fwd_args + [ctypes.c_uint32, vp, ctypes.c_size_t, vp]
        L.kda_workspace_size.restype = ctypes.c_size_t
        L.kda_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.kda_device_status.restype = ctypes.c_int
        L.kda_device_status.argtypes = [vp]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_last_error_message.restype = ctypes.c_char_p
        L.kda_last_error_message.argtypes = []
        L.kda_abi_version.restype = ctypes.c_int
        L.kda_abi_version.argtypes = []
        L.kda_last_path.restype = ctypes.c_int
        L.kda_last_path.argtypes = []
        L.kda_set_recurrence_kernel.restype = ctypes.c_int
        L.kda_set_recurrence_kernel.argtypes = [i32]
        L.kda_set_stage_events.restype = ctypes.c_int
        L.kda_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
        L.kda_set_wait_limit_ns.restype = ctypes.c_int
        L.kda_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.kda_bwd.restype = ctypes.c_int
        L.kda_bwd.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, f32, vp, ctypes.c_int, vp, vp, vp,
                              i32, i32, i32, i32, i32, i32] + [vp] * 8 + \
            [ctypes.c_uint32, vp, ctypes.c_size_t, vp]
        L.kda_bwd_workspace_size.restype = ctypes.c_size_t
        L.kda_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i32, ctypes.c_uint32]
        L.kda_selftest_tcgen05.restype = ctypes.c_int
        L.kda_selftest_tcgen05.argtypes = [vp, vp, vp, i32, i32, vp]
        _lib = L
    return _lib


def _check(rc: int):
    if rc != KDA_OK:
        msg = lib().kda_last_error_message()
        raise KDAError(rc, msg.decode() if msg else "")


def _stream_ptr(device):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _state_dtype(t):
    import torch
    if t is None:
        return DTYPE_NONE
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    raise TypeError(f"state dtype must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# Scratch buffers reused across calls, one per (device, stream).  Each buffer
# is allocated while its stream is current, so torch's caching allocator
# orders its reuse after that stream's work; keying by stream means calls on
# different streams never share one (they would race on it), and replacing a
# buffer that has grown frees memory that only its own stream has used.
_WS_CACHE = {}


def workspace_size(B: int, T: int, H: int, num_seqs: int = 0, has_cu_seqlens: bool = False) -> int:
    n = lib().kda_workspace_size(B, T, H, num_seqs, 1 if has_cu_seqlens else 0)
    if n == 0:
        _check(1)
    return int(n)


def _workspace(device, stream, nbytes):
    """The cached scratch buffer of (device, stream), grown to at least nbytes.
    Must be called with ``stream`` current on ``device``."""
    import torch
    key = (device.type, device.index, stream.value)
    ws = _WS_CACHE.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _WS_CACHE[key] = ws
    return ws


def fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
        final_state=None, cu_seqlens=None, workspace=None, use_qk_l2norm_in_kernel=False):
    """KDA forward pass on the GPU; writes ``out`` (and ``final_state``) in place.

    q, k, g: bf16 [B, T, H, 128]; v, out: bf16 [B, T, H, 128]; beta: bf16 [B, T, H];
    A_log: fp32 [H]; dt_bias: fp32 [H, 128]; initial_state / final_state:
    [N, H, 128, 128] bf16 or fp32 (same dtype when both given) or None;
    cu_seqlens: int32 [N + 1] on the device (requires B = 1) or None.
    ``workspace``: optional uint8 device tensor of at least ``workspace_size``
    bytes; by default a buffer from torch's allocator is reused, one per (device,
    stream), so calls on different streams may overlap.  A caller-supplied
    workspace must not be used by another call until this call's work on the
    current stream has finished.
    ``use_qk_l2norm_in_kernel``: scale every (token, head) row of q and k to
    x / sqrt(|x|^2 + 1e-6) inside the kernels first (kda_fwd_ex flag).
    Returns ``out``.
    """
    import torch
    L = lib()
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    V = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape:
        raise ValueError("k and g must have q's shape")
    if tuple(v.shape) != (B, T, H, V) or tuple(out.shape) != (B, T, H, V):
        raise ValueError("v and out must be [B, T, H, V]")
    if tuple(beta.shape) != (B, T, H):
        raise ValueError("beta must be [B, T, H]")
    for name, t, shp in (("A_log", A_log, (H,)), ("dt_bias", dt_bias, (H, K))):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 \
                or not t.is_contiguous() or tuple(t.shape) != shp:
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of shape {shp}")
    num_seqs = 0
    if cu_seqlens is not None:
        if not cu_seqlens.is_cuda or cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 \
                or not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be a contiguous 1-D int32 CUDA tensor")
        num_seqs = cu_seqlens.numel() - 1
    N = num_seqs if cu_seqlens is not None else B
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        if t is not None:
            if not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (N, H, K, V):
                raise ValueError(f"{name} must be a contiguous CUDA tensor of shape {(N, H, K, V)}")
    dev = q.device
    stream = _stream_ptr(dev)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out), _ptr(A_log),
            _ptr(dt_bias), float(lower_bound), _ptr(initial_state), _state_dtype(initial_state),
            _ptr(final_state), _state_dtype(final_state), _ptr(cu_seqlens), int(num_seqs), B, T,
            H, K, V]
    with torch.cuda.device(dev):
        need = L.kda_workspace_size(B, T, H, num_seqs, 1 if cu_seqlens is not None else 0)
        if need == 0:
            _check(L.kda_fwd(*args, stream))  # reports the size error
        ws = workspace if workspace is not None else _workspace(dev, stream, need)
        flags = FWD_QK_L2NORM if use_qk_l2norm_in_kernel else 0
        _check(L.kda_fwd_ex(*args, flags, ctypes.c_void_p(ws.data_ptr()),
                            ctypes.c_size_t(ws.numel()), stream))
    return out


def chunk_kda(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale=None, initial_state=None,
              output_final_state=False, cu_seqlens=None, use_qk_l2norm_in_kernel=False,
              low_memory_backward=False):
    """Allocating form of ``fwd``: returns ``(o, final_state)``.

    ``o`` is a new bf16 tensor shaped like ``v``.  ``scale`` defaults to K^-0.5.
    With ``output_final_state`` a new final state [N, H, K, V] is returned, in the
    initial state's dtype (float32 when there is no initial state); otherwise
    ``final_state`` is None.  Everything else is as for ``fwd``.

    Differentiable: when gradients are enabled and any of q, k, v, g, beta,
    A_log, dt_bias or initial_state requires grad, the call is recorded for
    autograd, and the backward pass is one ``kda_bwd`` call (see ``bwd``).  The
    incoming gradient of ``o`` is used in bf16 (the kernel's dout dtype), that
    of the final state in fp32; each returned gradient has its input's dtype.
    ``low_memory_backward``: run that backward pass with ``low_memory=True``.
    """
    import torch
    if scale is None:
        scale = q.shape[-1] ** -0.5
    tensors = (q, k, v, g, beta, A_log, dt_bias, initial_state)
    if torch.is_grad_enabled() and any(isinstance(t, torch.Tensor) and t.requires_grad
                                       for t in tensors):
        return _chunk_kda_function().apply(q, k, v, g, beta, A_log, dt_bias, initial_state,
                                           cu_seqlens, float(lower_bound), float(scale),
                                           bool(output_final_state),
                                           bool(use_qk_l2norm_in_kernel),
                                           bool(low_memory_backward))
    return _chunk_kda_forward(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                              initial_state, output_final_state, cu_seqlens,
                              use_qk_l2norm_in_kernel)


def _chunk_kda_forward(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                       output_final_state, cu_seqlens, use_qk_l2norm_in_kernel):
    import torch
    o = torch.empty_like(v)
    hT = None
    if output_final_state:
        N = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
        dt = torch.float32 if initial_state is None else initial_state.dtype
        hT = torch.empty((N, q.shape[2], q.shape[3], v.shape[3]), dtype=dt, device=q.device)
    fwd(q, k, v, g, beta, scale, o, A_log, dt_bias, lower_bound, initial_state=initial_state,
        final_state=hT, cu_seqlens=cu_seqlens, use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel)
    return o, hT


_CHUNK_KDA_FN = None


def _chunk_kda_function():
    """The autograd Function behind a differentiable ``chunk_kda`` (made on first use,
    so that importing this module does not import torch)."""
    global _CHUNK_KDA_FN
    if _CHUNK_KDA_FN is not None:
        return _CHUNK_KDA_FN
    import torch

    class ChunkKDAFunction(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens, lower_bound,
                    scale, output_final_state, qk_norm, low_memory):
            with torch.no_grad():
                o, hT = _chunk_kda_forward(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                                           initial_state, output_final_state, cu_seqlens, qk_norm)
            ctx.save_for_backward(q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens)
            ctx.cfg = (lower_bound, scale, qk_norm, low_memory)
            if hT is not None:
                return o, hT
            return o, None

        @staticmethod
        def backward(ctx, do, dhT):
            q, k, v, g, beta, A_log, dt_bias, h0, cu = ctx.saved_tensors
            lower_bound, scale, qk_norm, low_memory = ctx.cfg
            need = ctx.needs_input_grad
            if do is None:
                do = torch.zeros_like(v)
            r = bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound,
                    do.to(torch.bfloat16).contiguous(), initial_state=h0,
                    dfinal_state=None if dhT is None else dhT.to(torch.float32).contiguous(),
                    cu_seqlens=cu, want_dh0=h0 is not None and need[7],
                    use_qk_l2norm_in_kernel=qk_norm, low_memory=low_memory)

            def out(name, like, i):
                return r[name].to(like.dtype) if need[i] else None

            return (out("dq", q, 0), out("dk", k, 1), out("dv", v, 2), out("dg", g, 3),
                    out("dbeta", beta, 4), out("dA_log", A_log, 5), out("ddt_bias", dt_bias, 6),
                    None if h0 is None else out("dh0", h0, 7), None, None, None, None, None, None)

    _CHUNK_KDA_FN = ChunkKDAFunction
    return _CHUNK_KDA_FN


def bwd_workspace_size(B: int, T: int, H: int, num_seqs: int = 0,
                       has_cu_seqlens: bool = False, low_memory: bool = False) -> int:
    n = lib().kda_bwd_workspace_size(B, T, H, num_seqs, 1 if has_cu_seqlens else 0,
                                     BWD_LOW_MEMORY if low_memory else 0)
    if n == 0:
        _check(1)
    return int(n)


def bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout, initial_state=None,
        dfinal_state=None, cu_seqlens=None, workspace=None, want_dh0=True,
        use_qk_l2norm_in_kernel=False, low_memory=False):
    """Backward pass of ``fwd`` on the GPU (``kda_bwd``): gradients of
    L = sum(dout * out) + sum(dfinal_state * final_state).

    Inputs as for ``fwd``; ``dout``: bf16, shaped like ``v``; ``dfinal_state``:
    fp32 [N, H, 128, 128] or None.  Returns a dict of new fp32 tensors: dq, dk,
    dg (like q), dv (like v), dbeta (like beta), dA_log [H], ddt_bias [H, 128]
    and dh0 [N, H, 128, 128] (None when ``want_dh0`` is false).
    ``use_qk_l2norm_in_kernel``: the gradients of ``fwd`` with that flag (q and k
    normalised row by row inside the kernels); dq and dk are then with respect to
    the raw rows.  ``low_memory``: checkpoint the state every 64 tokens instead of
    every 8 (about 1 KB of scratch per token per head instead of 8 KB; the same
    results, bit for bit, and slower).  ``workspace``:
    optional uint8 device tensor of at least ``bwd_workspace_size`` bytes; by
    default the per-(device, stream) buffer that ``fwd`` also uses is grown and
    reused.
    """
    import torch
    L = lib()
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("dout", dout)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    V = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape:
        raise ValueError("k and g must have q's shape")
    if tuple(v.shape) != (B, T, H, V) or tuple(dout.shape) != (B, T, H, V):
        raise ValueError("v and dout must be [B, T, H, V]")
    if tuple(beta.shape) != (B, T, H):
        raise ValueError("beta must be [B, T, H]")
    for name, t, shp in (("A_log", A_log, (H,)), ("dt_bias", dt_bias, (H, K))):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 \
                or not t.is_contiguous() or tuple(t.shape) != shp:
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of shape {shp}")
    num_seqs = 0
    if cu_seqlens is not None:
        if not cu_seqlens.is_cuda or cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 \
                or not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be a contiguous 1-D int32 CUDA tensor")
        num_seqs = cu_seqlens.numel() - 1
    N = num_seqs if cu_seqlens is not None else B
    if initial_state is not None:
        if not initial_state.is_cuda or not initial_state.is_contiguous() \
                or tuple(initial_state.shape) != (N, H, K, V):
            raise ValueError(f"initial_state must be a contiguous CUDA tensor of shape {(N, H, K, V)}")
    if dfinal_state is not None:
        if not dfinal_state.is_cuda or not dfinal_state.is_contiguous() \
                or dfinal_state.dtype != torch.float32 or tuple(dfinal_state.shape) != (N, H, K, V):
            raise ValueError("dfinal_state must be a contiguous CUDA float32 tensor of shape "
                             f"{(N, H, K, V)}")
    dev = q.device
    f32 = torch.float32
    res = {"dq": torch.empty(q.shape, dtype=f32, device=dev),
           "dk": torch.empty(q.shape, dtype=f32, device=dev),
           "dv": torch.empty(v.shape, dtype=f32, device=dev),
           "dg": torch.empty(q.shape, dtype=f32, device=dev),
           "dbeta": torch.empty(beta.shape, dtype=f32, device=dev),
           "dA_log": torch.empty((H,), dtype=f32, device=dev),
           "ddt_bias": torch.empty((H, K), dtype=f32, device=dev),
           "dh0": torch.empty((N, H, K, V), dtype=f32, device=dev) if want_dh0 else None}
    stream = _stream_ptr(dev)
    with torch.cuda.device(dev):
        flags = (FWD_QK_L2NORM if use_qk_l2norm_in_kernel else 0) | \
            (BWD_LOW_MEMORY if low_memory else 0)
        need = L.kda_bwd_workspace_size(B, T, H, num_seqs, 1 if cu_seqlens is not None else 0,
                                        flags)
        if need == 0:
            _check(1)
        ws = workspace if workspace is not None else _workspace(dev, stream, need)
        _check(L.kda_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(A_log),
                         _ptr(dt_bias), float(lower_bound), _ptr(initial_state),
                         _state_dtype(initial_state), _ptr(dout), _ptr(dfinal_state),
                         _ptr(cu_seqlens), int(num_seqs), B, T, H, K, V,
                         *(_ptr(res[n]) for n in ("dq", "dk", "dv", "dg", "dbeta", "dA_log",
                                                  "ddt_bias", "dh0")),
                         flags, ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(ws.numel()),
                         stream))
    return res


def fwd_alloc(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
              final_state=None, cu_seqlens=None):
    """As ``fwd`` but through ``kda_fwd`` (library-side stream-ordered scratch)."""
    import torch
    B, T, H, K = q.shape
    V = v.shape[-1]
    num_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    with torch.cuda.device(q.device):
        _check(lib().kda_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                             _ptr(out), _ptr(A_log), _ptr(dt_bias), float(lower_bound),
                             _ptr(initial_state), _state_dtype(initial_state), _ptr(final_state),
                             _state_dtype(final_state), _ptr(cu_seqlens), int(num_seqs), B, T, H,
                             K, V, _stream_ptr(q.device)))
    return out


def device_status(device=None):
    """Synchronise the current stream and raise if a device-side check fired."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(lib().kda_device_status(_stream_ptr(dev)))


RECURRENCE_KERNELS = {"auto": 0, "sliced": 1, "transposed": 2, "fused": 3, "segmented": 4}


def set_recurrence_kernel(kind: str = "auto"):
    """Choose the recurrence kernel for later calls: "auto", "sliced", "transposed", "fused"
    (chunk kernel and transposed recurrence in one cooperative launch; falls back to the
    two-kernel path when the problem has too many (sequence, head) pairs for it) or
    "segmented" (each sequence split into segments whose state maps are scanned, then all
    segments run at once).  The workspace size depends on this choice: query
    ``workspace_size`` after setting it."""
    if kind not in RECURRENCE_KERNELS:
        raise ValueError(f"kind must be one of {sorted(RECURRENCE_KERNELS)}")
    _check(lib().kda_set_recurrence_kernel(RECURRENCE_KERNELS[kind]))


PATHS = {1: "sliced", 2: "transposed", 3: "fused", 4: "decode", 5: "segmented"}


def last_path():
    """How this thread's last forward pass ran: "sliced", "transposed", "fused", "decode" or
    "segmented" (None before any)."""
    return PATHS.get(lib().kda_last_path())


def set_stage_events(events):
    """Record 4 or 6 CUDA events around the library's kernels in later calls (None: off).

    ``events``: ``torch.cuda.Event(enable_timing=True)`` objects; they mark
    before schedule / after schedule / after the chunk kernel / after the
    recurrence kernel on the call's stream (segmented path: after the chunk
    kernel / after the map pass / after the scan / after the recurrence).
    """
    L = lib()
    if events is None:
        _check(L.kda_set_stage_events(None, 0))
        return
    for e in events:
        if e.cuda_event == 0:
            raise ValueError("events must be created (record them once) before use")
    n = len(events)
    arr = (ctypes.c_void_p * n)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(L.kda_set_stage_events(arr, n))


def set_wait_limit_ns(limit_ns: int = 2_000_000_000, device=None):
    """Limit of the kernels' bounded device-side waits on ``device`` (the current one
    by default), in ns; 2e9 restores the default.  A test hook: a short limit makes
    a wait give up, which ``device_status`` then reports as KDA_ERR_TIMEOUT."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(lib().kda_set_wait_limit_ns(int(limit_ns)))


def selftest_tcgen05(a, b, N, K):
    """Run the tcgen05 operand-layout self-test (a: bf16 [128, K], b: bf16 [K, N], CUDA)."""
    import torch
    d = torch.empty((4, 128, N), dtype=torch.float32, device=a.device)
    with torch.cuda.device(a.device):
        _check(lib().kda_selftest_tcgen05(_ptr(a), _ptr(b), _ptr(d), N, K, _stream_ptr(a.device)))
    return d
