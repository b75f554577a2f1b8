"""Seeded synthetic inputs for the KDA forward pass.

This module only draws random tensors; it holds none of the method's
arithmetic, and both the CUDA path and the fp64 oracle consume exactly the
tensors it returns.  All draws come from one CPU ``torch.Generator`` seeded
with ``seed``, in this order:

1. (packed/varlen only) sequence lengths ``randint(lo, hi + 1, (N,))`` (or
   the explicit ``lens`` of a custom workload, with no draw) and
   ``cu_seqlens = [0, cumsum(lens)]`` (int32);
2. ``q``, ``k``: ``randn(B, T, H, K)`` in fp32, L2-normalised over the last
   dimension in fp32, then rounded once to bf16;
3. ``v``, ``g``: ``randn(...)`` rounded to bf16;
4. ``beta``: ``sigmoid(randn(B, T, H))`` rounded to bf16;
5. ``A_log`` = ``log(U[1, 16))`` fp32 ``[H]``;
6. ``dt_bias`` = ``0.1 * randn(H, K)`` fp32 (0.1 read as a standard deviation);
7. ``initial_state`` = ``0.02 * randn(N, H, K, V)`` cast to the state dtype.

``lower_bound = -5`` and ``scale = K ** -0.5`` unless overridden.

``cotangents`` draws the backward pass's output gradients from a second
generator seeded with ``seed + 1000``: ``dout = randn`` shaped like ``v``
(bf16), then ``dfinal_state = randn(N, H, K, V)`` (fp32).

The five named workloads are those the benchmark and the parity tests use;
``shrink`` gives a smaller instance of the same recipe for fast tests.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

K_DIM = 128
V_DIM = 128


@dataclass
class Workload:
    name: str
    B: int
    T: int | None          # None for packed workloads (T = sum of lengths)
    H: int
    seed: int
    n_seqs: int | None = None      # packed: number of sequences
    len_range: tuple | None = None  # packed: (lo, hi) inclusive
    state_dtype: torch.dtype | None = None
    lower_bound: float = -5.0
    lens: tuple | None = None       # packed with explicit lengths (no length draw)
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "ref_small": Workload("ref_small: B=1 T=256 H=2, no state", 1, 256, 2, 0),
    "dense_prefill": Workload("dense_prefill: B=8 T=2048 H=16, fp32 state", 8, 2048, 16, 1,
                              state_dtype=torch.float32),
    "varlen_packed": Workload("varlen_packed: 32 seqs U[1,4096] H=32, bf16 state", 1, None, 32, 2,
                              n_seqs=32, len_range=(1, 4096), state_dtype=torch.bfloat16),
    "long_context": Workload("long_context: B=1 T=65536 H=32, fp32 state", 1, 65536, 32, 3,
                             state_dtype=torch.float32),
    "state_io": Workload("state_io: 1024 seqs U[1,128] H=32, fp32 state", 1, None, 32, 4,
                         n_seqs=1024, len_range=(1, 128), state_dtype=torch.float32),
}
# single-token step (one token per sequence with a state, as in decoding)
WORKLOADS["decode"] = Workload("decode: B=1024 T=1 H=32, fp32 state", 1024, 1, 32, 5,
                               state_dtype=torch.float32)
# long_context with its 32 heads split over 8 tensor-parallel GPUs: the 4 heads one GPU holds
WORKLOADS["long_context_4h"] = Workload("long_context_4h: B=1 T=65536 H=4, fp32 state", 1, 65536,
                                        4, 6, state_dtype=torch.float32)
# 16 heads of a 16k-token sequence (32 heads over 2 tensor-parallel GPUs): the smallest
# split the segmented path takes automatically (4 segments of 64 chunks)
WORKLOADS["prefill_16k_16h"] = Workload("prefill_16k_16h: B=1 T=16384 H=16, fp32 state", 1,
                                        16384, 16, 7, state_dtype=torch.float32)
# smaller instance of long_context used for profiler captures (inputs still exceed L2)
WORKLOADS["long_context_8k"] = Workload("long_context_8k: B=1 T=8192 H=32, fp32 state", 1, 8192,
                                        32, 3, state_dtype=torch.float32)
# smaller decoding step used for profiler captures (states still exceed L2: 2 x 0.5 GB)
WORKLOADS["decode_256"] = Workload("decode_256: B=256 T=1 H=32, fp32 state", 256, 1, 32, 5,
                                   state_dtype=torch.float32)
# smaller instance of state_io used for profiler captures (256 sequences; states and inputs
# still exceed L2: 1 GB of fp32 states in and out)
WORKLOADS["state_io_256"] = Workload("state_io_256: 256 seqs U[1,128] H=32, fp32 state", 1, None,
                                     32, 4, n_seqs=256, len_range=(1, 128),
                                     state_dtype=torch.float32)
WORKLOAD_ORDER = ["ref_small", "dense_prefill", "varlen_packed", "long_context", "state_io"]


def shrink(w: Workload, T: int | None = None, H: int | None = None, n_seqs: int | None = None,
           hi: int | None = None, B: int | None = None) -> Workload:
    """Same recipe, smaller sizes."""
    return Workload(w.name + " (shrunk)", B if B is not None else w.B,
                    T if (T is not None and w.T is not None) else w.T,
                    H if H is not None else w.H, w.seed,
                    n_seqs=n_seqs if (n_seqs is not None and w.n_seqs is not None) else w.n_seqs,
                    len_range=(w.len_range[0], hi) if (hi is not None and w.len_range) else
                    w.len_range, state_dtype=w.state_dtype, lower_bound=w.lower_bound)


def make(w: Workload, K: int = K_DIM, V: int = V_DIM) -> dict:
    """Draw the workload's tensors on the CPU (see module docstring)."""
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    cu = None
    if w.lens is not None or w.n_seqs is not None:
        if w.lens is not None:
            lens = torch.tensor(list(w.lens), dtype=torch.int64)
        else:
            lo, hi = w.len_range
            lens = torch.randint(lo, hi + 1, (w.n_seqs,), generator=gen, dtype=torch.int64)
        N = int(lens.numel())
        cu = torch.zeros(N + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lens, 0)
        B, T = 1, int(cu[-1])
        cu = cu.to(torch.int32)
    else:
        B, T, N = w.B, w.T, w.B
    H = w.H

    def unit(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True)
        return x.to(torch.bfloat16)

    q = unit((B, T, H, K))
    k = unit((B, T, H, K))
    v = torch.randn((B, T, H, V), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    g = torch.randn((B, T, H, K), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=gen, dtype=torch.float32)).to(
        torch.bfloat16)
    A_log = torch.log(torch.empty(H, dtype=torch.float32).uniform_(1.0, 16.0, generator=gen))
    dt_bias = 0.1 * torch.randn((H, K), generator=gen, dtype=torch.float32)
    h0 = None
    if w.state_dtype is not None:
        h0 = (0.02 * torch.randn((N, H, K, V), generator=gen, dtype=torch.float32)).to(
            w.state_dtype)
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
                lower_bound=float(w.lower_bound), scale=1.0 / math.sqrt(K),
                initial_state=h0, state_dtype=w.state_dtype, cu_seqlens=cu, B=B, T=T, H=H, N=N,
                K=K, V=V, name=w.name)


def cotangents(p: dict, seed: int) -> dict:
    """Seeded gradients of the forward's outputs for a problem drawn by ``make``
    (see module docstring); ``seed`` is the workload's seed."""
    gen = torch.Generator(device="cpu").manual_seed(seed + 1000)
    dout = torch.randn(tuple(p["v"].shape), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    dfinal = torch.randn((p["N"], p["H"], p["K"], p["V"]), generator=gen, dtype=torch.float32)
    return dict(dout=dout, dfinal_state=dfinal)


def head_tokens(p: dict) -> int:
    """Total (token, head) pairs in a problem drawn by ``make``."""
    return int(p["B"] * p["T"] * p["H"])
