"""kda_fwd_noalloc: the forward pass for callers that cannot allocate device
memory during a call (for instance a serving runtime that reserves all GPU
memory up front, or a plug-in under memory pools it does not own).  Its
scratch is a fixed area compiled into the library, so it is checked against
the allocating entry point, twice in a row on different problems (the area
keeps the previous call's contents), and its size limit is checked on the
host.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from gated_delta_rule_30_gb300 import inputs
from kda_testutil import assert_close, run_gpu, to_dev

FAKE = 0x10000


def _noalloc(kda):
    L = kda.lib()
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    L.kda_fwd_noalloc.restype = ctypes.c_int
    L.kda_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, vp, f32, vp, ctypes.c_int, vp,
                                  ctypes.c_int, vp, i32, i32, i32, i32, i32, i32, vp]
    L.kda_noalloc_scratch_bytes.restype = ctypes.c_size_t
    return L


def _run_noalloc(kda, p):
    L = _noalloc(kda)
    d = to_dev(p)
    out = torch.empty_like(d["v"])
    hT = None if d["initial_state"] is None else torch.empty_like(d["initial_state"])
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    B, T, H, K = d["q"].shape
    cu = d["cu_seqlens"]
    ns = 0 if cu is None else cu.numel() - 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.kda_fwd_noalloc(ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["g"]), ptr(d["beta"]),
                           d["scale"], ptr(out), ptr(d["A_log"]), ptr(d["dt_bias"]),
                           d["lower_bound"], ptr(d["initial_state"]), kda._state_dtype(hT),
                           ptr(hT), kda._state_dtype(hT), ptr(cu), ns, B, T, H, K, d["v"].shape[-1],
                           stream)
    assert rc == 0, L.kda_last_error_message().decode()
    kda.device_status()
    torch.cuda.synchronize()
    return out.cpu(), (None if hT is None else hT.cpu())


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_twice(kda_lib):
    cases = [inputs.Workload("noalloc a", 1, None, 4, 51, lens=(70, 5, 129),
                             state_dtype=torch.float32),
             inputs.Workload("noalloc b", 1, None, 2, 52, lens=(33, 64),
                             state_dtype=torch.bfloat16),
             # few long sequences: the automatic choice is the fused launch, whose
             # ready flags live in the same area
             inputs.Workload("noalloc c", 1, None, 2, 53, lens=(1024, 700),
                             state_dtype=torch.float32)]
    for w in cases:  # calls in a row; each sees the previous one's leftovers
        p = inputs.make(w)
        ref_out, ref_hT = run_gpu(p)
        out, hT = _run_noalloc(kda_lib, p)
        assert_close(out.double(), ref_out.double().numpy(), f"{w.name} out")
        assert_close(hT.double(), ref_hT.double().numpy(), f"{w.name} final_state")


@pytest.mark.gpu
def test_noalloc_single_token_batches_of_any_size(kda_lib):
    """A decoding step of 1024 sequences x 32 heads (T = 1): the single-token step
    uses no scratch, so the entry point accepts it and gives the same bits as the
    allocating entry point (the same kernel runs)."""
    kda_lib.set_recurrence_kernel("auto")
    L = _noalloc(kda_lib)
    assert L.kda_workspace_size(1024, 1, 32, 0, 0) <= L.kda_noalloc_scratch_bytes()
    p = inputs.make(inputs.WORKLOADS["decode"])
    ref_out, ref_hT = run_gpu(p)
    for _ in range(2):
        out, hT = _run_noalloc(kda_lib, p)
        assert kda_lib.last_path() == "decode"
        assert torch.equal(out, ref_out) and torch.equal(hT, ref_hT)


def test_noalloc_rejects_problems_above_the_area(kda_lib):
    L = _noalloc(kda_lib)
    limit = L.kda_noalloc_scratch_bytes()
    assert limit == 64 << 20
    need = L.kda_workspace_size(1, 65536, 32, 0, 0)
    assert need > limit
    rc = L.kda_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 0.088, FAKE, FAKE, FAKE, -5.0, None, 0,
                           None, 0, None, 0, 1, 65536, 32, 128, 128, None)
    assert rc == 2
    msg = L.kda_last_error_message().decode()
    assert "64 MiB" in msg and str(need) in msg
