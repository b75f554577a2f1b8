"""In-kernel q/k L2 normalisation (kda_fwd_ex with KDA_FWD_QK_L2NORM) on the GPU.

Inputs follow the workload recipe except that q and k are NOT normalised: raw
N(0, 1) rows, each scaled by a factor drawn from [0.05, 20], so the kernels'
normalisation matters.  Every chunked path and the single-token step are
compared with the oracle run with ``qk_l2norm=True`` (rows normalised in fp64
before the recurrence), within the usual tolerances; the allocating entry
``chunk_kda`` must give the same bits as ``fwd``.
"""
import pytest
import torch

from gated_delta_rule_30_gb300 import inputs
from kda_testutil import assert_close, errors, to_dev

pytestmark = pytest.mark.gpu


def raw_qk(p, seed):
    """Replace q and k by un-normalised rows with widely varying norms."""
    gen = torch.Generator().manual_seed(seed)
    shp = p["q"].shape
    for key in ("q", "k"):
        x = torch.randn(shp, generator=gen)
        f = torch.exp(torch.empty(shp[:-1] + (1,)).uniform_(-3.0, 3.0, generator=gen))
        p[key] = (x * f).to(torch.bfloat16).contiguous()
    return p


def oracle_norm(oracle_mod, p):
    return oracle_mod.recurrent(p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"],
                                p["A_log"], p["dt_bias"], p["lower_bound"],
                                initial_state=p["initial_state"], cu_seqlens=p["cu_seqlens"],
                                qk_l2norm=True)


def run_norm(p, norm=True):
    import gated_delta_rule_30_gb300 as kda
    d = to_dev(p)
    out = torch.empty_like(d["v"])
    hT = None if d["initial_state"] is None else torch.empty_like(d["initial_state"])
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"], d["dt_bias"],
            d["lower_bound"], initial_state=d["initial_state"], final_state=hT,
            cu_seqlens=d["cu_seqlens"], use_qk_l2norm_in_kernel=norm)
    kda.device_status()
    return out.cpu(), (None if hT is None else hT.cpu())


CASES = [
    ("packed", inputs.Workload("qknorm packed", 1, None, 3, 71, lens=(70, 1, 129, 64, 0, 200),
                               state_dtype=torch.float32)),
    ("dense bf16 state", inputs.Workload("qknorm dense", 2, 300, 2, 72,
                                         state_dtype=torch.bfloat16)),
    ("long", inputs.Workload("qknorm long", 1, 4096, 4, 73, state_dtype=torch.float32)),
]


@pytest.mark.parametrize("kind", ["sliced", "transposed", "fused", "segmented"])
@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_qknorm_matches_oracle(kda_lib, oracle_mod, kind, name, w):
    p = raw_qk(inputs.make(w), 700 + w.seed)
    o_ref, h_ref = oracle_norm(oracle_mod, p)
    kda_lib.set_recurrence_kernel(kind)
    try:
        out, hT = run_norm(p)
    finally:
        kda_lib.set_recurrence_kernel("auto")
    eo = assert_close(out.reshape(o_ref.shape), o_ref, f"{name} [{kind}] out")
    es = assert_close(hT, h_ref, f"{name} [{kind}] final_state")
    print(f"\n[qknorm] {name} [{kind}]: out rel_fro={eo[0]:.3e} max_abs={eo[1]:.3e}; "
          f"state rel_fro={es[0]:.3e}")


def test_qknorm_changes_the_result(kda_lib, oracle_mod):
    """Without the flag the same raw inputs give a different pass (the flag runs).
    Un-normalised keys with |k|^2 >> 2 make the delta rule itself unstable, so the
    un-normalised result may even overflow: compare NaN-safely."""
    p = raw_qk(inputs.make(CASES[0][1]), 999)
    o_ref, _ = oracle_norm(oracle_mod, p)
    out, _ = run_norm(p, norm=False)
    rel = errors(out.reshape(o_ref.shape), o_ref)[0]
    assert not (rel <= 0.1), rel


@pytest.mark.parametrize("state", [torch.float32, torch.bfloat16, None])
def test_qknorm_single_token(kda_lib, oracle_mod, state):
    p = raw_qk(inputs.make(inputs.Workload("qknorm decode", 64, 1, 4, 74, state_dtype=state)), 74)
    o_ref, h_ref = oracle_norm(oracle_mod, p)
    out, hT = run_norm(p)
    assert kda_lib.last_path() == "decode"
    assert_close(out.reshape(o_ref.shape), o_ref, "decode out")
    if hT is not None:
        assert_close(hT, h_ref, "decode final_state")


def test_qknorm_full_size_dense_prefill(kda_lib, oracle_mod):
    w = inputs.WORKLOADS["dense_prefill"]
    p = raw_qk(inputs.make(w), 75)
    o_ref, h_ref = oracle_norm(oracle_mod, p)
    out, hT = run_norm(p)
    eo = assert_close(out.reshape(o_ref.shape), o_ref, "dense_prefill qknorm out")
    es = assert_close(hT, h_ref, "dense_prefill qknorm final_state")
    print(f"\n[qknorm] dense_prefill full: out rel_fro={eo[0]:.3e}; state rel_fro={es[0]:.3e}")


def test_chunk_kda_allocating_entry(kda_lib):
    import gated_delta_rule_30_gb300 as kda
    p = raw_qk(inputs.make(CASES[0][1]), 76)
    d = to_dev(p)
    o, hT = kda.chunk_kda(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                          d["lower_bound"], initial_state=d["initial_state"],
                          output_final_state=True, cu_seqlens=d["cu_seqlens"],
                          use_qk_l2norm_in_kernel=True)
    out, h2 = run_norm(p)
    assert o.dtype == torch.bfloat16 and hT.dtype == torch.float32
    assert torch.equal(o.cpu(), out) and torch.equal(hT.cpu(), h2)
    o2, none = kda.chunk_kda(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                             d["lower_bound"], cu_seqlens=d["cu_seqlens"])
    assert none is None and o2.shape == d["v"].shape
