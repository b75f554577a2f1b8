"""The single-token step (T = 1 per sequence, no cu_seqlens) on the GPU.

kda_fwd takes it automatically for such problems: one pass over the states
instead of the chunk records.  It is checked against the fp64 oracle (the
token-by-token recurrence, which for one token is the definition itself) for
every state-dtype combination, in place, at the decode workload's full size
(whole tensors), and against the chunked path on the same inputs.
"""
import pytest
import torch

from gated_delta_rule_30_gb300 import inputs
from kda_testutil import assert_close, errors, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def one_token(B=16, H=4, state=torch.float32, seed=61, lower_bound=-5.0):
    w = inputs.Workload("one token", B, 1, H, seed, state_dtype=state, lower_bound=lower_bound)
    return inputs.make(w)


@pytest.fixture(autouse=True)
def auto_path(kda_lib):
    kda_lib.set_recurrence_kernel("auto")
    yield
    kda_lib.set_recurrence_kernel("auto")


@pytest.mark.parametrize("h0,hT", [(torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
                                   (None, torch.float32), (None, torch.bfloat16),
                                   (torch.float32, None), (torch.bfloat16, None), (None, None)])
def test_decode_matches_oracle(kda_lib, oracle_mod, h0, hT):
    p = one_token(state=h0, seed=62)
    out, st = run_gpu(p, final_dtype=hT)
    assert kda_lib.last_path() == "decode"
    o_ref, h_ref = run_oracle(oracle_mod, p)
    eo = errors(out.reshape(o_ref.shape), o_ref)
    print(f"\n[decode] h0={h0} hT={hT}: out rel_fro={eo[0]:.3e} max_abs={eo[1]:.3e}")
    assert_close(out.reshape(o_ref.shape), o_ref, "decode out")
    if st is not None:
        assert_close(st, h_ref, "decode final_state")


@pytest.mark.parametrize("lb", [0.0, -1.0, -10.0])
def test_decode_lower_bound(kda_lib, oracle_mod, lb):
    p = one_token(seed=63, lower_bound=lb)
    out, st = run_gpu(p)
    o_ref, h_ref = run_oracle(oracle_mod, p)
    assert_close(out.reshape(o_ref.shape), o_ref, f"lb={lb} out")
    assert_close(st, h_ref, f"lb={lb} final_state")


def test_decode_in_place(kda_lib, oracle_mod):
    import gated_delta_rule_30_gb300 as kda
    p = one_token(B=8, H=3, seed=64)
    o_ref, h_ref = run_oracle(oracle_mod, p)
    d = to_dev(p)
    out = torch.empty_like(d["v"])
    st = d["initial_state"].clone()
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"], d["dt_bias"],
            d["lower_bound"], initial_state=st, final_state=st)
    kda.device_status()
    assert kda.last_path() == "decode"
    assert_close(out.cpu().reshape(o_ref.shape), o_ref, "in-place out")
    assert_close(st.cpu(), h_ref, "in-place state")


def test_decode_agrees_with_chunked_path(kda_lib):
    p = one_token(B=32, H=4, seed=65)
    o1, h1 = run_gpu(p)
    kda_lib.set_recurrence_kernel("transposed")
    o2, h2 = run_gpu(p)
    assert kda_lib.last_path() == "transposed"
    assert_close(o1.double(), o2.double().numpy(), "decode vs chunked out")
    assert_close(h1.double(), h2.double().numpy(), "decode vs chunked state")


def test_decode_full_size(kda_lib, oracle_mod):
    """The decode workload (B=1024, T=1, H=32, fp32 state), whole tensors."""
    p = inputs.make(inputs.WORKLOADS["decode"])
    out, st = run_gpu(p)
    assert kda_lib.last_path() == "decode"
    o_ref, h_ref = run_oracle(oracle_mod, p)
    eo = assert_close(out.reshape(o_ref.shape), o_ref, "decode full out")
    es = assert_close(st, h_ref, "decode full final_state")
    print(f"\n[full] decode: out rel_fro={eo[0]:.3e} max_abs={eo[1]:.3e}; "
          f"state rel_fro={es[0]:.3e} max_abs={es[1]:.3e}")
