"""A device-side wait that runs out (GPU).

Every wait of the kernels that can give up is bounded; on running out a CTA
records KDA_ERR_TIMEOUT in the library's status word, waits (with a longer,
fixed limit) for its own copies and MMAs in flight, frees its tensor memory and
leaves, and the launch's later CTAs leave at once.  The test makes that happen
on purpose with the test hook kda_set_wait_limit_ns: with a 1 ns limit every
wait that does not complete at once gives up (a short limit makes the kernels
poll without suspending).  No GPU fault is involved: the status comes back
through kda_device_status, and the next call with the default limit must match
the oracle, which shows that the aborted launch left no tensor memory
allocated and no copy in flight.
"""
import pytest
import torch

from gated_delta_rule_30_gb300 import inputs
from kda_testutil import assert_close, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def problem(T, H, seed, lens=None):
    w = inputs.Workload("timeout", 1, T, H, seed, state_dtype=torch.float32,
                        lens=None if lens is None else tuple(lens))
    return inputs.make(w)


CASES = {
    # few long sequences: the fused cooperative launch (the recurrence waits on
    # record-ready flags that the chunk workers set)
    "fused": ("fused", dict(T=4096, H=4, seed=81)),
    # segments, scan and the value-sliced recurrence over the segments
    "segmented": ("segmented", dict(T=4096, H=2, seed=82)),
    "transposed": ("transposed", dict(T=None, H=3, seed=83, lens=[300, 64, 129, 5])),
    "sliced": ("sliced", dict(T=None, H=3, seed=84, lens=[300, 64, 129, 5])),
    # the single-token step (its one bulk copy of the state)
    "decode": ("auto", dict(T=1, H=4, seed=85)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_wait_runs_out_then_next_call_is_correct(kda_lib, oracle_mod, case):
    import gated_delta_rule_30_gb300 as kda
    kind, kw = CASES[case]
    p = problem(**kw) if case != "decode" else inputs.make(
        inputs.Workload("timeout decode", 64, 1, 4, 85, state_dtype=torch.float32))
    d = to_dev(p)
    kda.set_recurrence_kernel(kind)
    try:
        out = torch.empty_like(d["v"])
        hT = torch.empty_like(d["initial_state"])
        kda.device_status()  # start from a clear status word
        kda.set_wait_limit_ns(1)
        try:
            kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"],
                    d["dt_bias"], d["lower_bound"], initial_state=d["initial_state"],
                    final_state=hT, cu_seqlens=d["cu_seqlens"])
            ran = kda.last_path()
            with pytest.raises(kda.KDAError) as ei:
                kda.device_status()
        finally:
            kda.set_wait_limit_ns()  # back to the default 2 s
        assert ei.value.code == 4, ei.value   # KDA_ERR_TIMEOUT
        want = {"auto": "decode"}.get(kind, kind)
        assert ran == want, (ran, want)
        kda.device_status()  # the word was cleared by the read above
        # the next call, with the default limit, is unaffected
        o_ref, h_ref = run_oracle(oracle_mod, p)
        out2, h2 = run_gpu(p)
        assert_close(out2.reshape(o_ref.shape), o_ref, f"{case}: out after a timeout")
        assert_close(h2, h_ref, f"{case}: final_state after a timeout")
    finally:
        kda.set_recurrence_kernel("auto")


def test_wait_limit_validation(kda_lib):
    L = kda_lib.lib()
    assert L.kda_set_wait_limit_ns(0) == 1
    assert L.kda_set_wait_limit_ns(2_000_000_001) == 1
    assert L.kda_set_wait_limit_ns(2_000_000_000) == 0
