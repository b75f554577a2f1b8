"""Calls on two streams at once through the Python binding (GPU).

The binding reuses one scratch buffer per (device, stream), so two forward
passes enqueued on different streams without synchronising between them do not
share scratch memory; each result must match the oracle.
"""
import pytest
import torch

from gated_delta_rule_30_gb300 import inputs
from kda_testutil import assert_close, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def test_two_streams_overlap(kda_lib, oracle_mod):
    import gated_delta_rule_30_gb300 as kda
    kda.set_recurrence_kernel("auto")
    probs = [inputs.make(inputs.Workload("stream a", 1, None, 4, 91, lens=(900, 64, 3, 400),
                                         state_dtype=torch.float32)),
             inputs.make(inputs.Workload("stream b", 2, 700, 3, 92,
                                         state_dtype=torch.bfloat16))]
    devs = [to_dev(p) for p in probs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs, states = [], []
    torch.cuda.synchronize()
    for rep in range(3):  # the second and third rounds reuse each stream's cached buffer
        outs, states = [], []
        for d, s in zip(devs, streams):
            with torch.cuda.stream(s):
                out = torch.empty_like(d["v"])
                hT = torch.empty_like(d["initial_state"])
                kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"],
                        d["dt_bias"], d["lower_bound"], initial_state=d["initial_state"],
                        final_state=hT, cu_seqlens=d["cu_seqlens"])
                outs.append(out)
                states.append(hT)
    torch.cuda.synchronize()
    kda.device_status()
    keys = [k for k in kda._WS_CACHE if k[0] == "cuda"]
    assert len({k[2] for k in keys}) >= 2  # one buffer per stream
    for p, out, hT in zip(probs, outs, states):
        o_ref, h_ref = run_oracle(oracle_mod, p)
        assert_close(out.cpu().reshape(o_ref.shape), o_ref, "two streams: out")
        assert_close(hT.cpu(), h_ref, "two streams: final_state")
