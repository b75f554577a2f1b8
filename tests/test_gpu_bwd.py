"""Parity of the GPU backward pass (``kda.bwd`` through ``kda_bwd``) with the fp64
reverse-mode oracle (``oracle.recurrent_bwd``).

Inputs are the seeded workloads of ``gated_delta_rule_30_gb300.inputs`` and the
output gradients its ``cotangents`` draws.  All eight gradients are compared over
the whole tensors.  The kernel computes in fp32 token by token, so the bound is
far tighter than the forward's bf16 one: a relative Frobenius error of at most
1e-3 per gradient (fp32 rounding over a few thousand dependent steps stays
below 1e-5), and a max-abs error of at most 1e-3 of the gradient's largest
magnitude.  A mistake in any step of the reverse mode moves some gradient by
O(1) of its norm.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_30_gb300 import inputs
from kda_testutil import errors, to_dev

pytestmark = pytest.mark.gpu

RTOL = 1e-3
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dh0")


def custom(T=None, lens=None, H=2, state=torch.float32, seed=7, lower_bound=-5.0, B=1):
    w = inputs.Workload("custom", B, T, H, seed, state_dtype=state, lower_bound=lower_bound,
                        lens=None if lens is None else tuple(lens))
    return inputs.make(w), seed


def run_bwd(p, ct, with_dhT=True, workspace=None, qkn=False, low_memory=False):
    import gated_delta_rule_30_gb300 as kda
    d = to_dev(p)
    dout = ct["dout"].cuda()
    dhT = ct["dfinal_state"].cuda() if with_dhT else None
    r = kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"], d["dt_bias"],
                d["lower_bound"], dout, initial_state=d["initial_state"], dfinal_state=dhT,
                cu_seqlens=d["cu_seqlens"], workspace=workspace, use_qk_l2norm_in_kernel=qkn,
                low_memory=low_memory)
    kda.device_status()
    torch.cuda.synchronize()
    return {n: r[n].cpu() for n in NAMES}


def run_ref(oracle_mod, p, ct, with_dhT=True, qkn=False):
    return oracle_mod.recurrent_bwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"],
                                    p["A_log"], p["dt_bias"], p["lower_bound"], ct["dout"],
                                    initial_state=p["initial_state"],
                                    dfinal_state=ct["dfinal_state"] if with_dhT else None,
                                    cu_seqlens=p["cu_seqlens"], qk_l2norm=qkn)


def compare(got, ref, what, names=NAMES):
    for n in names:
        g = got[n].to(torch.float64).numpy().reshape(np.shape(ref[n]))
        rel, mx = errors(g, ref[n])
        scale = float(np.abs(ref[n]).max()) if np.size(ref[n]) else 0.0
        print(f"[bwd parity] {what} {n}: rel_fro={rel:.3e} max_abs={mx:.3e} (max |ref| {scale:.3e})")
        assert np.isfinite(rel) and rel <= RTOL, f"{what} {n}: rel_fro={rel:.3e} > {RTOL}"
        assert mx <= RTOL * max(scale, 1e-30), f"{what} {n}: max_abs={mx:.3e}"


def check(oracle_mod, p, seed, what, with_dhT=True, qkn=False):
    ct = inputs.cotangents(p, seed)
    got = run_bwd(p, ct, with_dhT, qkn=qkn)
    ref = run_ref(oracle_mod, p, ct, with_dhT, qkn=qkn)
    compare(got, ref, what)
    return got


def test_dense_ragged_tail(oracle_mod):
    """Two sequences of 40 tokens: two full 16-token segments and an 8-token tail."""
    p, s = custom(T=40, B=2, H=3)
    check(oracle_mod, p, s, "B=2 T=40")


@pytest.mark.parametrize("T", [1, 8, 9, 16, 17, 100])
def test_segment_edges(oracle_mod, T):
    """Lengths at and around the 8-token half and 16-token segment boundaries."""
    p, s = custom(T=T, H=2, seed=T)
    check(oracle_mod, p, s, f"T={T}")


def test_varlen_bf16_state(oracle_mod):
    """Packed sequences with empty and one-token members, bf16 initial state."""
    p, s = custom(lens=[0, 1, 7, 8, 9, 16, 17, 33, 64, 100, 0], H=2, state=torch.bfloat16, seed=11)
    check(oracle_mod, p, s, "varlen bf16")


def test_no_state_no_final_gradient(oracle_mod):
    p, s = custom(T=70, H=2, state=None, seed=12)
    check(oracle_mod, p, s, "no state", with_dhT=False)


@pytest.mark.parametrize("lb", [-0.6, -12.0])
def test_clamp(oracle_mod, lb):
    """lb = -0.6 clamps about half of the channels (their gate gradient is zero);
    lb = -12 is below the forward's range but valid for the backward pass."""
    p, s = custom(T=50, H=2, lower_bound=lb, seed=13)
    check(oracle_mod, p, s, f"lb={lb}")


def test_empty_sequences_pass_the_final_gradient():
    """T = 0: no token gradients, dh0 = dfinal_state, parameter gradients zero."""
    p, s = custom(T=0, B=2, H=2, seed=14)
    ct = inputs.cotangents(p, s)
    got = run_bwd(p, ct)
    assert torch.equal(got["dh0"], ct["dfinal_state"])
    assert torch.count_nonzero(got["dA_log"]) == 0 and torch.count_nonzero(got["ddt_bias"]) == 0


def test_deterministic():
    """Every sum is taken in a fixed order: two runs agree bit for bit."""
    p, s = custom(lens=[33, 70, 5], H=3, seed=15)
    ct = inputs.cotangents(p, s)
    a = run_bwd(p, ct)
    b = run_bwd(p, ct)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n


def test_malformed_cu_seqlens_reported():
    """A decreasing cu_seqlens is caught on the device and reported."""
    import gated_delta_rule_30_gb300 as kda
    p, s = custom(lens=[10, 20], H=1, seed=16)
    ct = inputs.cotangents(p, s)
    p2 = dict(p)
    p2["cu_seqlens"] = torch.tensor([0, 31, 30], dtype=torch.int32)
    with pytest.raises(kda.KDAError) as e:
        run_bwd(p2, ct)
    assert e.value.code == 5
    kda.device_status()  # cleared


def test_dense_prefill_full_size(oracle_mod):
    """The full dense_prefill workload (B=8 T=2048 H=16, fp32 state): every
    gradient element of all 128 (sequence, head) pairs."""
    w = inputs.WORKLOADS["dense_prefill"]
    check(oracle_mod, inputs.make(w), w.seed, "dense_prefill")


def test_long_context_full_size_suffix(oracle_mod):
    """The full long_context workload (T=65536 H=32, the benchmark's launch) with
    dout zero before the last 1024 tokens.  On two heads the oracle gives the
    state entering the suffix (its forward over the first 64512 tokens) and then
    the exact gradients of the suffix's tokens, which the GPU must match: they
    depend on the checkpoints the kernel took over the whole length."""
    w = inputs.WORKLOADS["long_context"]
    p = inputs.make(w)
    ct = inputs.cotangents(p, w.seed)
    P = 1024
    T = p["T"]
    ct["dout"][:, : T - P] = 0
    got = run_bwd(p, ct)
    heads = [0, 17]
    hs = torch.tensor(heads)
    sub = {key: p[key].index_select(2, hs).contiguous() for key in ("q", "k", "v", "g", "beta")}
    A_log = p["A_log"].index_select(0, hs).contiguous()
    dt_bias = p["dt_bias"].index_select(0, hs).contiguous()
    h0 = p["initial_state"].index_select(1, hs).contiguous()
    pre = {key: x[:, : T - P].contiguous() for key, x in sub.items()}
    suf = {key: x[:, T - P:].contiguous() for key, x in sub.items()}
    _, S_mid = oracle_mod.recurrent(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"],
                                    p["scale"], A_log, dt_bias, p["lower_bound"], initial_state=h0)
    ref = oracle_mod.recurrent_bwd(suf["q"], suf["k"], suf["v"], suf["g"], suf["beta"],
                                   p["scale"], A_log, dt_bias, p["lower_bound"],
                                   ct["dout"].index_select(2, hs)[:, T - P:].contiguous(),
                                   initial_state=S_mid,
                                   dfinal_state=ct["dfinal_state"].index_select(1, hs).contiguous())
    part = {n: got[n].index_select(2, hs)[:, T - P:] for n in ("dq", "dk", "dv", "dg")}
    part["dbeta"] = got["dbeta"].index_select(2, hs)[:, T - P:]
    compare(part, ref, "long_context suffix", names=("dq", "dk", "dv", "dg", "dbeta"))


@pytest.mark.parametrize("name", ["varlen_packed", "state_io"])
def test_packed_workloads_full_size(oracle_mod, name):
    """The full varlen_packed (32 sequences of 1..4096 tokens, H=32, bf16 state) and
    state_io (1024 sequences of 1..128 tokens, H=32, fp32 state) workloads: every
    element of all eight gradients of every (sequence, head) pair."""
    w = inputs.WORKLOADS[name]
    check(oracle_mod, inputs.make(w), w.seed, name)


@pytest.mark.parametrize("case", ["packed", "dense_no_state"])
def test_qk_l2norm(oracle_mod, case):
    """The gradients of the forward with in-kernel q/k normalisation: raw q and k rows
    with norms spread over [0.05, 20] (the recipe of the forward's normalisation
    tests), against the oracle's reverse mode through the normalisation."""
    from test_gpu_qknorm import raw_qk
    if case == "packed":
        p, s = custom(lens=[70, 1, 129, 0, 33], H=2, seed=31)
    else:
        p, s = custom(T=100, B=2, H=3, state=None, seed=32)
    check(oracle_mod, raw_qk(p, s), s, f"qk_l2norm {case}", qkn=True)


def test_qk_l2norm_dense_prefill_full_size(oracle_mod):
    """dense_prefill at full size with raw q and k normalised in the kernel: every
    element of all eight gradients of all 128 pairs."""
    from test_gpu_qknorm import raw_qk
    w = inputs.WORKLOADS["dense_prefill"]
    check(oracle_mod, raw_qk(inputs.make(w), w.seed), w.seed, "qk_l2norm dense_prefill", qkn=True)


@pytest.mark.parametrize("qkn,low_memory", [(False, False), (True, False), (False, True)])
def test_autograd_chunk_kda(oracle_mod, qkn, low_memory):
    """chunk_kda is differentiable: loss.backward() through it gives, for every input,
    the bf16/fp32 cast of kda.bwd's gradient bit for bit, and those gradients match
    the oracle."""
    import gated_delta_rule_30_gb300 as kda
    from test_gpu_qknorm import raw_qk
    p, s = custom(lens=[40, 17, 0, 66], H=2, seed=41)
    if qkn:
        p = raw_qk(p, s)
    ct = inputs.cotangents(p, s)
    d = to_dev(p)
    names = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state")
    leaf = {n: d[n].clone().requires_grad_(True) for n in names}
    o, hT = kda.chunk_kda(leaf["q"], leaf["k"], leaf["v"], leaf["g"], leaf["beta"], leaf["A_log"],
                          leaf["dt_bias"], p["lower_bound"], scale=p["scale"],
                          initial_state=leaf["initial_state"], output_final_state=True,
                          cu_seqlens=d["cu_seqlens"], use_qk_l2norm_in_kernel=qkn,
                          low_memory_backward=low_memory)
    loss = (o.float() * ct["dout"].cuda().float()).sum() + (hT * ct["dfinal_state"].cuda()).sum()
    loss.backward()
    kda.device_status()
    direct = run_bwd(p, ct, qkn=qkn)
    grads = dict(zip(names, ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dh0")))
    for n, gname in grads.items():
        got = leaf[n].grad.cpu()
        assert got.dtype == leaf[n].dtype, n
        assert torch.equal(got, direct[gname].to(got.dtype)), n
    ref = run_ref(oracle_mod, p, ct, qkn=qkn)
    compare(direct, ref, f"autograd qkn={qkn}")
    # without any input requiring grad, no graph is recorded
    o2, _ = kda.chunk_kda(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                          p["lower_bound"], scale=p["scale"], initial_state=d["initial_state"],
                          cu_seqlens=d["cu_seqlens"], use_qk_l2norm_in_kernel=qkn)
    assert o2.grad_fn is None and torch.equal(o2, o.detach())


@pytest.mark.parametrize("case", ["packed", "dense", "qk_l2norm"])
def test_low_memory_bit_identical(oracle_mod, case):
    """KDA_BWD_LOW_MEMORY keeps one state per 64 tokens and replays each chunk once
    more: the same operations in the same order, so every gradient is bit-identical
    to the default mode's.  Lengths sit on and around the 8-, 16- and 64-token
    boundaries (0, 1, 8, 16, 17, 63, 64, 65, 100, 130, 192, 256, 257)."""
    lens = [0, 1, 8, 16, 17, 63, 64, 65, 100, 130, 192, 256, 257]
    if case == "dense":
        p, s = custom(T=321, B=2, H=2, seed=51)
    else:
        p, s = custom(lens=lens, H=2, seed=52, state=torch.bfloat16)
    qkn = case == "qk_l2norm"
    if qkn:
        from test_gpu_qknorm import raw_qk
        p = raw_qk(p, s)
    ct = inputs.cotangents(p, s)
    a = run_bwd(p, ct, qkn=qkn)
    b = run_bwd(p, ct, qkn=qkn, low_memory=True)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n
    compare(b, run_ref(oracle_mod, p, ct, qkn=qkn), f"low memory {case}")


@pytest.mark.parametrize("name", ["dense_prefill", "state_io"])
def test_low_memory_full_size(name):
    """Full workloads: low-memory gradients bit-identical to the default mode's
    (which the full-size parity tests compare with the oracle).  state_io runs
    131,072 short CTAs, so replay slots are claimed and returned at a high rate."""
    w = inputs.WORKLOADS[name]
    p = inputs.make(w)
    ct = inputs.cotangents(p, w.seed)
    a = run_bwd(p, ct)
    b = run_bwd(p, ct, low_memory=True)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n


def test_caller_workspace_stream_and_no_dh0(oracle_mod):
    """kda_bwd with an exactly sized caller workspace, on a side stream while the
    default stream runs another backward pass, and without dinitial_state: the
    gradients equal those of the plain call bit for bit."""
    import gated_delta_rule_30_gb300 as kda
    p, s = custom(lens=[90, 7, 33], H=2, seed=61)
    ct = inputs.cotangents(p, s)
    ref = run_bwd(p, ct)
    d = to_dev(p)
    need = kda.bwd_workspace_size(p["B"], p["T"], p["H"], p["N"], True)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    big, bs_ = custom(T=600, B=2, H=4, seed=62)
    bct = inputs.cotangents(big, bs_)
    bd = to_dev(big)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    # the default stream's pass (own cached workspace) overlaps the side stream's
    kda.bwd(bd["q"], bd["k"], bd["v"], bd["g"], bd["beta"], bd["scale"], bd["A_log"],
            bd["dt_bias"], bd["lower_bound"], bct["dout"].cuda(),
            initial_state=bd["initial_state"], dfinal_state=bct["dfinal_state"].cuda())
    with torch.cuda.stream(side):
        r = kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                    d["dt_bias"], d["lower_bound"], ct["dout"].cuda(side.device),
                    initial_state=d["initial_state"], dfinal_state=ct["dfinal_state"].cuda(),
                    cu_seqlens=d["cu_seqlens"], workspace=ws, want_dh0=False)
    torch.cuda.synchronize()
    kda.device_status()
    assert r["dh0"] is None
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias"):
        assert torch.equal(r[n].cpu(), ref[n]), n


def test_no_sequences():
    """cu_seqlens = [0] (no sequences, no tokens): nothing is walked; dA_log and
    ddt_bias are written as zeros and the state gradient is empty."""
    import gated_delta_rule_30_gb300 as kda
    p, s = custom(lens=[], H=3, seed=71, state=None)
    assert p["N"] == 0 and p["T"] == 0
    d = to_dev(p)
    ct = inputs.cotangents(p, s)
    r = kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"], d["dt_bias"],
                d["lower_bound"], ct["dout"].cuda(), cu_seqlens=d["cu_seqlens"])
    kda.device_status()
    assert torch.count_nonzero(r["dA_log"]) == 0 and torch.count_nonzero(r["ddt_bias"]) == 0
    assert r["dh0"].shape == (0, 3, 128, 128) and r["dq"].numel() == 0
