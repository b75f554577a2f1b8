"""Pins for the fp64 oracle (CPU only).

The oracle is the reference for every GPU parity test, so it is checked here
against things other than itself: an exact-rational computation, a numpy
brute force with explicit transition matrices, closed forms of special cases
(single token, beta = 0, orthonormal overwrite, strong decay, linear-attention
limits), an independent softplus (torch), and the invariants of the method
(chunked form = recurrence, state passing = one call, packed = separate
calls).  Each is chosen so that a plausible slip (a dropped or mis-signed
term, a transposed state, decay applied after the write, a wrong clamp)
fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import brute

RNG_SEED = 1234


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_problem(rng, T, H, K, V, lower_bound=-5.0, h0=True, N=1):
    q = _unit(rng.standard_normal((T, H, K)))
    k = _unit(rng.standard_normal((T, H, K)))
    v = rng.standard_normal((T, H, V))
    g = rng.standard_normal((T, H, K))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    A_log = np.log(rng.uniform(1.0, 16.0, H))
    dt_bias = 0.1 * rng.standard_normal((H, K))
    s0 = 0.02 * rng.standard_normal((N, H, K, V)) if h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
                lower_bound=lower_bound, scale=K ** -0.5, h0=s0)


def run_oracle(oracle_mod, p, cu=None, erase=1.0):
    return oracle_mod.recurrent(p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"], p["A_log"],
                                p["dt_bias"], p["lower_bound"], initial_state=p["h0"],
                                cu_seqlens=cu, erase=erase)


# ----------------------------------------------------------------------------- gate

def test_gate_matches_torch_softplus(oracle_mod):
    rng = np.random.default_rng(RNG_SEED)
    H, K = 3, 16
    g = rng.uniform(-40, 40, (50, H, K))
    A_log = np.log(rng.uniform(0.1, 16.0, H))
    dt_bias = rng.standard_normal((H, K))
    for lb in (-5.0, -50.0, -1e9):
        la = oracle_mod.log_decay(g, A_log, dt_bias, lb)
        x = torch.tensor(g + dt_bias[None], dtype=torch.float64)
        sp = torch.nn.functional.softplus(x, beta=1.0, threshold=1e6)
        ref = torch.clamp(-torch.exp(torch.tensor(A_log))[None, :, None] * sp, min=lb).numpy()
        np.testing.assert_allclose(la, ref, rtol=1e-14, atol=1e-300)


def test_gate_special_values(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 1)
    g = rng.standard_normal((10, 2, 8)) * 5
    # lower_bound = 0 clamps every log-decay to exactly 0 (alpha = 1)
    la = oracle_mod.log_decay(g, np.zeros(2), np.zeros((2, 8)), 0.0)
    assert np.all(la == 0.0)
    # a huge A_log saturates at lower_bound exactly
    la = oracle_mod.log_decay(g, np.full(2, 60.0), np.zeros((2, 8)), -7.25)
    assert np.all(la == -7.25)
    # softplus(0) = log 2 with A_log = 0, no clamp
    la = oracle_mod.log_decay(np.zeros((1, 1, 1)), np.zeros(1), np.zeros((1, 1)), -100.0)
    assert la.item() == pytest.approx(-np.log(2.0), rel=1e-15)
    # brute module's logaddexp softplus agrees with the C one
    la_b = brute.log_decay(g[3, 1], 0.3, rng.standard_normal(8) * 0 + 0.1, -5.0)
    la_c = oracle_mod.log_decay(g[3:4, 1:2], np.array([0.3]), np.full((1, 8), 0.1), -5.0)[0, 0]
    np.testing.assert_allclose(la_b, la_c, rtol=1e-14)


# ----------------------------------------------------------------------------- closed forms

def test_single_token_closed_form(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 2)
    p = rand_problem(rng, 1, 2, 8, 5)
    out, hT = run_oracle(oracle_mod, p)
    for h in range(2):
        la = brute.log_decay(p["g"][0, h], p["A_log"][h], p["dt_bias"][h], p["lower_bound"])
        k, q, v, b = p["k"][0, h], p["q"][0, h], p["v"][0, h], p["beta"][0, h]
        S0 = p["h0"][0, h]
        S1 = (np.eye(8) - b * np.outer(k, k)) @ np.diag(np.exp(la)) @ S0 + b * np.outer(k, v)
        np.testing.assert_allclose(hT[0, h], S1, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(out[0, h], p["scale"] * S1.T @ q, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_brute_force(oracle_mod, T):
    rng = np.random.default_rng(RNG_SEED + 10 + T)
    p = rand_problem(rng, T, 3, 6, 4, lower_bound=-3.0)
    out, hT = run_oracle(oracle_mod, p)
    bo, bh = brute.run(p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"], p["A_log"],
                       p["dt_bias"], p["lower_bound"], p["h0"][0])
    np.testing.assert_allclose(out, bo, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT[0], bh, rtol=1e-12, atol=1e-14)
    cf = brute.closed_form_final_state(p["k"], p["v"], p["g"], p["beta"], p["A_log"],
                                       p["dt_bias"], p["lower_bound"], p["h0"][0])
    np.testing.assert_allclose(hT[0], cf, rtol=1e-12, atol=1e-14)


def test_exact_rational(oracle_mod):
    """lower_bound = 0 forces alpha = 1; the delta rule is then rational and is
    evaluated exactly with Fractions (K = 3, V = 2, T = 4)."""
    K, V, T = 3, 2, 4
    fr = Fraction
    q = [[fr(1, 2), fr(-1, 4), fr(3, 4)], [fr(0), fr(1), fr(1, 8)], [fr(-1, 2), fr(1, 2), fr(1, 2)],
         [fr(1), fr(0), fr(-1, 4)]]
    k = [[fr(1, 2), fr(1, 2), fr(0)], [fr(-1, 4), fr(3, 4), fr(1, 2)], [fr(1), fr(0), fr(0)],
         [fr(1, 2), fr(-1, 2), fr(1, 4)]]
    v = [[fr(2), fr(-1)], [fr(1, 2), fr(3, 2)], [fr(-3, 4), fr(1, 4)], [fr(5, 4), fr(0)]]
    beta = [fr(1, 2), fr(3, 4), fr(1), fr(1, 4)]
    S0 = [[fr(1, 8), fr(0)], [fr(0), fr(-1, 4)], [fr(1, 2), fr(1, 16)]]
    scale = fr(1, 2)
    S = [row[:] for row in S0]
    exp_out = []
    for t in range(T):
        r = [sum(S[c][j] * k[t][c] for c in range(K)) for j in range(V)]
        d = [beta[t] * (v[t][j] - r[j]) for j in range(V)]
        S = [[S[c][j] + k[t][c] * d[j] for j in range(V)] for c in range(K)]
        exp_out.append([scale * sum(S[c][j] * q[t][c] for c in range(K)) for j in range(V)])

    def arr(x):
        return np.array([[float(e) for e in row] for row in x])

    p = dict(q=arr(q)[:, None], k=arr(k)[:, None], v=arr(v)[:, None],
             g=np.random.default_rng(0).standard_normal((T, 1, K)),
             beta=np.array([float(b) for b in beta])[:, None], A_log=np.zeros(1),
             dt_bias=np.zeros((1, K)), lower_bound=0.0, scale=float(scale),
             h0=arr(S0)[None, None])
    out, hT = run_oracle(oracle_mod, p)
    np.testing.assert_allclose(out[:, 0], arr(exp_out), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(hT[0, 0], arr(S), rtol=1e-14, atol=1e-15)


def test_beta_zero_is_pure_decay(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 3)
    p = rand_problem(rng, 30, 2, 8, 5)
    p["beta"] = np.zeros_like(p["beta"])
    out, hT = run_oracle(oracle_mod, p)
    for h in range(2):
        la = np.stack([brute.log_decay(p["g"][t, h], p["A_log"][h], p["dt_bias"][h],
                                       p["lower_bound"]) for t in range(30)])
        decay = np.exp(np.cumsum(la, axis=0))  # [T, K]
        for t in range(30):
            St = decay[t][:, None] * p["h0"][0, h]
            np.testing.assert_allclose(out[t, h], p["scale"] * St.T @ p["q"][t, h], rtol=1e-11,
                                       atol=1e-300)
        np.testing.assert_allclose(hT[0, h], decay[-1][:, None] * p["h0"][0, h], rtol=1e-11,
                                   atol=1e-300)


def test_state_orientation(oracle_mod):
    """S is indexed [key channel][value channel]: a one-hot S0[a][b] read with
    beta = 0, alpha = 1 returns scale * q[a] in value channel b only."""
    rng = np.random.default_rng(RNG_SEED + 4)
    K, V = 8, 6
    p = rand_problem(rng, 3, 1, K, V, lower_bound=0.0)
    p["beta"][:] = 0.0
    a, b = 5, 2
    p["h0"] = np.zeros((1, 1, K, V))
    p["h0"][0, 0, a, b] = 1.0
    out, hT = run_oracle(oracle_mod, p)
    for t in range(3):
        exp = np.zeros(V)
        exp[b] = p["scale"] * p["q"][t, 0, a]
        np.testing.assert_allclose(out[t, 0], exp, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(hT, p["h0"])


def test_orthonormal_overwrite(oracle_mod):
    """beta = 1, alpha = 1, orthonormal keys: every write stores v exactly and a
    second write to the same key replaces (not adds to) the stored value."""
    rng = np.random.default_rng(RNG_SEED + 5)
    K, V = 8, 5
    Q, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Q.T  # rows orthonormal
    vals = rng.standard_normal((6, V))
    order = [0, 1, 2, 1, 3, 0]  # key index written at each step
    T = len(order)
    p = rand_problem(rng, T, 1, K, V, lower_bound=0.0, h0=False)
    p["k"] = keys[order][:, None, :]
    p["v"] = vals[:, None, :]
    p["beta"][:] = 1.0
    # query each step with the key written two steps earlier (or the current one)
    qidx = [0, 0, 1, 1, 2, 0]
    p["q"] = keys[qidx][:, None, :]
    out, hT = run_oracle(oracle_mod, p)
    latest = {}
    for t in range(T):
        latest[order[t]] = vals[t]
        np.testing.assert_allclose(out[t, 0], p["scale"] * latest[qidx[t]], atol=1e-13)
    S_exp = sum(np.outer(keys[i], latest[i]) for i in latest)
    np.testing.assert_allclose(hT[0, 0], S_exp, atol=1e-13)


def test_strong_decay_forgets(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 6)
    p = rand_problem(rng, 12, 2, 8, 4, lower_bound=-700.0)
    p["A_log"] = np.full(2, 10.0)  # -exp(10) * softplus(.) < -700 for every channel here
    la = oracle_mod.log_decay(p["g"], p["A_log"], p["dt_bias"], p["lower_bound"])
    assert np.all(la == -700.0)
    out, hT = run_oracle(oracle_mod, p)
    for t in range(12):
        for h in range(2):
            k, q, v, b = p["k"][t, h], p["q"][t, h], p["v"][t, h], p["beta"][t, h]
            np.testing.assert_allclose(out[t, h], p["scale"] * b * (k @ q) * v, rtol=1e-12,
                                       atol=1e-14)
    np.testing.assert_allclose(hT[0, 1], p["beta"][-1, 1] * np.outer(p["k"][-1, 1], p["v"][-1, 1]),
                               rtol=1e-12, atol=1e-14)


def test_linear_attention_limits(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 7)
    T, K, V = 20, 8, 4
    p = rand_problem(rng, T, 1, K, V, lower_bound=0.0, h0=False)
    q, k, v = p["q"][:, 0], p["k"][:, 0], p["v"][:, 0]
    lin = np.stack([p["scale"] * sum((q[t] @ k[i]) * v[i] for i in range(t + 1))
                    for t in range(T)])
    # (a) erase coefficient 0, beta = 1: exactly causal linear attention
    p1 = dict(p, beta=np.ones((T, 1)))
    out, _ = run_oracle(oracle_mod, p1, erase=0.0)
    np.testing.assert_allclose(out[:, 0], lin, rtol=1e-12, atol=1e-13)
    # (b) first-order limit beta = eps: o / eps -> causal linear attention
    eps = 1e-6
    p2 = dict(p, beta=np.full((T, 1), eps))
    out, _ = run_oracle(oracle_mod, p2)
    err = np.abs(out[:, 0] / eps - lin).max() / np.abs(lin).max()
    assert err < 50 * eps * T


# ----------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("C", [1, 7, 16, 64])
def test_chunked_equals_recurrent(oracle_mod, C):
    rng = np.random.default_rng(RNG_SEED + 20 + C)
    lens = [1, 63, 64, 65, 150, 0, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    p = rand_problem(rng, int(cu[-1]), 2, 16, 12, N=len(lens))
    ro, rh = run_oracle(oracle_mod, p, cu=cu)
    co, ch = oracle_mod.chunked(p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"],
                                p["A_log"], p["dt_bias"], p["lower_bound"], p["h0"], cu, chunk=C)
    np.testing.assert_allclose(co, ro, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ch, rh, rtol=1e-10, atol=1e-12)


def test_state_passing_equals_one_call(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 8)
    T, split = 97, 41
    p = rand_problem(rng, T, 2, 12, 10)
    out, hT = run_oracle(oracle_mod, p)
    a = {key: (val[:split] if key in ("q", "k", "v", "g", "beta") else val)
         for key, val in p.items()}
    b = {key: (val[split:] if key in ("q", "k", "v", "g", "beta") else val)
         for key, val in p.items()}
    oa, ha = run_oracle(oracle_mod, a)
    b["h0"] = ha
    ob, hb = run_oracle(oracle_mod, b)
    np.testing.assert_allclose(np.concatenate([oa, ob]), out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hb, hT, rtol=1e-12, atol=1e-14)


def test_final_state_affine_in_initial_state(oracle_mod):
    """Over any run of tokens the state map is affine, S_end = M S_start + X, with
    one K x K matrix M for every value column: X is the state reached from zero and
    M the image of the identity with v = 0 (the reading the segmented path's map
    pass and scan rely on).  Two segments then compose through M and X alone."""
    rng = np.random.default_rng(RNG_SEED + 12)
    T, H, K, V, split = 70, 2, 8, 6, 29
    p = rand_problem(rng, T, H, K, V)
    p["A_log"] = np.full(H, np.log(0.02))  # weak decay: M stays O(1) over the segment
    _, h_ref = run_oracle(oracle_mod, p)

    def seg_map(sl):
        a = {key: (val[sl] if key in ("q", "k", "v", "g", "beta") else val)
             for key, val in p.items()}
        a["h0"] = None
        _, X = run_oracle(oracle_mod, a)                       # from zero
        a["v"] = np.zeros((a["v"].shape[0], H, K))
        a["h0"] = np.broadcast_to(np.eye(K), (1, H, K, K)).copy()
        _, M = run_oracle(oracle_mod, a)                       # identity, v = 0
        return M[0], X[0]

    M1, X1 = seg_map(slice(0, split))
    M2, X2 = seg_map(slice(split, T))
    for h in range(H):
        S1 = M1[h] @ p["h0"][0, h] + X1[h]
        S2 = M2[h] @ S1 + X2[h]
        np.testing.assert_allclose(S2, h_ref[0, h], rtol=1e-11, atol=1e-13)
    # M is not the identity or a pure decay: the delta term couples key channels
    off = np.abs(M1[0] - np.diag(np.diag(M1[0]))).max()
    assert off > 0.05 * np.abs(np.diag(M1[0])).max(), off


@pytest.mark.parametrize("segs", [2, 3, 5])
def test_segmented_decomposition_is_exact(oracle_mod, segs):
    """The segmented path's algorithm, done with oracle calls: split each sequence's
    64-token chunks into `segs` runs (run j starts at chunk floor(j * c / segs); short
    sequences get empty runs), find every run's map (M from v = 0 and S = I, X from
    S = 0), scan S_{j+1} = M_j S_j + X_j, rerun each run from its S_j.  Outputs and
    final states equal one call over the whole sequences."""
    rng = np.random.default_rng(RNG_SEED + 13)
    lens = [200, 1, 0, 130]
    H, K, V = 2, 8, 6
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    p = rand_problem(rng, int(cu[-1]), H, K, V, N=len(lens))
    p["A_log"] = np.full(H, np.log(0.05))  # weak decay: runs see their entering state
    out_ref, h_ref = run_oracle(oracle_mod, p, cu=cu)
    acts = ("q", "k", "v", "g", "beta")
    out = np.full_like(out_ref, np.nan)
    for n, L in enumerate(lens):
        c = -(-L // 64)
        bounds = [cu[n] + min(L, 64 * ((j * c) // segs)) for j in range(segs)] + [cu[n + 1]]
        S = p["h0"][n]                                      # [H, K, V]
        for j in range(segs):
            a, b = bounds[j], bounds[j + 1]
            run = {key: (val[a:b] if key in acts else val) for key, val in p.items()}
            run["h0"] = S[None]
            o, _ = run_oracle(oracle_mod, run)             # outputs from the entering state
            out[a:b] = o
            run["h0"] = None
            _, X = run_oracle(oracle_mod, run)
            run["v"] = np.zeros((b - a, H, K))
            run["h0"] = np.broadcast_to(np.eye(K), (1, H, K, K)).copy()
            _, M = run_oracle(oracle_mod, run)
            S = np.einsum("hik,hkv->hiv", M[0], S) + X[0]
        np.testing.assert_allclose(S, h_ref[n], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out, out_ref, rtol=1e-10, atol=1e-12)


def test_packed_equals_separate(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 9)
    lens = [5, 0, 12, 1, 70]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    p = rand_problem(rng, int(cu[-1]), 2, 8, 6, N=len(lens))
    out, hT = run_oracle(oracle_mod, p, cu=cu)
    for n, L in enumerate(lens):
        s = slice(cu[n], cu[n + 1])
        pn = {key: (val[s] if key in ("q", "k", "v", "g", "beta") else val)
              for key, val in p.items()}
        pn["h0"] = p["h0"][n:n + 1]
        on, hn = run_oracle(oracle_mod, pn)
        np.testing.assert_allclose(out[s], on, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(hT[n], hn[0], rtol=1e-13, atol=1e-15)
        if L == 0:
            np.testing.assert_array_equal(hT[n], p["h0"][n])


def test_chunk_stage_identities(oracle_mod):
    rng = np.random.default_rng(RNG_SEED + 11)
    c, K, V = 37, 16, 8
    p = rand_problem(rng, c, 1, K, V)
    la = oracle_mod.log_decay(p["g"], p["A_log"], p["dt_bias"], p["lower_bound"])[:, 0]
    st = oracle_mod.chunk_stage(p["q"][:, 0], p["k"][:, 0], p["v"][:, 0], la, p["beta"][:, 0])
    np.testing.assert_allclose(st["G"], np.cumsum(la, axis=0), rtol=1e-13)
    A = st["A"]
    assert np.all(np.triu(A) == 0.0)
    np.testing.assert_allclose(st["T"] @ (np.eye(c) + A), np.eye(c), atol=1e-10)
    Kd = p["beta"][:, 0][:, None] * p["k"][:, 0] * np.exp(st["G"])
    np.testing.assert_allclose(st["W"], st["T"] @ Kd, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(st["U"], st["T"] @ (p["beta"][:, 0][:, None] * p["v"][:, 0]),
                               rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(st["gamma"], np.exp(st["G"][-1]), rtol=1e-13)
    assert np.all(np.triu(st["Aqk"], 1) == 0.0)


def test_invalid_cu_rejected(oracle_mod):
    rng = np.random.default_rng(0)
    p = rand_problem(rng, 10, 1, 4, 4, N=2)
    with pytest.raises(ValueError):
        run_oracle(oracle_mod, p, cu=np.array([0, 7, 5], dtype=np.int64))
    with pytest.raises(ValueError):
        run_oracle(oracle_mod, p, cu=np.array([1, 5, 10], dtype=np.int64))


# ----------------------------------------------------------------------------- typed entry

def test_bf16_entry_matches_f64_entry(oracle_mod):
    from gated_delta_rule_30_gb300 import inputs
    for name in ("ref_small", "varlen_packed"):
        w = inputs.shrink(inputs.WORKLOADS[name], T=96, H=2, n_seqs=3, hi=70)
        p = inputs.make(w)
        args = (p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"], p["A_log"], p["dt_bias"],
                p["lower_bound"])
        o1, h1 = oracle_mod.recurrent(*args, initial_state=p["initial_state"],
                                      cu_seqlens=p["cu_seqlens"])
        f = [x.to(torch.float64) for x in args[:5]]
        h0 = None if p["initial_state"] is None else p["initial_state"].to(torch.float64)
        o2, h2 = oracle_mod.recurrent(*f, *args[5:], initial_state=h0, cu_seqlens=p["cu_seqlens"])
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(h1, h2)


def test_workload_generator_recipe():
    from gated_delta_rule_30_gb300 import inputs
    p = inputs.make(inputs.shrink(inputs.WORKLOADS["state_io"], n_seqs=50, H=3))
    cu = p["cu_seqlens"]
    assert cu.dtype == torch.int32 and cu[0] == 0 and int(cu[-1]) == p["T"]
    lens = cu[1:] - cu[:-1]
    assert int(lens.min()) >= 1 and int(lens.max()) <= 128
    assert p["q"].dtype == torch.bfloat16 and p["q"].shape == (1, p["T"], 3, 128)
    nq = p["q"].float().norm(dim=-1)
    assert torch.allclose(nq, torch.ones_like(nq), atol=1e-2)
    assert float(p["beta"].float().min()) > 0 and float(p["beta"].float().max()) < 1
    A = torch.exp(p["A_log"])
    assert float(A.min()) >= 1.0 and float(A.max()) < 16.0
    assert p["initial_state"].shape == (50, 3, 128, 128)
    p2 = inputs.make(inputs.shrink(inputs.WORKLOADS["state_io"], n_seqs=50, H=3))
    assert torch.equal(p["q"], p2["q"]) and torch.equal(p["cu_seqlens"], p2["cu_seqlens"])


# ----------------------------------------------------------------------------- q/k normalisation

def test_l2norm_closed_form(oracle_mod):
    """Each (token, head) row becomes x / sqrt(|x|^2 + eps): its norm is
    sqrt(s / (s + eps)) with s = |x|^2, its direction is unchanged, and a zero
    row stays zero."""
    rng = np.random.default_rng(RNG_SEED + 700)
    x = rng.standard_normal((7, 3, 16)) * rng.uniform(0.01, 5.0, (7, 3, 1))
    x[2, 1] = 0.0
    y = oracle_mod.l2norm(x)
    s = np.sum(x * x, axis=-1)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1),
                               np.sqrt(s / (s + oracle_mod.L2NORM_EPS)), rtol=1e-14, atol=0)
    cos = np.sum(x * y, -1) / np.maximum(np.linalg.norm(x, axis=-1) * np.linalg.norm(y, axis=-1),
                                         1e-300)
    np.testing.assert_allclose(cos[s > 0], 1.0, rtol=1e-14)
    assert np.all(y[2, 1] == 0.0)


def _with_norm(oracle_mod, p, **kw):
    return oracle_mod.recurrent(p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"],
                                p["A_log"], p["dt_bias"], p["lower_bound"],
                                initial_state=p["h0"], qk_l2norm=True, **kw)


def test_l2norm_is_scale_free_per_row(oracle_mod):
    """Scaling any (token, head) row of q or k by a positive factor leaves the
    normalised pass unchanged (up to the eps term, ~1e-7 here); the same scaling
    without normalisation changes it.  Catches normalising over the wrong axis."""
    rng = np.random.default_rng(RNG_SEED + 701)
    p = rand_problem(rng, 40, 3, 16, 8)
    p["q"] = rng.standard_normal((40, 3, 16))  # |row|^2 ~ 16: eps is a 6e-8 effect
    p["k"] = rng.standard_normal((40, 3, 16))
    o1, h1 = _with_norm(oracle_mod, p)
    p2 = dict(p)
    p2["q"] = p["q"] * rng.uniform(0.5, 4.0, (40, 3, 1))
    p2["k"] = p["k"] * rng.uniform(0.5, 4.0, (40, 3, 1))
    o2, h2 = _with_norm(oracle_mod, p2)
    assert np.linalg.norm(o2 - o1) <= 1e-6 * np.linalg.norm(o1)
    assert np.linalg.norm(h2 - h1) <= 1e-6 * np.linalg.norm(h1)
    o3, _ = run_oracle(oracle_mod, p2)
    assert np.abs(o3 - o1).max() > 1e-2


def test_l2norm_unit_rows_change_nothing(oracle_mod):
    """Inputs whose rows already have unit norm: the flag changes the result only
    through eps (relative 5e-7 on q and k)."""
    rng = np.random.default_rng(RNG_SEED + 702)
    p = rand_problem(rng, 50, 2, 16, 8)   # q, k unit rows
    o0, h0 = run_oracle(oracle_mod, p)
    o1, h1 = _with_norm(oracle_mod, p)
    np.testing.assert_allclose(o1, o0, rtol=1e-5, atol=1e-8)
    np.testing.assert_allclose(h1, h0, rtol=1e-5, atol=1e-8)
    assert np.abs(o1 - o0).max() > 0  # the flag did run


def test_l2norm_matches_brute_force(oracle_mod):
    """Un-normalised q, k through the flag equal the numpy brute force run on rows
    normalised in numpy."""
    rng = np.random.default_rng(RNG_SEED + 703)
    p = rand_problem(rng, 6, 2, 6, 4, lower_bound=-3.0)
    p["q"] = p["q"] * rng.uniform(0.2, 3.0, (6, 2, 1))
    p["k"] = p["k"] * rng.uniform(0.2, 3.0, (6, 2, 1))
    out, hT = _with_norm(oracle_mod, p)
    nq = p["q"] / np.sqrt(np.sum(p["q"] ** 2, -1, keepdims=True) + 1e-6)
    nk = p["k"] / np.sqrt(np.sum(p["k"] ** 2, -1, keepdims=True) + 1e-6)
    bo, bh = brute.run(nq, nk, p["v"], p["g"], p["beta"], p["scale"], p["A_log"], p["dt_bias"],
                       p["lower_bound"], p["h0"][0])
    np.testing.assert_allclose(out, bo, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT[0], bh, rtol=1e-12, atol=1e-14)
