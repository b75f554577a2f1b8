"""Pins of the oracle's reverse mode (``oracle.recurrent_bwd``), CPU only.

The backward pass is checked against the forward oracle itself, which the
pins of ``test_oracle.py`` tie to closed forms and a brute force: central
finite differences of L = <dout, out> + <dfinal, final_state> along random
directions for every input, an element-by-element finite-difference Jacobian
on a tiny case, and closed forms where a branch of the recurrence switches off
(beta = 0; every channel clamped at lower_bound).
"""
import numpy as np
import pytest

RNG_SEED = 4321


def problem(rng, lens, H, K, V, lower_bound=-3.0, A_range=(1.0, 4.0)):
    T = int(sum(lens))
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V))
    g = rng.standard_normal((T, H, K))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    N = len(lens)
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=np.log(rng.uniform(*A_range, H)),
                dt_bias=0.3 * rng.standard_normal((H, K)), h0=0.1 * rng.standard_normal((N, H, K, V)),
                cu=cu, scale=K ** -0.5, lb=lower_bound,
                dout=rng.standard_normal((T, H, V)), dhT=rng.standard_normal((N, H, K, V)))


NAMES = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "A_log": "dA_log",
         "dt_bias": "ddt_bias", "h0": "dh0"}


def loss(oracle_mod, p, **over):
    x = dict(p)
    x.update(over)
    out, hT = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                                   x["A_log"], x["dt_bias"], x["lb"], initial_state=x["h0"],
                                   cu_seqlens=x["cu"])
    return float(np.sum(out * x["dout"]) + np.sum(hT * x["dhT"]))


def grads(oracle_mod, p):
    return oracle_mod.recurrent_bwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"],
                                    p["A_log"], p["dt_bias"], p["lb"], p["dout"],
                                    initial_state=p["h0"], dfinal_state=p["dhT"],
                                    cu_seqlens=p["cu"])


@pytest.mark.parametrize("lb", [-3.0, -0.6])
def test_directional_derivatives(oracle_mod, lb):
    """<grad, D> equals the central difference of the forward oracle along a random
    direction D, for all eight inputs; packed sequences including an empty one.
    lb = -0.6 clamps about half of the channels (their gate gradient is zero)."""
    rng = np.random.default_rng(RNG_SEED + int(-lb * 10))
    p = problem(rng, [7, 0, 12, 1], H=2, K=8, V=6, lower_bound=lb)
    G = grads(oracle_mod, p)
    pre = -np.exp(p["A_log"])[None, :, None] * np.logaddexp(0.0, p["g"] + p["dt_bias"][None])
    frac = np.mean(pre < lb)
    assert (frac > 0.2) if lb > -1 else True
    for name, gname in NAMES.items():
        D = rng.standard_normal(np.shape(p[name]))
        eps = 1e-6
        fd = (loss(oracle_mod, p, **{name: p[name] + eps * D})
              - loss(oracle_mod, p, **{name: p[name] - eps * D})) / (2 * eps)
        an = float(np.sum(G[gname] * D))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def test_jacobian_elementwise_tiny(oracle_mod):
    """Every element of every gradient on a 2-token, 2-channel problem by central
    differences (catches a transposed or misplaced index that a random direction
    could average away)."""
    rng = np.random.default_rng(RNG_SEED + 1)
    p = problem(rng, [2, 1], H=1, K=2, V=2, lower_bound=-2.0)
    G = grads(oracle_mod, p)
    eps = 1e-6
    for name, gname in NAMES.items():
        base = np.array(p[name], dtype=np.float64)
        for idx in np.ndindex(base.shape):
            e = np.zeros_like(base)
            e[idx] = 1.0
            fd = (loss(oracle_mod, p, **{name: base + eps * e})
                  - loss(oracle_mod, p, **{name: base - eps * e})) / (2 * eps)
            assert abs(fd - G[gname][idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd,
                                                                         G[gname][idx])


def test_beta_zero_closed_form(oracle_mod):
    """beta = 0: the state only decays, S_t = prod_{s<=t} Diag(alpha_s) S_0, so the keys
    and values get no gradient, dq_t = scale S_t dout_t, and
    dh0 = sum_t scale prod Diag(alpha) q_t dout_t^T + prod_all Diag(alpha) dhT."""
    rng = np.random.default_rng(RNG_SEED + 2)
    p = problem(rng, [9], H=1, K=5, V=4)
    p["beta"] = np.zeros_like(p["beta"])
    G = grads(oracle_mod, p)
    assert np.all(G["dk"] == 0.0) and np.all(G["dv"] == 0.0)
    la = np.maximum(-np.exp(p["A_log"][0]) * np.logaddexp(0.0, p["g"][:, 0] + p["dt_bias"][0]),
                    p["lb"])                                    # [T, K]
    cum = np.exp(np.cumsum(la, axis=0))                         # prod_{s<=t} alpha_s
    S0 = p["h0"][0, 0]
    for t in range(9):
        St = cum[t][:, None] * S0
        np.testing.assert_allclose(G["dq"][t, 0], p["scale"] * St @ p["dout"][t, 0],
                                   rtol=1e-12, atol=1e-14)
    dh0 = cum[-1][:, None] * p["dhT"][0, 0]
    for t in range(9):
        dh0 = dh0 + p["scale"] * cum[t][:, None] * np.outer(p["q"][t, 0], p["dout"][t, 0])
    np.testing.assert_allclose(G["dh0"][0, 0], dh0, rtol=1e-12, atol=1e-14)


def test_all_clamped_gate_has_no_gradient(oracle_mod):
    """exp(A_log) so large that every channel sits at lower_bound: the decay no longer
    depends on g, dt_bias or A_log, so their gradients are exactly zero."""
    rng = np.random.default_rng(RNG_SEED + 3)
    p = problem(rng, [6, 5], H=2, K=4, V=3, lower_bound=-1.0, A_range=(1e6, 2e6))
    G = grads(oracle_mod, p)
    assert np.all(G["dg"] == 0.0) and np.all(G["ddt_bias"] == 0.0)
    assert np.all(G["dA_log"] == 0.0)
    assert np.abs(G["dq"]).max() > 0 and np.abs(G["dk"]).max() > 0


def loss_qkn(oracle_mod, p, **over):
    x = dict(p)
    x.update(over)
    out, hT = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                                   x["A_log"], x["dt_bias"], x["lb"], initial_state=x["h0"],
                                   cu_seqlens=x["cu"], qk_l2norm=True)
    return float(np.sum(out * x["dout"]) + np.sum(hT * x["dhT"]))


def test_qk_l2norm_directional_derivatives(oracle_mod):
    """With the in-kernel q/k normalisation, <grad, D> equals the central difference
    of the forward oracle run with qk_l2norm=True, for all eight inputs; q and k are
    drawn with row norms far from 1, so the normalisation's Jacobian matters."""
    rng = np.random.default_rng(RNG_SEED + 7)
    p = problem(rng, [6, 0, 9], H=2, K=8, V=5, lower_bound=-3.0)
    p["q"] = p["q"] * rng.uniform(0.2, 5.0, size=p["q"].shape[:-1] + (1,))
    p["k"] = p["k"] * rng.uniform(0.2, 5.0, size=p["k"].shape[:-1] + (1,))
    G = oracle_mod.recurrent_bwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["scale"],
                                 p["A_log"], p["dt_bias"], p["lb"], p["dout"],
                                 initial_state=p["h0"], dfinal_state=p["dhT"],
                                 cu_seqlens=p["cu"], qk_l2norm=True)
    for name, gname in NAMES.items():
        D = rng.standard_normal(np.shape(p[name]))
        eps = 1e-6
        fd = (loss_qkn(oracle_mod, p, **{name: p[name] + eps * D})
              - loss_qkn(oracle_mod, p, **{name: p[name] - eps * D})) / (2 * eps)
        an = float(np.sum(G[gname] * D))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def test_l2norm_bwd_radial_component(oracle_mod):
    """x / sqrt(|x|^2 + eps) changes along x only through eps: for any dxhat,
    x . dx = (xhat . dxhat) eps / (|x|^2 + eps), and the tangential part of dx is
    the tangential part of dxhat divided by n."""
    rng = np.random.default_rng(RNG_SEED + 8)
    x = rng.standard_normal((7, 3, 16)) * rng.uniform(0.01, 10.0, size=(7, 3, 1))
    dxh = rng.standard_normal((7, 3, 16))
    eps = oracle_mod.L2NORM_EPS
    dx = oracle_mod.l2norm_bwd(x, dxh)
    nn = np.sum(x * x, axis=-1)
    n = np.sqrt(nn + eps)
    xh = x / n[..., None]
    np.testing.assert_allclose(np.sum(x * dx, axis=-1),
                               np.sum(xh * dxh, axis=-1) * eps / (nn + eps), rtol=1e-9, atol=1e-15)
    u = x / np.sqrt(nn)[..., None]
    tan = lambda y: y - u * np.sum(u * y, axis=-1, keepdims=True)
    np.testing.assert_allclose(tan(dx), tan(dxh) / n[..., None], rtol=1e-10, atol=1e-13)


@pytest.mark.parametrize("mistake", ["radial term dropped", "not divided by n", "sign of the radial term"])
def test_qk_l2norm_pin_catches_planted_mistakes(oracle_mod, monkeypatch, mistake):
    """Each plausible slip in the normalisation's chain rule, planted in the oracle's
    l2norm_bwd, makes the directional-derivative pin above fail."""
    eps = oracle_mod.L2NORM_EPS

    def wrong(x, dxhat, eps=eps):
        a = np.asarray(x, dtype=np.float64)
        d = np.asarray(dxhat, dtype=np.float64).reshape(a.shape)
        n = np.sqrt(np.sum(a * a, axis=-1, keepdims=True) + eps)
        xh = a / n
        radial = xh * np.sum(xh * d, axis=-1, keepdims=True)
        if mistake == "radial term dropped":
            return d / n
        if mistake == "not divided by n":
            return d - radial
        return (d + radial) / n

    monkeypatch.setattr(oracle_mod, "l2norm_bwd", wrong)
    with pytest.raises(AssertionError):
        test_qk_l2norm_directional_derivatives(oracle_mod)
