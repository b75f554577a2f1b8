"""Independent numpy brute force for tiny KDA problems -- TEST INFRASTRUCTURE ONLY.

Written separately from ``kda_oracle.c`` (matrix form, numpy, a different
softplus evaluation) so that the test-suite can pin the C oracle against it.
For each head it builds the explicit K x K transition matrix of every token,

    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t),   alpha_t = exp(la_t),

and propagates S_t = M_t S_{t-1} + beta_t k_t v_t^T, o_t = scale S_t^T q_t
(reading of "Flashkda Delta Attention", section "Core Kernel API": recurrent
state updates of delta attention; the gate form is the reading stated in
``kda_oracle.c``).  ``closed_form_final_state`` evaluates the same final state
through products of the transition matrices instead of a running state.
Intended for T <= 8 and small K, V.
"""
from __future__ import annotations

import numpy as np


def log_decay(g, A_log_h, dt_bias_h, lower_bound):
    """la = max(-exp(A_log) softplus(g + dt_bias), lower_bound), softplus via logaddexp."""
    x = np.asarray(g, dtype=np.float64) + np.asarray(dt_bias_h, dtype=np.float64)
    sp = np.logaddexp(0.0, x)
    return np.maximum(-np.exp(float(A_log_h)) * sp, float(lower_bound))


def transitions(k, beta, la):
    """Per-token K x K transition matrices for one head: k [T, K], beta [T], la [T, K]."""
    T, K = k.shape
    I = np.eye(K)
    return [(I - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(la[t])) for t in range(T)]


def run(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, h0=None):
    """One sequence.  q, k, g: [T, H, K]; v: [T, H, V]; beta: [T, H]; h0: [H, K, V].

    Returns (out [T, H, V], final state [H, K, V]).
    """
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T, H, K = q.shape
    V = v.shape[-1]
    out = np.zeros((T, H, V))
    hT = np.zeros((H, K, V))
    for h in range(H):
        S = np.zeros((K, V)) if h0 is None else np.array(h0[h], dtype=np.float64)
        la = np.stack([log_decay(g[t, h], A_log[h], dt_bias[h], lower_bound) for t in range(T)]) \
            if T else np.zeros((0, K))
        Ms = transitions(k[:, h], beta[:, h], la)
        for t in range(T):
            S = Ms[t] @ S + beta[t, h] * np.outer(k[t, h], v[t, h])
            out[t, h] = scale * (S.T @ q[t, h])
        hT[h] = S
    return out, hT


def closed_form_final_state(k, v, g, beta, A_log, dt_bias, lower_bound, h0=None):
    """S_T = Phi_{T,0} S_0 + sum_t Phi_{T,t} beta_t k_t v_t^T with Phi_{T,t} = M_T ... M_{t+1}."""
    k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (k, v, g, beta))
    T, H, K = k.shape
    V = v.shape[-1]
    hT = np.zeros((H, K, V))
    for h in range(H):
        la = np.stack([log_decay(g[t, h], A_log[h], dt_bias[h], lower_bound) for t in range(T)])
        Ms = transitions(k[:, h], beta[:, h], la)
        S = np.zeros((K, V))
        for t in range(T):
            Phi = np.eye(K)
            for s in range(t + 1, T):
                Phi = Ms[s] @ Phi
            S += Phi @ (beta[t, h] * np.outer(k[t, h], v[t, h]))
        if h0 is not None:
            Phi = np.eye(K)
            for s in range(T):
                Phi = Ms[s] @ Phi
            S += Phi @ np.asarray(h0[h], dtype=np.float64)
        hT[h] = S
    return hT
