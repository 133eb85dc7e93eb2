"""Second, independent oracle for tiny cases (TEST INFRASTRUCTURE ONLY).

Plain float64 numpy that writes the KDA transition out as explicit matrices,
S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T and
o_t = S_t^T q_t (the gated delta rule the Kimi-K3 pages name as the "KDA
recurrence"; PR #60683, section Purpose), with the gate written with numpy's
logaddexp rather than the C oracle's softplus. It uses none of the C oracle's
update-by-parts algebra, so agreement between the two pins that algebra.
Meant for K, V <= 8 and a handful of tokens.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def run_sequence(q, k, v, raw_g, raw_beta, A_log_h, dt_bias_h, lower_bound, scale, eps, S0):
    """One head of one sequence. q, k: [T, K]; v: [T, V]; raw_g: [T, K]; raw_beta: [T];
    A_log_h: scalar; dt_bias_h: [K]; S0: [K, V]. Returns (o [T, V], S_T [K, V])."""
    T, K = q.shape
    S = np.array(S0, dtype=np.float64)
    outs = np.zeros((T, v.shape[1]))
    for t in range(T):
        x = raw_g[t] + dt_bias_h
        if lower_bound is None:
            g = -np.exp(A_log_h) * np.logaddexp(0.0, x)
        else:
            g = lower_bound * (0.5 * (1.0 + np.tanh(0.5 * np.exp(A_log_h) * x)))
        alpha = np.exp(g)
        beta = 0.5 * (1.0 + np.tanh(0.5 * raw_beta[t]))
        kn = k[t] / np.linalg.norm(np.append(k[t], np.sqrt(eps)))
        qn = scale * q[t] / np.linalg.norm(np.append(q[t], np.sqrt(eps)))
        transition = (np.eye(K) - beta * np.outer(kn, kn)) @ np.diag(alpha)
        S = transition @ S + beta * np.outer(kn, v[t])
        outs[t] = S.T @ qn
    return outs, S


def run_workload(w, entry_slots=None):
    """All heads of all entries of a small `Workload`; returns (out [N, H*V], states [E, H, K, V])."""
    H, K, V = w.H, w.K, w.V
    qkv = bf16_to_f64(w.mixed_qkv)
    rg = bf16_to_f64(w.raw_g)
    rb = bf16_to_f64(w.raw_beta)
    dt = np.zeros(H * K) if w.dt_bias is None else np.asarray(w.dt_bias, dtype=np.float64)
    slots = w.indices() if entry_slots is None else entry_slots
    bounds = w.seq_bounds()
    out = np.zeros((w.N, H * V))
    states = np.zeros((len(bounds), H, K, V))
    for e, (b0, b1) in enumerate(bounds):
        s = int(slots[e])
        for h in range(H):
            S0 = np.zeros((K, V)) if s < 0 else \
                w.pool[s, h * K * V:(h + 1) * K * V].reshape(K, V).astype(np.float64)
            q = qkv[b0:b1, h * K:(h + 1) * K]
            k = qkv[b0:b1, H * K + h * K:H * K + (h + 1) * K]
            v = qkv[b0:b1, 2 * H * K + h * V:2 * H * K + (h + 1) * V]
            o, S = run_sequence(q, k, v, rg[b0:b1, h * K:(h + 1) * K], rb[b0:b1, h],
                                float(w.A_log[h]), dt[h * K:(h + 1) * K], w.lower_bound,
                                w.scale, w.eps, S0)
            out[b0:b1, h * V:(h + 1) * V] = o
            states[e, h] = S
    return out, states
