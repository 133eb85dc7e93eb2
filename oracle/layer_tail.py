"""fp64 oracle of the two steps around the KDA recurrence in the fused layer tail
(TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the bench's CPU-baseline
leg may import this module).

The Kimi-K3 decode layer ("K1" of vLLM PR #60683 "specialized decode for Kimi-K3 on
MI355X", section Purpose, whole-layer list) runs "spec conv, KDA recurrence, gated
RMSNorm" back to back. The pages name the two steps and nothing more; the readings here:

* short causal convolution: depthwise over the 2HK+HV channels of the q|k|v row, width W
  (1..4), with the W-1 previous inputs of each channel kept per state slot (oldest first)
  in a bf16 conv-state pool addressed by the same slot index as the KDA state:
      y_t[ch] = sum_{w<W} weight[ch, w] * hist[t + w, ch] + bias[ch],
      hist    = [conv_state (W-1 rows); x_{row0} .. x_{row0+T-1}],
      x'_t    = SiLU(y_t) = y_t * sigmoid(y_t),
  after which the conv state holds the last W-1 rows of hist. The same slot rules as the
  KDA state apply (negative: zero history, no write; null slot: read, no write; out of
  range: nothing read or written).
* gated RMSNorm, per (token, head) over the V outputs:
      o'_j = o_j / sqrt(mean_j o_j^2 + eps) * weight[j] * sigmoid(gate[t, h*V + j]).

Nothing here is shared with the CUDA path.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from oracle import kda_oracle as ko


def _bf16(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    e = np.exp(x[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def silu(y: np.ndarray) -> np.ndarray:
    return y * _sigmoid(y)


def short_conv(x: np.ndarray, weight: np.ndarray, bias: np.ndarray | None, state: np.ndarray):
    """One entry's convolution. x fp64 [T, C] (the entry's raw rows), weight fp64 [C, W],
    bias fp64 [C] or None, state fp64 [W-1, C]. Returns (y [T, C] before the activation,
    SiLU(y), new state [W-1, C])."""
    T, C = x.shape
    W = weight.shape[1]
    hist = np.concatenate([state.reshape(W - 1, C), x], axis=0)
    y = np.zeros((T, C), dtype=np.float64)
    for t in range(T):
        for w in range(W):
            y[t] += weight[:, w] * hist[t + w]
    if bias is not None:
        y += bias
    return y, silu(y), hist[hist.shape[0] - (W - 1):].copy()


def gated_rmsnorm(o: np.ndarray, gate: np.ndarray, weight: np.ndarray, eps: float, V: int):
    """o fp64 [N, H*V], gate fp64 [N, H*V], weight [V]: the normalised, gated outputs."""
    N = o.shape[0]
    oh = o.reshape(N, -1, V)
    ms = np.mean(oh * oh, axis=2, keepdims=True)
    out = oh / np.sqrt(ms + eps) * np.asarray(weight, np.float64) * _sigmoid(gate.reshape(N, -1, V))
    return out.reshape(N, -1)


@dataclasses.dataclass
class FusedResult:
    out: np.ndarray            # fp64 [N, H*V]
    final_states: np.ndarray   # fp64 [E, H, K, V]
    conv_states: np.ndarray    # fp64 [E, W-1, C] (empty when there is no convolution)
    slots: np.ndarray
    writes: np.ndarray
    err_flags: int
    heads: tuple


def run_fused(w, nthreads: int = 0) -> FusedResult:
    """The fused decode / spec-verify call on a Workload made by `with_layer_tail`."""
    lib = ko._load()
    H, K, V = w.H, w.K, w.V
    C = 2 * H * K + H * V
    bounds = w.seq_bounds()
    slots = w.indices().astype(np.int64)
    E = len(bounds)
    conv = w.conv_weight is not None
    Wd = w.conv_width if conv else 1
    x = _bf16(w.mixed_qkv)[:, :C]
    qkv = x.copy()
    states = np.zeros((E, H, K, V), dtype=np.float64)
    conv_states = np.zeros((E, Wd - 1, C), dtype=np.float64)
    valid = np.ones(E, dtype=bool)
    writes = np.zeros(E, dtype=bool)
    err = 0
    wt = _bf16(w.conv_weight).reshape(C, Wd) if conv else None
    bias = _bf16(w.conv_bias) if conv and w.conv_bias is not None else None
    for e in range(E):
        s = int(slots[e])
        if s >= w.num_slots:
            valid[e] = False
            err |= ko.ERR_SLOT_OUT_OF_RANGE
            continue
        cs = np.zeros((Wd - 1, C))
        if s >= 0:
            states[e] = w.pool[s, : H * K * V].reshape(H, K, V).astype(np.float64)
            if conv:
                cs = _bf16(w.conv_pool[s, : (Wd - 1) * C]).reshape(Wd - 1, C)
            writes[e] = s != w.null_slot
        if conv:
            b0, b1 = bounds[e]
            _, act, new = short_conv(x[b0:b1], wt, bias, cs)
            qkv[b0:b1] = act
            conv_states[e] = new
    out = np.zeros((w.N, H * V), dtype=np.float64)
    vidx = np.nonzero(valid)[0]
    if len(vidx):
        rb = np.array([bounds[e][0] for e in vidx], dtype=np.int64)
        re = np.array([bounds[e][1] for e in vidx], dtype=np.int64)
        sub = np.ascontiguousarray(states[vidx])
        q64 = np.ascontiguousarray(qkv)
        rg = np.ascontiguousarray(w.raw_g, dtype=np.uint16)
        rbeta = np.ascontiguousarray(w.raw_beta, dtype=np.uint16)
        A_log = np.ascontiguousarray(w.A_log, dtype=np.float32)
        dt = None if w.dt_bias is None else np.ascontiguousarray(w.dt_bias, dtype=np.float32)
        lb = w.lower_bound
        _call_f64in(lib, q64, rg, rbeta, rb, re, len(vidx), H, K, V, A_log, dt, lb, w.scale,
                    w.eps, sub, out, nthreads)
        states[vidx] = sub
    if w.norm_weight is not None:
        out = gated_rmsnorm(out, _bf16(w.out_gate)[:, : H * V], w.norm_weight, w.norm_eps, V)
    for e in range(E):
        if not valid[e]:
            b0, b1 = bounds[e]
            out[b0:b1] = 0.0
    return FusedResult(out=out, final_states=states, conv_states=conv_states, slots=slots,
                       writes=writes & valid, err_flags=err, heads=(0, H))


def _call_f64in(lib, q64, rg, rbeta, rb, re, n, H, K, V, A_log, dt, lb, scale, eps, states,
                out, nthreads):
    import ctypes
    P, I64, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    f = lib.kda_oracle_recurrent_f64in
    f.argtypes = [P, I64, P, I64, P, I64, P, P, I64, I, I, I, P, P, I, D, D, D, P, P, I64, I]
    f.restype = None
    p = ko._ptr
    f(p(q64), q64.shape[1], p(rg), rg.shape[1], p(rbeta), rbeta.shape[1], p(rb), p(re), n, H, K,
      V, p(A_log), p(dt), int(lb is not None), float(lb or 0.0), float(scale), float(eps),
      p(states), p(out), H * V, int(nthreads))
