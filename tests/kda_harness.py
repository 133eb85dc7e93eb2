"""Helpers for the GPU parity tests: upload a Workload, run one library call through
the C ABI (via the ctypes binding), and compare with the fp64 oracle.

Tolerances (the bar stated for this path): relative L2 <= 2e-3 and max-abs <= 1e-2
on the bf16 outputs against the exact fp64 oracle, relative L2 <= 2e-3 on the
updated fp32 states, no NaN/Inf anywhere, untouched pool slots byte-identical.
For the fp32 recurrent kernels a tighter element-wise bound also holds: every
output is within one bf16 ulp of the exact value (fp32 arithmetic carries ~1e-6
relative error, far below bf16's 2^-8 spacing), plus a small absolute slack for
outputs that are the difference of nearly equal terms.
"""
from __future__ import annotations

import numpy as np
import torch

from linear_attention_state_recurrent_gb300.workloads import (  # noqa: F401
    DeviceWorkload, bf16_tensor, bf16_to_f64, run_gpu)
from oracle import kda_oracle as ko

REL_L2 = 2e-3
MAX_ABS = 1e-2


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits)."""
    return np.exp2(np.floor(np.log2(np.maximum(np.abs(x), 1e-30))) - 7)


def check(dw: DeviceWorkload, out: torch.Tensor, ref: ko.OracleResult, *, fp32_path: bool,
          rows=None, label="", max_abs=MAX_ABS, elementwise_abs=False):
    """Compares one call's GPU results with the oracle. Returns a dict of measured errors.

    elementwise_abs: the max-abs bar becomes per element max(MAX_ABS, half a bf16 ulp of
    the larger of |exact| and |result| + 1e-4 |exact|): rounding the output once to bf16
    costs up to half an ulp, which exceeds MAX_ABS only where |o| >= 4 (normalised
    outputs)."""
    w = dw.w
    torch.cuda.synchronize()
    h_lo, h_hi = ref.heads
    V = w.V
    cols = slice(h_lo * V, h_hi * V)
    got = bf16_to_f64(out)[:, cols]
    exp = ref.out[:, cols]
    if rows is not None:
        got, exp = got[rows], exp[rows]
    assert np.all(np.isfinite(got)), f"{label}: non-finite outputs"
    assert np.all(np.isfinite(exp)), f"{label}: oracle produced non-finite values"
    res = {"out_rel_l2": rel_l2(got, exp), "out_max_abs": float(np.abs(got - exp).max(initial=0.0))}
    assert res["out_rel_l2"] <= REL_L2, f"{label}: output rel L2 {res['out_rel_l2']:.3e}"
    if elementwise_abs:
        bound = np.maximum(MAX_ABS, 0.5 * bf16_ulp(np.maximum(np.abs(exp), np.abs(got))) + 1e-4 * np.abs(exp))
        over = np.abs(got - exp) > bound
        assert not over.any(), f"{label}: {over.sum()} outputs beyond max(1e-2, half a bf16 ulp)"
    else:
        assert res["out_max_abs"] <= max_abs, f"{label}: output max abs {res['out_max_abs']:.3e}"
    if fp32_path:
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exp), 1e-30))) - 7)
        slack = 1e-5 * max(np.abs(exp).max(initial=0.0), 1e-30)
        bad = np.abs(got - exp) > ulp + slack
        assert not bad.any(), f"{label}: {bad.sum()} outputs more than 1 bf16 ulp off"
    # state pool
    pool = dw.pool_flat.cpu().numpy()
    orig = w.pool
    written = set()
    HKV = w.H * w.K * w.V
    st_got, st_exp = [], []
    for e in range(len(ref.slots)):
        if ref.writes[e]:
            s = int(ref.slots[e])
            written.add(s)
            g = pool[s, :HKV].reshape(w.H, w.K, w.V)[h_lo:h_hi].astype(np.float64)
            st_got.append(g.reshape(-1))
            st_exp.append(ref.final_states[e][h_lo:h_hi].reshape(-1))
    if st_got:
        sg, se = np.concatenate(st_got), np.concatenate(st_exp)
        assert np.all(np.isfinite(sg)), f"{label}: non-finite states"
        res["state_rel_l2"] = rel_l2(sg, se)
        assert res["state_rel_l2"] <= REL_L2, f"{label}: state rel L2 {res['state_rel_l2']:.3e}"
        if fp32_path:
            assert res["state_rel_l2"] <= 1e-5, f"{label}: fp32 state rel L2 {res['state_rel_l2']:.3e}"
    untouched = np.array(sorted(set(range(w.num_slots)) - written), dtype=np.int64)
    if untouched.size:
        assert np.array_equal(pool[untouched].view(np.uint32), orig[untouched].view(np.uint32)), \
            f"{label}: an untouched slot changed"
    for s in written:  # bytes beyond H*K*V inside a written slot stay untouched too
        assert np.array_equal(pool[s, HKV:].view(np.uint32), orig[s, HKV:].view(np.uint32))
    err = int(dw.err.cpu().item())
    assert err == ref.err_flags, f"{label}: err flags {err} != {ref.err_flags}"
    return res


def check_ckpt(dw: DeviceWorkload, out: torch.Tensor, ref: ko.CheckpointResult, label=""):
    """Spec-verify with checkpoints: outputs within the bf16 tolerances and 1 bf16 ulp
    (fp32 path), every written checkpoint slot within 1e-5 relative L2 of the oracle's
    state after its token, every other slot byte-identical, the error word equal."""
    w = dw.w
    torch.cuda.synchronize()
    got = bf16_to_f64(out)
    exp = ref.out
    assert np.all(np.isfinite(got)), f"{label}: non-finite outputs"
    res = {"out_rel_l2": rel_l2(got, exp), "out_max_abs": float(np.abs(got - exp).max(initial=0.0))}
    assert res["out_rel_l2"] <= REL_L2, f"{label}: output rel L2 {res['out_rel_l2']:.3e}"
    assert res["out_max_abs"] <= MAX_ABS, f"{label}: output max abs {res['out_max_abs']:.3e}"
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exp), 1e-30))) - 7)
    slack = 1e-5 * max(np.abs(exp).max(initial=0.0), 1e-30)
    bad = np.abs(got - exp) > ulp + slack
    assert not bad.any(), f"{label}: {bad.sum()} outputs more than 1 bf16 ulp off"
    pool = dw.pool_flat.cpu().numpy()
    HKV = w.H * w.K * w.V
    written = {}
    R, T = ref.slots.shape
    for r in range(R):
        for t in range(T):
            if ref.writes[r, t]:
                written[int(ref.slots[r, t])] = ref.ckpt[r, t].reshape(-1)
    if written:
        sl = sorted(written)
        sg = pool[sl, :HKV].astype(np.float64).reshape(-1)
        se = np.concatenate([written[s] for s in sl])
        assert np.all(np.isfinite(sg)), f"{label}: non-finite checkpoints"
        res["state_rel_l2"] = rel_l2(sg, se)
        assert res["state_rel_l2"] <= 1e-5, f"{label}: checkpoint rel L2 {res['state_rel_l2']:.3e}"
    untouched = np.array(sorted(set(range(w.num_slots)) - set(written)), dtype=np.int64)
    if untouched.size:
        assert np.array_equal(pool[untouched].view(np.uint32), w.pool[untouched].view(np.uint32)), \
            f"{label}: a slot that is not a checkpoint changed"
    for s in written:
        assert np.array_equal(pool[s, HKV:].view(np.uint32), w.pool[s, HKV:].view(np.uint32))
    err = int(dw.err.cpu().item())
    assert err == ref.err_flags, f"{label}: err flags {err} != {ref.err_flags}"
    return res


def check_fused(dw: DeviceWorkload, out: torch.Tensor, ref, label=""):
    """Fused decode / spec-verify: outputs and KDA states as `check` (fp32 path), and the
    conv-state pool bit-exact: written slots hold the last W-1 inputs, every other byte
    (other slots, the spare tail of written slots) is unchanged.

    The gated RMSNorm makes the outputs O(1) (RMS 1 before weight and gate); rounding them
    once to bf16 costs up to half an ulp, which is above the 1e-2 max-abs bar where
    |o| >= 4. The max-abs bar is therefore applied per element as max(1e-2, half a bf16 ulp
    + fp32 slack); the bound of one bf16 ulp of the exact value holds unchanged."""
    res = check(dw, out, ref, fp32_path=True, label=label, elementwise_abs=True)
    w = dw.w
    if w.conv_weight is None or w.conv_width < 2:
        return res
    C = 2 * w.H * w.K + w.H * w.V
    n = (w.conv_width - 1) * C
    got = dw.conv_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    exp = w.conv_pool.copy()
    for e in range(len(ref.slots)):
        if ref.writes[e]:
            st = ref.conv_states[e].astype(np.float32).view(np.uint32) >> 16
            exp[int(ref.slots[e]), :n] = st.astype(np.uint16).reshape(-1)
    bad = np.argwhere(got != exp)
    assert bad.size == 0, f"{label}: conv state differs at {bad[:5].tolist()}"
    return res
