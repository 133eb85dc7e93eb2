"""Pins of the fused layer-tail oracle (short causal conv + gated RMSNorm around the
recurrence), CPU only. Each pin is independent of the oracle's own loops: a library
correlation, an activation identity, closed forms of the norm, and invariances."""
import numpy as np
import pytest

from linear_attention_state_recurrent_gb300 import workloads as wl
from oracle import kda_oracle as ko
from oracle import layer_tail as lt


def test_silu_identities():
    x = np.linspace(-30, 30, 601)
    # x sigmoid(x) - (-x) sigmoid(-x) = x, SiLU(0) = 0, SiLU(x) -> x and -> 0 at the ends
    np.testing.assert_allclose(lt.silu(x) - lt.silu(-x), x, rtol=0, atol=1e-12)
    assert lt.silu(np.array([0.0]))[0] == 0.0
    assert abs(lt.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    assert abs(lt.silu(np.array([-40.0]))[0]) < 1e-15


@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_conv_matches_numpy_correlate(W):
    rng = np.random.default_rng(W)
    T, C = 7, 5
    x = rng.standard_normal((T, C))
    wt = rng.standard_normal((C, W))
    b = rng.standard_normal(C)
    st = rng.standard_normal((W - 1, C))
    y, act, new = lt.short_conv(x, wt, b, st)
    hist = np.concatenate([st, x])
    for ch in range(C):
        np.testing.assert_allclose(y[:, ch], np.correlate(hist[:, ch], wt[ch], "valid") + b[ch],
                                   rtol=0, atol=1e-12)
    np.testing.assert_array_equal(new, hist[T:])


def test_conv_one_hot_taps_shift_the_history():
    """A one-hot weight at tap w returns the input W-1-w steps back (state rows before the
    first token): the tap order and the history order."""
    T, C, W = 5, 3, 4
    x = np.arange(T * C, dtype=np.float64).reshape(T, C) + 1
    st = -np.arange((W - 1) * C, dtype=np.float64).reshape(W - 1, C) - 1
    for w in range(W):
        wt = np.zeros((C, W))
        wt[:, w] = 1.0
        y, _, _ = lt.short_conv(x, wt, None, st)
        lag = W - 1 - w
        for t in range(T):
            exp = x[t - lag] if t - lag >= 0 else st[W - 1 + t - lag]
            np.testing.assert_array_equal(y[t], exp)


def test_conv_split_invariance():
    """T tokens in one call == T calls of one token with the state carried."""
    rng = np.random.default_rng(3)
    T, C, W = 6, 4, 4
    x, wt, b = rng.standard_normal((T, C)), rng.standard_normal((C, W)), rng.standard_normal(C)
    st = rng.standard_normal((W - 1, C))
    _, a_all, s_all = lt.short_conv(x, wt, b, st)
    s = st
    for t in range(T):
        _, a, s = lt.short_conv(x[t:t + 1], wt, b, s)
        np.testing.assert_allclose(a[0], a_all[t], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(s, s_all)


def test_gated_rmsnorm_closed_forms():
    rng = np.random.default_rng(4)
    N, H, V = 3, 2, 8
    o = rng.standard_normal((N, H * V))
    eps = 1e-3
    one = np.ones(V)
    big = np.full((N, H * V), np.inf)
    out = lt.gated_rmsnorm(o, big, one, eps, V).reshape(N, H, V)
    ms = np.mean(o.reshape(N, H, V) ** 2, axis=2)
    # gate -> +inf (sigmoid 1), unit weight: mean square of the result = ms / (ms + eps)
    np.testing.assert_allclose(np.mean(out ** 2, axis=2), ms / (ms + eps), rtol=1e-12)
    # gate = 0 halves it; weight scales column j; eps = 0 makes it scale invariant
    half = lt.gated_rmsnorm(o, np.zeros_like(o), one, eps, V).reshape(N, H, V)
    np.testing.assert_allclose(half, out / 2, rtol=1e-12)
    wv = np.arange(1, V + 1, dtype=np.float64)
    np.testing.assert_allclose(lt.gated_rmsnorm(o, big, wv, eps, V).reshape(N, H, V), out * wv, rtol=1e-12)
    np.testing.assert_allclose(lt.gated_rmsnorm(7.5 * o, big, one, 0.0, V),
                               lt.gated_rmsnorm(o, big, one, 0.0, V), rtol=1e-12)


def test_fused_without_conv_or_norm_is_the_plain_call():
    w = wl.with_layer_tail(wl.decode_case(5, 2, 16, 8, seed=1, num_slots=12), seed=2,
                           conv_width=None, norm=False)
    a, b = lt.run_fused(w), ko.run(w)
    np.testing.assert_array_equal(a.out, b.out)
    np.testing.assert_array_equal(a.final_states, b.final_states)
    s = wl.with_layer_tail(wl.spec_verify(num_reqs=3, T=4, H=2, K=8, V=8, num_slots=16,
                                          num_padding=1), seed=3, conv_width=None, norm=False)
    a, b = lt.run_fused(s), ko.run(s)
    np.testing.assert_array_equal(a.out, b.out)


def test_fused_conv_decode_chain_equals_spec():
    """T fused decodes, conv and KDA state carried through the pools, == one fused
    spec-verify over the T tokens (conv history and recurrence both continue)."""
    T, H, K, V = 4, 2, 8, 8
    s = wl.with_layer_tail(wl.spec_verify(num_reqs=2, T=T, H=H, K=K, V=V, num_slots=8,
                                          num_padding=0), seed=5, conv_width=4, norm=True)
    ref = lt.run_fused(s)
    pool, cpool = s.pool.copy(), s.conv_pool.copy()
    C = 2 * H * K + H * V
    outs = []
    for t in range(T):
        rows = [r * T + t for r in range(2)]
        d = wl.Workload(**{**s.__dict__, "kind": "decode", "tokens_per_req": 1,
                           "mixed_qkv": s.mixed_qkv[rows], "raw_g": s.raw_g[rows],
                           "raw_beta": s.raw_beta[rows], "out_gate": s.out_gate[rows],
                           "pool": pool, "conv_pool": cpool})
        r = lt.run_fused(d)
        outs.append(r.out)
        pool = pool.copy()
        cpool = cpool.copy()
        for e, sl in enumerate(r.slots):
            pool[sl, : H * K * V] = r.final_states[e].reshape(-1).astype(np.float32)
            bits = (r.conv_states[e].astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            cpool[sl, : 3 * C] = bits.reshape(-1)
    got = np.stack(outs, 1).reshape(2 * T, -1)
    np.testing.assert_allclose(got, ref.out, rtol=0, atol=2e-6 * np.abs(ref.out).max())
    # the conv state after T tokens is exactly the last W-1 raw inputs
    x = s.mixed_qkv.reshape(2, T, -1)[:, :, :C]
    np.testing.assert_array_equal(cpool[s.indices()[0], : 3 * C].reshape(3, C), x[0, 1:])


def test_fused_slot_rules():
    w = wl.with_layer_tail(wl.decode_case(4, 1, 8, 8, seed=6, num_slots=6), seed=7)
    w.index_buf = np.array([2, -1, 6, 0], np.int32)
    w.null_slot = 0
    r = lt.run_fused(w)
    assert r.err_flags == ko.ERR_SLOT_OUT_OF_RANGE
    assert list(r.writes) == [True, False, False, False]
    assert np.all(r.out[2] == 0)
    # a negative slot convolves over a zero history
    C = 3 * 8
    wt = lt._bf16(w.conv_weight).reshape(C, 4)
    x = lt._bf16(w.mixed_qkv)[1, :C]
    y = wt[:, 3] * x + lt._bf16(w.conv_bias)
    np.testing.assert_allclose(r.conv_states[1][-1], x)
    assert np.all(r.conv_states[1][:2] == 0)
    assert np.isfinite(y).all()
