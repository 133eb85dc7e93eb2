"""Pins for the fp64 oracle (CPU only).

The pages print no worked numbers for the KDA kernels, so the oracle is pinned
by what the mathematics fixes: a hand-derived example, closed forms of the gate
and of special cases of the update (pure decay at beta = 0, the textbook delta
rule write at alpha = 1, beta = 1, unit keys, the plain linear-attention readout
at alpha = 1, beta = 0), a contraction bound, an independent numpy brute force
that writes the transition as explicit matrices, and chunked == sequential.
"""
import math
import os

import numpy as np
import pytest

from linear_attention_state_recurrent_gb300 import workloads as wl
from oracle import brute
from oracle import kda_oracle as ko

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

NEG_INF = 0xFF80
POS_INF = 0x7F80


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _bf(x):
    return wl.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _hand_workload(lower_bound=None):
    gd = _read_golden("kda_hand_2x2.txt")
    K, V = int(gd["K"][0]), int(gd["V"][0])
    q = np.array(gd["q"]).reshape(2, K)
    k = np.array(gd["k"]).reshape(2, K)
    v = np.array(gd["v"]).reshape(2, V)
    mixed = _bf(np.concatenate([q, k, v], axis=1))
    pool = np.array(gd["S0"], dtype=np.float32).reshape(1, K * V)
    cu = np.array([0, 2], dtype=np.int32)
    w = wl.Workload(name="hand", kind="prefill", H=1, K=K, V=V, mixed_qkv=mixed,
                    raw_g=_bf(np.array(gd["raw_g"]).reshape(2, K)),
                    raw_beta=_bf(np.array(gd["raw_beta"]).reshape(2, 1)),
                    A_log=np.zeros(1, np.float32), dt_bias=np.zeros(K, np.float32),
                    lower_bound=lower_bound, scale=1.0, eps=0.0, pool=pool,
                    index_buf=np.array([0], np.int32), index_stride=1, num_entries=1,
                    cu_seqlens=cu)
    return w, gd


@pytest.mark.parametrize("use_lb", [False, True])
@pytest.mark.parametrize("chunked", [False, True])
def test_hand_derived_example(use_lb, chunked):
    gd = _read_golden("kda_hand_2x2.txt")
    lb = gd["lower_bound_equivalent"][0] if use_lb else None
    w, gd = _hand_workload(lb)
    r = ko.run(w, chunked=chunked, chunk_size=2)
    np.testing.assert_allclose(r.out.reshape(-1), gd["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r.final_states.reshape(-1), gd["S_final"], rtol=0, atol=1e-14)
    ob, sb = brute.run_workload(w)
    np.testing.assert_allclose(ob.reshape(-1), gd["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(sb.reshape(-1), gd["S_final"], rtol=0, atol=1e-14)


def test_gate_closed_forms():
    H, K = 2, 4
    # row 0: x = 0; row 1: x = -inf; row 2: x = 3 (bf16-exact); row 3: x = -3
    raw_g = np.zeros((4, H * K), np.uint16)
    raw_g[1] = NEG_INF
    raw_g[2] = _bf(np.full(H * K, 3.0))
    raw_g[3] = _bf(np.full(H * K, -3.0))
    raw_beta = np.array([[0, 0], [NEG_INF, POS_INF], _bf([2.0, -2.0]), _bf([0.5, 1.0])], np.uint16)
    A_log = np.array([0.0, math.log(2.0)], np.float32)
    g, b = ko.gate(raw_g, raw_beta, A_log, None, None, H, K)
    a = np.exp(np.array(A_log, np.float64))
    sp = lambda x: math.log1p(math.exp(x)) if x < 30 else x  # noqa: E731
    for h in range(H):
        sl = slice(h * K, (h + 1) * K)
        np.testing.assert_allclose(g[0, sl], -a[h] * math.log(2.0), rtol=1e-15)
        assert np.all(g[1, sl] == 0.0)
        np.testing.assert_allclose(g[2, sl], -a[h] * sp(3.0), rtol=1e-15)
        np.testing.assert_allclose(g[3, sl], -a[h] * sp(-3.0), rtol=1e-15)
    np.testing.assert_allclose(b[0], [0.5, 0.5], rtol=0)
    np.testing.assert_allclose(b[1], [0.0, 1.0], rtol=0)
    np.testing.assert_allclose(b[2], [1 / (1 + math.exp(-2.0)), 1 / (1 + math.exp(2.0))], rtol=1e-15)
    # lower bound: g = L * sigmoid(e^{A_log} x)
    L = -5.0
    g2, _ = ko.gate(raw_g, raw_beta, A_log, None, L, H, K)
    for h in range(H):
        sl = slice(h * K, (h + 1) * K)
        np.testing.assert_allclose(g2[0, sl], L / 2, rtol=1e-15)
        assert np.all(g2[1, sl] == 0.0)
        np.testing.assert_allclose(g2[2, sl], L / (1 + math.exp(-a[h] * 3.0)), rtol=1e-14)
    # dt_bias shifts x per channel: raw_g = -dt_bias gives x = 0 exactly when both are bf16-exact
    dt = np.array([0.5, -0.25, 1.0, 2.0] * H, np.float32)
    raw = np.tile(_bf(-dt), (1, 1))
    g3, _ = ko.gate(raw, raw_beta[:1], A_log, dt, None, H, K)
    for h in range(H):
        np.testing.assert_allclose(g3[0, h * K:(h + 1) * K], -a[h] * math.log(2.0), rtol=1e-15)


def test_gate_ranges_random():
    rng = np.random.default_rng(7)
    H, K, N = 4, 16, 64
    raw_g = _bf(rng.standard_normal((N, H * K)) * 4)
    raw_beta = _bf(rng.standard_normal((N, H)))
    A_log = rng.uniform(-1, 1, H).astype(np.float32)
    dt = (rng.standard_normal(H * K) * 0.1).astype(np.float32)
    g, b = ko.gate(raw_g, raw_beta, A_log, dt, None, H, K)
    assert np.all(g <= 0) and np.all(np.isfinite(g))
    assert np.all((b > 0) & (b < 1))
    g2, _ = ko.gate(raw_g, raw_beta, A_log, dt, -5.0, H, K)
    assert np.all((g2 <= 0) & (g2 >= -5.0))


def _varlen(lengths, H, K, V, seed, **kw):
    return wl.varlen_case(lengths, H, K, V, seed=seed, **kw)


def test_beta_zero_is_pure_decay():
    w = _varlen([5, 1, 9], 2, 8, 6, seed=11, pool_std=0.5)
    w.raw_beta[:] = NEG_INF
    r = ko.run(w)
    g, b = ko.gate(w.raw_g, w.raw_beta, w.A_log, w.dt_bias, None, w.H, w.K)
    assert np.all(b == 0)
    qkv = brute.bf16_to_f64(w.mixed_qkv)
    for e, (b0, b1) in enumerate(w.seq_bounds()):
        s = int(w.indices()[e])
        for h in range(w.H):
            S0 = w.pool[s, h * 48:(h + 1) * 48].reshape(8, 6).astype(np.float64)
            cum = np.cumsum(g[b0:b1, h * 8:(h + 1) * 8], axis=0)
            exp_final = np.exp(cum[-1])[:, None] * S0
            np.testing.assert_allclose(r.final_states[e, h], exp_final, rtol=1e-13, atol=1e-300)
            for t in range(b1 - b0):
                q = qkv[b0 + t, h * 8:(h + 1) * 8]
                qh = w.scale * q / math.sqrt(q @ q + w.eps)
                o = (np.exp(cum[t])[:, None] * S0).T @ qh
                np.testing.assert_allclose(r.out[b0 + t, h * 6:(h + 1) * 6], o, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("chunked", [False, True])
def test_delta_rule_write_recovers_value(chunked):
    """alpha = 1, beta = 1, |k^| = 1: after token t, S_t^T k^_t = v_t; with q = k and
    scale 1 the output is v_t exactly (up to rounding)."""
    w = _varlen([7, 3], 2, 8, 8, seed=5, eps=0.0, scale=1.0)
    w.raw_g[:] = NEG_INF
    w.raw_beta[:] = POS_INF
    HK = w.H * w.K
    w.mixed_qkv[:, :HK] = w.mixed_qkv[:, HK:2 * HK]
    r = ko.run(w, chunked=chunked, chunk_size=4)
    v = brute.bf16_to_f64(w.mixed_qkv[:, 2 * HK:])
    np.testing.assert_allclose(r.out, v, rtol=0, atol=1e-12)


def test_alpha_one_beta_zero_is_plain_readout():
    w = _varlen([4], 3, 8, 4, seed=9, pool_std=1.0)
    w.raw_g[:] = NEG_INF
    w.raw_beta[:] = NEG_INF
    r = ko.run(w)
    qkv = brute.bf16_to_f64(w.mixed_qkv)
    s = int(w.indices()[0])
    for h in range(3):
        S0 = w.pool[s, h * 32:(h + 1) * 32].reshape(8, 4).astype(np.float64)
        np.testing.assert_array_equal(r.final_states[0, h], S0)
        for t in range(4):
            q = qkv[t, h * 8:(h + 1) * 8]
            qh = w.scale * q / math.sqrt(q @ q + w.eps)
            np.testing.assert_allclose(r.out[t, h * 4:(h + 1) * 4], S0.T @ qh, rtol=1e-13)


def test_contraction_bound():
    """0 < beta < 1, alpha <= 1, |k^| <= 1  =>  |S_t|_F <= |S_{t-1}|_F + beta |v_t|."""
    w = _varlen([1] * 12, 2, 8, 8, seed=13, pool_std=2.0)
    # chain one-token calls through one state
    g, beta = ko.gate(w.raw_g, w.raw_beta, w.A_log, w.dt_bias, None, w.H, w.K)
    v = brute.bf16_to_f64(w.mixed_qkv[:, 2 * w.H * w.K:])
    pool = w.pool.copy()
    slot = int(w.indices()[0])
    for t in range(12):
        step = wl.Workload(**{**w.__dict__, "mixed_qkv": w.mixed_qkv[t:t + 1],
                              "raw_g": w.raw_g[t:t + 1], "raw_beta": w.raw_beta[t:t + 1],
                              "pool": pool, "cu_seqlens": np.array([0, 1], np.int32),
                              "num_entries": 1, "index_buf": np.array([slot], np.int32)})
        r = ko.run(step)
        for h in range(w.H):
            before = np.linalg.norm(pool[slot, h * 64:(h + 1) * 64].astype(np.float64))
            after = np.linalg.norm(r.final_states[0, h])
            assert after <= before + beta[t, h] * np.linalg.norm(v[t, h * 8:(h + 1) * 8]) + 1e-12
        pool[slot, :w.H * 64] = r.final_states[0].reshape(-1)


@pytest.mark.parametrize("K,V", [(4, 4), (8, 4), (32, 32)])
@pytest.mark.parametrize("C", [4, 16, 64])
@pytest.mark.parametrize("lb", [None, -5.0])
def test_chunked_equals_sequential(K, V, C, lb):
    lengths = [1, 2, 5, 17, 64, 65, 130] if K < 32 else [1, 63, 64, 65, 200]
    w = _varlen(lengths, 2, K, V, seed=K * 100 + C, lower_bound=lb, pool_std=0.3)
    a = ko.run(w)
    b = ko.run(w, chunked=True, chunk_size=C)
    scale_o = np.abs(a.out).max()
    np.testing.assert_allclose(b.out, a.out, rtol=0, atol=1e-10 * scale_o)
    np.testing.assert_allclose(b.final_states, a.final_states, rtol=0,
                               atol=1e-10 * np.abs(a.final_states).max())


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_agrees(seed):
    rng = np.random.default_rng(seed)
    K = int(rng.integers(1, 5))
    V = int(rng.integers(1, 5))
    lengths = [int(x) for x in rng.integers(1, 4, size=3)]
    lb = None if seed % 2 else -3.0
    w = _varlen(lengths, 2, K, V, seed=seed, lower_bound=lb, pool_std=0.7,
                index_stride=1 + seed % 3)
    a = ko.run(w)
    ob, sb = brute.run_workload(w)
    np.testing.assert_allclose(a.out, ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a.final_states, sb, rtol=1e-12, atol=1e-13)


def test_brute_force_decode_and_spec_kinds():
    w = wl.decode_case(5, 2, 4, 4, seed=3, index_stride=8, num_slots=64)
    a = ko.run(w)
    ob, sb = brute.run_workload(w)
    np.testing.assert_allclose(a.out, ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a.final_states, sb, rtol=1e-12, atol=1e-13)
    s = wl.spec_verify(num_reqs=4, T=3, H=2, K=4, V=4, num_slots=16, num_padding=1)
    a = ko.run(s)
    ob, sb = brute.run_workload(s)
    np.testing.assert_allclose(a.out, ob, rtol=1e-12, atol=1e-13)


def test_strided_and_contiguous_indices_agree_bitwise():
    w = wl.decode_case(8, 2, 8, 8, seed=21, index_stride=8, num_slots=128)
    a = ko.run(w)
    contiguous = wl.Workload(**{**w.__dict__, "index_buf": w.indices().copy(), "index_stride": 1})
    b = ko.run(contiguous)
    assert np.array_equal(a.out, b.out)
    assert np.array_equal(a.final_states, b.final_states)
    assert np.array_equal(a.slots, b.slots)


def test_slot_semantics():
    w = wl.decode_case(4, 1, 4, 4, seed=2, num_slots=8)
    w.index_buf = np.array([3, -1, 9, 5], np.int32)
    w.null_slot = 5
    r = ko.run(w)
    assert r.err_flags == ko.ERR_SLOT_OUT_OF_RANGE
    assert list(r.writes) == [True, False, False, False]
    assert np.all(r.out[2] == 0.0)
    exp = r.expected_pool(w.pool)
    untouched = [s for s in range(8) if s != 3]
    assert np.array_equal(exp[untouched], w.pool[untouched].astype(np.float64))
    # negative slot: zero initial state
    zero = wl.Workload(**{**w.__dict__, "pool": np.zeros_like(w.pool)})
    rz = ko.run(zero, slots=np.array([0, 0, 0, 0]))
    assert np.array_equal(r.out[1], rz.out[1])


def test_split_prefill_equals_one_shot():
    w = _varlen([150], 2, 16, 16, seed=31)
    one = ko.run(w)
    a = wl.Workload(**{**w.__dict__, "cu_seqlens": np.array([0, 70], np.int32),
                       "mixed_qkv": w.mixed_qkv[:70], "raw_g": w.raw_g[:70],
                       "raw_beta": w.raw_beta[:70]})
    ra = ko.run(a)
    pool2 = w.pool.copy()
    slot = int(w.indices()[0])
    pool2[slot] = ra.final_states[0].reshape(-1)
    b = wl.Workload(**{**w.__dict__, "cu_seqlens": np.array([0, 80], np.int32),
                       "mixed_qkv": w.mixed_qkv[70:], "raw_g": w.raw_g[70:],
                       "raw_beta": w.raw_beta[70:], "pool": pool2})
    rb = ko.run(b)
    # the carried state passes through the fp32 pool once, hence the fp32-level tolerance
    np.testing.assert_allclose(ra.out, one.out[:70], rtol=0, atol=0)
    np.testing.assert_allclose(rb.out, one.out[70:], rtol=0, atol=1e-6 * np.abs(one.out).max())
    np.testing.assert_allclose(rb.final_states, one.final_states, rtol=0,
                               atol=1e-6 * np.abs(one.final_states).max())


def test_spec_verify_equals_sequential_decodes():
    s = wl.spec_verify(num_reqs=3, T=4, H=2, K=8, V=8, num_slots=16, num_padding=1)
    r = ko.run(s)
    pool = s.pool.copy()
    slots = s.indices()
    outs = np.zeros_like(r.out)
    for t in range(4):
        rows = np.array([q * 4 + t for q in range(3)])
        d = wl.Workload(**{**s.__dict__, "kind": "decode", "mixed_qkv": s.mixed_qkv[rows],
                           "raw_g": s.raw_g[rows], "raw_beta": s.raw_beta[rows], "pool": pool,
                           "index_buf": slots.copy(), "index_stride": 1, "null_slot": -1})
        rd = ko.run(d)
        outs[rows] = rd.out
        for e in range(3):
            # the padding request's state also advances token by token inside the
            # spec-verify call (it is only never written back), so thread it here too
            pool[slots[e], :2 * 64] = rd.final_states[e].reshape(-1)
    # the decode chain passes its state through the fp32 pool between tokens
    tol = 2e-6 * np.abs(r.out).max()
    np.testing.assert_allclose(outs, r.out, rtol=0, atol=tol)
    first = np.array([0, 4, 8])
    np.testing.assert_array_equal(outs[first], r.out[first])
    assert not r.writes[2]


def test_mixed_batch_equals_parts():
    lengths = [1, 1, 1, 37, 80]
    w = _varlen(lengths, 2, 8, 8, seed=41, num_decodes=3, kind="mixed", index_stride=4)
    r = ko.run(w)
    dec = ko.run(w, bounds=w.seq_bounds()[:3], slots=w.indices()[:3])
    pre = ko.run(w, bounds=w.seq_bounds()[3:], slots=w.indices()[3:])
    np.testing.assert_array_equal(r.out[:3], dec.out[:3])
    np.testing.assert_array_equal(r.out[3:], pre.out[3:])
    np.testing.assert_array_equal(r.final_states[:3], dec.final_states)
    np.testing.assert_array_equal(r.final_states[3:], pre.final_states)


def test_length_one_prefill_equals_decode():
    w = _varlen([1, 1, 1], 2, 16, 16, seed=51)
    a = ko.run(w, chunked=True, chunk_size=64)
    d = wl.Workload(**{**w.__dict__, "kind": "decode"})
    b = ko.run(d)
    np.testing.assert_allclose(a.out, b.out, rtol=1e-13, atol=1e-15)
    assert np.all(np.isfinite(a.out))


def test_prefill_lengths_seed1():
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(1)
    assert torch.randint(512, 8193, (8,), generator=g).tolist() == wl.PREFILL_LENGTHS_SEED1
    assert sum(wl.PREFILL_LENGTHS_SEED1) == 33494
    assert wl.num_chunks(wl.PREFILL_LENGTHS_SEED1) == 527


def test_planted_mistakes_are_caught():
    """Each plausible slip in the brute-force transition changes the hand-derived answer."""
    gd = _read_golden("kda_hand_2x2.txt")
    q = np.array(gd["q"]).reshape(2, 2)
    k = q.copy()
    v = np.array(gd["v"]).reshape(2, 2)
    S0 = np.array(gd["S0"]).reshape(2, 2)
    a, b = 0.5, 0.5

    def step(S, t, transpose=False, sign=1.0, decay_after=False):
        M = (np.eye(2) - b * np.outer(k[t], k[t]))
        Sd = np.diag([a, a]) @ (S.T if transpose else S)
        if decay_after:
            Snew = np.diag([a, a]) @ (M @ S + b * np.outer(k[t], v[t]))
        else:
            Snew = M @ Sd + sign * b * np.outer(k[t], v[t])
        return Snew, Snew.T @ q[t]

    def run(**kw):
        S, outs = S0, []
        for t in range(2):
            S, o = step(S, t, **kw)
            outs.append(o)
        return np.concatenate(outs)

    np.testing.assert_allclose(run(), gd["o"], atol=1e-15)
    for kw in ({"transpose": True}, {"sign": -1.0}, {"decay_after": True}):
        assert not np.allclose(run(**kw), gd["o"])


def test_spec_checkpoints_pinned_to_recurrence():
    """Checkpoint t equals the final state of running the first t+1 tokens alone from the
    accepted column's state (the pinned recurrence), bit-exactly; the outputs equal plain
    spec-verify's from the same initial state; writes go to columns 0..T-1."""
    s = wl.spec_checkpoints(num_reqs=3, T=5, H=2, K=8, V=8, num_slots=64, num_padding=1)
    s.num_accepted = np.array([3, 1, 1], np.int32)
    ck = ko.run_spec_checkpoints(s)
    init = np.array([s.index_buf[0, 2], s.index_buf[1, 0], 0])
    plain = ko.run(s, slots=init)
    np.testing.assert_array_equal(ck.out, plain.out)
    for t in range(5):
        part = wl.Workload(**{**s.__dict__, "tokens_per_req": t + 1,
                              "mixed_qkv": s.mixed_qkv.reshape(3, 5, -1)[:, :t + 1].reshape(3 * (t + 1), -1),
                              "raw_g": s.raw_g.reshape(3, 5, -1)[:, :t + 1].reshape(3 * (t + 1), -1),
                              "raw_beta": s.raw_beta.reshape(3, 5, -1)[:, :t + 1].reshape(3 * (t + 1), -1)})
        r = ko.run(part, slots=init)
        np.testing.assert_array_equal(ck.ckpt[:, t], r.final_states)
    assert not ck.writes[2].any()          # padding request on the null slot writes nothing
    assert ck.writes[:2].all()
    exp = ck.expected_pool(s.pool)
    np.testing.assert_array_equal(exp[s.index_buf[0, 4]], ck.ckpt[0, 4].reshape(-1))
    np.testing.assert_array_equal(exp[s.index_buf[1, 0]], ck.ckpt[1, 0].reshape(-1))


def test_spec_checkpoint_slot_rules():
    s = wl.spec_checkpoints(num_reqs=3, T=3, H=1, K=4, V=4, num_slots=16, num_padding=0,
                            index_stride=4)
    s.index_buf = np.array([[5, -1, 99, 0], [40, 1, 2, 3], [6, 7, 8, 9]], np.int32)
    s.num_accepted = np.array([1, 1, 4], np.int32)
    ck = ko.run_spec_checkpoints(s)
    assert ck.err_flags == ko.ERR_SLOT_OUT_OF_RANGE
    assert list(ck.writes[0]) == [True, False, False]
    assert not ck.writes[1].any() and not ck.writes[2].any()
    assert np.all(ck.out[3:9] == 0)
    # a negative accepted column starts from zero
    s.index_buf = np.array([[-1, 3, 4, 0], [5, 6, 7, 0], [8, 9, 10, 0]], np.int32)
    s.num_accepted = np.array([1, 2, 3], np.int32)
    ck = ko.run_spec_checkpoints(s)
    assert ck.err_flags == 0 and ck.writes[0, 0] is np.False_ and ck.writes[0, 1:].all()
    zero = wl.Workload(**{**s.__dict__, "pool": np.zeros_like(s.pool)})
    np.testing.assert_array_equal(ko.run_spec_checkpoints(zero).out[:3], ck.out[:3])
