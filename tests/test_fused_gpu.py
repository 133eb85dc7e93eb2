"""GPU parity of the fused layer tail (short causal conv -> KDA recurrence -> gated
RMSNorm; the "spec conv, KDA recurrence, gated RMSNorm" run of the Kimi-K3 decode layer,
vLLM PR #60683 section Purpose) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from linear_attention_state_recurrent_gb300 import workloads as wl
from oracle import layer_tail as lt
from tests import kda_harness as hx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    from linear_attention_state_recurrent_gb300 import kda as k
    return k


def _run(kda, w, label):
    dw = hx.DeviceWorkload(w)
    out = hx.run_gpu(dw, kda)
    ref = lt.run_fused(w)
    return hx.check_fused(dw, out, ref, label=label), dw, out


@pytest.mark.parametrize("conv", [4, None])
@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("lower_bound", [-5.0, None])
def test_fused_serving_decode(kda, conv, norm, lower_bound):
    base = wl.decode_case(128, 32, 128, 128, seed=21, lower_bound=lower_bound, index_stride=8,
                          num_slots=512, pool_std=0.05, name="serving_decode")
    w = wl.with_layer_tail(base, seed=22, conv_width=conv, norm=norm)
    _run(kda, w, f"fused decode conv={conv} norm={norm} lb={lower_bound}")


@pytest.mark.parametrize("conv", [4, None])
@pytest.mark.parametrize("norm", [True, False])
def test_fused_spec_verify_16x8(kda, conv, norm):
    w = wl.with_layer_tail(wl.spec_verify(seed=23), seed=24, conv_width=conv, norm=norm)
    _run(kda, w, f"fused spec conv={conv} norm={norm}")


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [1, 2, 3, 5, 16])
def test_fused_conv_widths_and_lengths(kda, W, T):
    w = wl.with_layer_tail(wl.spec_verify(seed=30 + T, num_reqs=5, T=T, H=3, num_slots=16,
                                          num_padding=1), seed=40 + W, conv_width=W,
                           conv_bias=(W % 2 == 0))
    _run(kda, w, f"fused W={W} T={T}")


@pytest.mark.parametrize("K,V", [(64, 128), (128, 64), (32, 32), (64, 64), (32, 128)])
def test_fused_dims(kda, K, V):
    w = wl.with_layer_tail(wl.spec_verify(seed=50 + K + V, num_reqs=4, T=3, H=3, K=K, V=V,
                                          num_slots=16, num_padding=1), seed=51)
    _run(kda, w, f"fused K={K} V={V}")
    d = wl.with_layer_tail(wl.decode_case(6, 2, K, V, seed=52, index_stride=3, num_slots=24),
                           seed=53)
    _run(kda, d, f"fused decode K={K} V={V}")


def test_fused_slot_semantics(kda):
    """Negative slot: zero state and zero conv history, nothing written; null slot: read,
    never written; out of range: error bit, zero outputs, nothing touched."""
    base = wl.decode_case(6, 2, 64, 64, seed=60, num_slots=10)
    w = wl.with_layer_tail(base, seed=61)
    w.index_buf = np.array([3, -1, 10, 7, 1 << 30, 5], np.int32)
    w.null_slot = 7
    res, dw, out = _run(kda, w, "fused slot semantics")
    o = out.float().cpu()
    assert torch.all(o[2] == 0) and torch.all(o[4] == 0)


def test_fused_decode_chain_equals_fused_spec(kda):
    """T fused decodes (conv history and state carried in the pools) give the outputs of one
    fused spec-verify over the T tokens."""
    T = 4
    s = wl.with_layer_tail(wl.spec_verify(seed=70, num_reqs=6, T=T, H=4, num_slots=16,
                                          num_padding=0), seed=71)
    ds = hx.DeviceWorkload(s)
    o_spec = hx.run_gpu(ds, kda).float().cpu()
    d = wl.Workload(**{**s.__dict__, "kind": "decode", "tokens_per_req": 1})
    dd = hx.DeviceWorkload(d)
    rows = torch.arange(6) * T
    outs = []
    for t in range(T):
        r = (rows + t).to(dd.mixed_qkv.device)
        o, _ = kda.kda_fused_decode(dd.mixed_qkv[r], dd.raw_g[r], dd.raw_beta[r], dd.A_log,
                                    dd.dt_bias, None, dd.pool_view(), dd.indices_view(),
                                    conv=(dd.conv_weight, dd.conv_bias, dd.conv_pool),
                                    norm=(dd.out_gate[r], dd.norm_weight, s.norm_eps),
                                    scale=s.scale, null_slot=s.null_slot)
        outs.append(o.float().cpu())
    got = torch.stack(outs, 1).reshape(6 * T, -1)
    torch.cuda.synchronize()
    assert torch.allclose(got, o_spec, rtol=2e-2, atol=1e-2)
    assert torch.equal(dd.conv_pool.cpu(), ds.conv_pool.cpu())
    np.testing.assert_allclose(dd.pool_flat.cpu().numpy(), ds.pool_flat.cpu().numpy(),
                               rtol=0, atol=1e-5)


def test_fused_rejects_bad_arguments(kda):
    w = wl.with_layer_tail(wl.decode_case(4, 2, 64, 64, seed=80), seed=81)
    dw = hx.DeviceWorkload(w)
    args = (dw.mixed_qkv, dw.raw_g, dw.raw_beta, dw.A_log, dw.dt_bias, None, dw.pool_view(),
            dw.indices_view())
    wide = torch.zeros(dw.conv_weight.shape[0], 5, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="conv width"):
        kda.kda_fused_decode(*args, conv=(wide, None, dw.conv_pool))
    short = dw.conv_pool[:, :10]
    with pytest.raises(ValueError, match="slot_stride"):
        kda.kda_fused_decode(*args, conv=(dw.conv_weight, None, short.contiguous()))
    with pytest.raises(ValueError, match="tokens_per_req"):
        kda.kda_fused_spec_verify(*args, 17)


def test_fused_graph_replay_and_repeat(kda):
    w = wl.with_layer_tail(wl.spec_verify(seed=90, num_reqs=8, T=4, H=4, num_slots=32,
                                          num_padding=1), seed=91)
    dw = hx.DeviceWorkload(w)
    out = torch.empty(w.N, w.H * w.V, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        hx.run_gpu(dw, kda, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hx.run_gpu(dw, kda, out=out, stream=s)
    ref = lt.run_fused(w)
    first = None
    for _ in range(3):
        dw.reset_pool()
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        hx.check_fused(dw, out, ref, label="fused graph replay")
        if first is None:
            first = out.clone()
        assert torch.equal(out, first)


def test_fused_without_dt_bias_scale_one(kda):
    base = wl.decode_case(7, 3, 128, 128, seed=95, index_stride=2, scale=1.0, with_dt_bias=False)
    _run(kda, wl.with_layer_tail(base, seed=96), "fused decode no dt_bias, scale 1")
    s = wl.spec_verify(seed=97, num_reqs=3, T=6, H=2, num_slots=16, num_padding=1)
    s.dt_bias = None
    _run(kda, wl.with_layer_tail(s, seed=98, conv_width=3), "fused spec no dt_bias")
