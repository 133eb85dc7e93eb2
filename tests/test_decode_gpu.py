"""GPU parity of the gate, packed decode and spec-verify calls against the fp64 oracle,
run through the C ABI. The parameter matrix is the one the vLLM packed-decode test
runs for every implementation of the call (PR #51682: num_seqs in {1, 8, 32},
lower_bound in {-5.0, None}, state index stride in {1, 8}); here every entry point
runs it."""
import time

import numpy as np
import pytest
import torch

from linear_attention_state_recurrent_gb300 import workloads as wl
from oracle import kda_oracle as ko
from tests import kda_harness as hx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    from linear_attention_state_recurrent_gb300 import kda as k
    return k


def _run_and_check(kda, w, label, fp32_path=True, heads=None):
    dw = hx.DeviceWorkload(w)
    out = hx.run_gpu(dw, kda)
    ref = ko.run(w, heads=heads)
    return hx.check(dw, out, ref, fp32_path=fp32_path, label=label)


def test_gate_matches_oracle(kda):
    for lb in (None, -5.0):
        w = wl.decode_case(37, 4, 128, 128, seed=4, lower_bound=lb)
        dw = hx.DeviceWorkload(w)
        g, b = kda.kda_gate(dw.raw_g, dw.raw_beta, dw.A_log, dw.dt_bias, lb)
        gr, br = ko.gate(w.raw_g, w.raw_beta, w.A_log, w.dt_bias, lb, w.H, w.K)
        np.testing.assert_allclose(g.cpu().numpy(), gr, rtol=2e-6, atol=1e-6)
        np.testing.assert_allclose(b.cpu().numpy(), br, rtol=2e-6, atol=1e-7)
        assert torch.all(g <= 0)


def test_gate_odd_K(kda):
    w = wl.decode_case(5, 3, 32, 32, seed=8)
    H, K = 3, 20
    raw_g = w.raw_g[:, :H * K].copy()
    dw = hx.DeviceWorkload(w)
    rg = hx.bf16_tensor(raw_g, "cuda:0")
    dt = torch.from_numpy(w.dt_bias[:H * K].copy()).cuda()
    g, b = kda.kda_gate(rg, dw.raw_beta, dw.A_log, dt, None, K=K)
    gr, _ = ko.gate(raw_g, w.raw_beta, w.A_log, w.dt_bias[:H * K], None, H, K)
    np.testing.assert_allclose(g.cpu().numpy(), gr, rtol=2e-6, atol=1e-6)


def test_tiny_decode(kda):
    r = _run_and_check(kda, wl.tiny_decode(), "tiny")
    assert r["out_rel_l2"] < 2e-3


@pytest.mark.parametrize("num_seqs", [1, 8, 32])
@pytest.mark.parametrize("lower_bound", [-5.0, None])
@pytest.mark.parametrize("stride", [1, 8])
def test_packed_decode_matrix(kda, num_seqs, lower_bound, stride):
    w = wl.decode_case(num_seqs, 4, 128, 128, seed=100 + num_seqs + stride, lower_bound=lower_bound,
                       index_stride=stride, num_slots=2 * num_seqs * stride + 3)
    _run_and_check(kda, w, f"decode n={num_seqs} lb={lower_bound} s={stride}")


@pytest.mark.parametrize("K,V", [(32, 32), (32, 128), (64, 64), (128, 32), (64, 128)])
def test_packed_decode_dims(kda, K, V):
    w = wl.decode_case(9, 3, K, V, seed=K + V, index_stride=2, extra_slot_stride=8)
    _run_and_check(kda, w, f"decode K={K} V={V}")


@pytest.mark.parametrize("lower_bound", [-5.0, None])
def test_serving_decode(kda, lower_bound):
    w = wl.serving_decode(lower_bound)
    _run_and_check(kda, w, f"serving decode lb={lower_bound}")


def test_serving_decode_strided_equals_contiguous(kda):
    w = wl.serving_decode(-5.0)
    dw = hx.DeviceWorkload(w)
    a = hx.run_gpu(dw, kda).clone()
    pa = dw.pool_flat.clone()
    dw.reset_pool()
    idx = dw.indices_view().contiguous()
    b, _ = kda.kda_packed_decode(dw.mixed_qkv, dw.raw_g, dw.raw_beta, dw.A_log, dw.dt_bias,
                                 -5.0, dw.pool_view(), idx, scale=w.scale)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(pa.view(torch.int32), dw.pool_flat.view(torch.int32))


def test_spec_verify(kda):
    _run_and_check(kda, wl.spec_verify(), "spec verify 16x8")


@pytest.mark.parametrize("num_reqs", [1, 8, 32])
@pytest.mark.parametrize("lower_bound", [-5.0, None])
@pytest.mark.parametrize("stride", [1, 8])
def test_spec_verify_matrix(kda, num_reqs, lower_bound, stride):
    w = wl.spec_verify(seed=200 + num_reqs, num_reqs=num_reqs, T=4, H=4, num_slots=64,
                       num_padding=min(1, num_reqs - 1), lower_bound=lower_bound,
                       index_stride=stride)
    _run_and_check(kda, w, f"spec n={num_reqs} lb={lower_bound} s={stride}")


@pytest.mark.parametrize("T", [1, 2, 3, 8, 17])
def test_spec_verify_widths(kda, T):
    w = wl.spec_verify(seed=300 + T, num_reqs=5, T=T, H=2, num_slots=16, num_padding=1)
    _run_and_check(kda, w, f"spec T={T}")


def test_slot_semantics(kda):
    """Out-of-range slots set the error bit and write zero outputs; negative slots start
    from zero and write nothing; the null slot is read but never written."""
    w = wl.decode_case(6, 2, 64, 64, seed=9, num_slots=10)
    w.index_buf = np.array([3, -1, 10, 7, 1 << 30, 7], np.int32)
    w.null_slot = 7
    dw = hx.DeviceWorkload(w)
    out = hx.run_gpu(dw, kda)
    ref = ko.run(w)
    assert ref.err_flags == ko.ERR_SLOT_OUT_OF_RANGE
    hx.check(dw, out, ref, fp32_path=True, label="slot semantics")
    o = out.float().cpu()
    assert torch.all(o[2] == 0) and torch.all(o[4] == 0)


def test_rejects_bad_arguments(kda):
    w = wl.decode_case(4, 2, 64, 64, seed=1)
    dw = hx.DeviceWorkload(w)
    args = (dw.mixed_qkv, dw.raw_g, dw.raw_beta, dw.A_log, dw.dt_bias, None, dw.pool_view())
    with pytest.raises(ValueError, match="one-dimensional"):
        kda.kda_packed_decode(*args, dw.index_buf.reshape(-1, 1))
    with pytest.raises(ValueError):
        kda.kda_packed_decode(*args, dw.indices_view(), null_slot=w.num_slots)
    short_out = torch.empty(4, 100, dtype=torch.bfloat16, device="cuda:0")[:, :99]
    with pytest.raises(ValueError, match="ld_out"):
        kda.kda_packed_decode(*args, dw.indices_view(), out=short_out)
    with pytest.raises(ValueError, match="index_stride"):
        kda.kda_packed_decode(*args, dw.index_buf.reshape(-1)[:1].expand(4))
    assert int(dw.err.item()) == 0


def test_repeat_launches_bit_identical(kda):
    """300 launches of the same decode from the same state give identical bits (no races)."""
    w = wl.decode_case(32, 8, 128, 128, seed=77, index_stride=8)
    dw = hx.DeviceWorkload(w)
    first = hx.run_gpu(dw, kda).clone()
    first_pool = dw.pool_flat.clone()
    ref_pool = torch.from_numpy(w.pool).cuda()
    out = torch.empty_like(first)
    for _ in range(300):
        dw.pool_flat.copy_(ref_pool)
        hx.run_gpu(dw, kda, out=out)
        assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    assert torch.equal(dw.pool_flat.view(torch.int32), first_pool.view(torch.int32))


def test_cuda_graph_replay(kda):
    """A captured decode replays bit-identically (no host sync or allocation inside)."""
    w = wl.decode_case(16, 4, 128, 128, seed=78, index_stride=4)
    dw = hx.DeviceWorkload(w)
    eager = hx.run_gpu(dw, kda).clone()
    eager_pool = dw.pool_flat.clone()
    ref_pool = torch.from_numpy(w.pool).cuda()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    dw.pool_flat.copy_(ref_pool)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hx.run_gpu(dw, kda, out=out, stream=s)
    for _ in range(20):
        dw.pool_flat.copy_(ref_pool)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
        assert torch.equal(dw.pool_flat.view(torch.int32), eager_pool.view(torch.int32))


@pytest.mark.parametrize("T", [1, 3, 8])
def test_spec_verify_unaligned_rows(kda, T):
    """Rows whose pitch is not a multiple of 4 elements take the V-split spec kernel (the
    one-CTA-per-head kernel needs 8-byte channel loads); both give the same results."""
    w = wl.spec_verify(seed=700 + T, num_reqs=6, T=T, H=3, num_slots=16, num_padding=1)
    pad = np.zeros((w.N, 1), np.uint16)
    w.mixed_qkv = np.concatenate([w.mixed_qkv, pad], axis=1)
    w.raw_g = np.concatenate([w.raw_g, pad], axis=1)
    _run_and_check(kda, w, f"spec unaligned T={T}")


@pytest.mark.parametrize("K,V", [(32, 32), (32, 128), (64, 64), (128, 32), (128, 64)])
@pytest.mark.parametrize("T", [3, 8])
def test_spec_verify_dims(kda, K, V, T):
    w = wl.spec_verify(seed=800 + K + V + T, num_reqs=5, T=T, H=3, K=K, V=V, num_slots=16,
                       num_padding=1, index_stride=2)
    _run_and_check(kda, w, f"spec K={K} V={V} T={T}")


def test_spec_verify_without_dt_bias_scale_one(kda):
    w = wl.spec_verify(seed=810, num_reqs=4, T=5, H=2, num_slots=16, num_padding=1)
    w.dt_bias = None
    w.scale = 1.0
    _run_and_check(kda, w, "spec no dt_bias, scale 1")


def test_spec_verify_slot_semantics(kda):
    """Spec-verify requests on out-of-range slots (error bit, zero outputs), a negative
    slot (zero state, no write) and the null slot (read, never written)."""
    w = wl.spec_verify(seed=820, num_reqs=6, T=4, H=2, num_slots=10, num_padding=0)
    w.index_buf = np.array([[3], [-1], [10], [7], [1 << 30], [5]], np.int32)
    w.null_slot = 7
    dw = hx.DeviceWorkload(w)
    out = hx.run_gpu(dw, kda)
    ref = ko.run(w)
    assert ref.err_flags == ko.ERR_SLOT_OUT_OF_RANGE
    hx.check(dw, out, ref, fp32_path=True, label="spec slot semantics")
    o = out.float().cpu()
    assert torch.all(o[8:12] == 0) and torch.all(o[16:20] == 0)


def test_bounded_wait_gives_up_and_context_stays_usable(kda):
    """The tensor-core kernels' bounded mbarrier wait, made to run out (nothing arrives):
    the kernel sets the timeout bit and returns; later calls on the context still work."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    kda.kda_selftest_bounded_wait(err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda.KDA_ERRFLAG_TIMEOUT
    assert time.perf_counter() - t0 >= 1.5
    _run_and_check(kda, wl.tiny_decode(), "decode after a timed-out wait")


def test_back_to_back_dependent_decodes(kda):
    """T decode calls in a row on the same slots, nothing launched between them: each one
    reads the state the previous one wrote (the decode grid may launch while its
    predecessor finishes, and must wait for it before its first read). Together they equal
    spec-verify over the same T tokens."""
    w = wl.spec_verify(seed=81, num_reqs=12, T=6, H=4, num_padding=0, lower_bound=-5.0)
    dw = hx.DeviceWorkload(w)
    R, T, H, K, V = w.num_entries, w.tokens_per_req, w.H, w.K, w.V
    C = dw.mixed_qkv.shape[1]
    out = torch.zeros(w.N, H * V, dtype=torch.bfloat16, device=dw.device)
    qkv3, g3, b3 = dw.mixed_qkv.view(R, T, C), dw.raw_g.view(R, T, -1), dw.raw_beta.view(R, T, -1)
    out3 = out.view(R, T, H * V)
    for t in range(T):
        kda.kda_packed_decode(qkv3[:, t], g3[:, t], b3[:, t], dw.A_log, dw.dt_bias, w.lower_bound,
                              dw.pool_view(), dw.indices_view(), scale=w.scale, l2_eps=w.eps,
                              null_slot=w.null_slot, out=out3[:, t], err_flags=dw.err)
    ref = ko.run(w)
    hx.check(dw, out, ref, fp32_path=True, label="back-to-back decodes")
