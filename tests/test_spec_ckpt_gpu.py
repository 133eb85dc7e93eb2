"""GPU parity of spec-verify with per-token state checkpoints against the fp64 oracle,
through the C ABI: request r reads its state from column num_accepted[r] - 1 of its
block-table row and writes the state after token t to column t (the block table of
1 + num_speculative_blocks columns, vLLM PR #51682; the padded requests' one accepted
token, PR #60683 "Refusal and steps")."""
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


def _run(kda, w, label):
    dw = hx.DeviceWorkload(w)
    out = hx.run_gpu(dw, kda)
    ref = ko.run_spec_checkpoints(w)
    return hx.check_ckpt(dw, out, ref, label=label), dw, out


@pytest.mark.parametrize("lower_bound", [None, -5.0])
def test_spec_checkpoints_16x8(kda, lower_bound):
    _run(kda, wl.spec_checkpoints(lower_bound=lower_bound), f"ckpt 16x8 lb={lower_bound}")


@pytest.mark.parametrize("num_reqs", [1, 8, 32])
@pytest.mark.parametrize("lower_bound", [-5.0, None])
@pytest.mark.parametrize("extra_cols", [0, 3])
def test_spec_checkpoints_matrix(kda, num_reqs, lower_bound, extra_cols):
    w = wl.spec_checkpoints(seed=400 + num_reqs, num_reqs=num_reqs, T=4, H=4, num_slots=160,
                            num_padding=min(1, num_reqs - 1), lower_bound=lower_bound,
                            index_stride=4 + extra_cols)
    _run(kda, w, f"ckpt n={num_reqs} lb={lower_bound} +{extra_cols}")


@pytest.mark.parametrize("T", [1, 2, 3, 8, 16])
def test_spec_checkpoints_widths(kda, T):
    w = wl.spec_checkpoints(seed=500 + T, num_reqs=5, T=T, H=2, num_slots=80, num_padding=1)
    _run(kda, w, f"ckpt T={T}")


@pytest.mark.parametrize("K,V", [(64, 128), (128, 64), (32, 32), (64, 64)])
def test_spec_checkpoints_dims(kda, K, V):
    w = wl.spec_checkpoints(seed=600 + K + V, num_reqs=4, T=5, H=3, K=K, V=V, num_slots=32,
                            num_padding=1)
    _run(kda, w, f"ckpt K={K} V={V}")


def test_every_accepted_count_and_default(kda):
    T = 6
    w = wl.spec_checkpoints(seed=7, num_reqs=T, T=T, H=2, num_slots=64, num_padding=0)
    w.num_accepted = np.arange(1, T + 1, dtype=np.int32)
    _run(kda, w, "accepted 1..T")
    w.num_accepted = None                       # NULL: every request reads column 0
    _run(kda, w, "accepted NULL")


def test_checkpoints_match_prefix_spec_verify(kda):
    """Checkpoint t equals the final state of plain spec-verify over the first t+1 tokens
    from the same slot (the state a rejected draft rolls back to)."""
    T, R = 6, 4
    w = wl.spec_checkpoints(seed=8, num_reqs=R, T=T, H=4, num_slots=64, num_padding=0)
    w.num_accepted = np.ones(R, np.int32)
    _, dw, _ = _run(kda, w, "prefix base")
    ck = dw.pool_flat.cpu().numpy()
    HKV = w.H * w.K * w.V
    for t in range(T):
        rows = np.concatenate([np.arange(r * T, r * T + t + 1) for r in range(R)])
        pre = wl.Workload(**{**w.__dict__, "kind": "spec", "tokens_per_req": t + 1,
                             "mixed_qkv": w.mixed_qkv[rows], "raw_g": w.raw_g[rows],
                             "raw_beta": w.raw_beta[rows], "num_accepted": None})
        dp = hx.DeviceWorkload(pre)
        hx.run_gpu(dp, kda)
        torch.cuda.synchronize()
        got = dp.pool_flat.cpu().numpy()
        for r in range(R):
            a = ck[w.index_buf[r, t], :HKV]
            b = got[w.index_buf[r, 0], :HKV]
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-6 * np.abs(b).max())


def test_checkpoint_slot_semantics(kda):
    """Negative columns: zero read state / no write; null-slot columns: never written;
    out-of-range columns and accepted counts outside [1, T]: error bit, and a bad read
    column or count zeroes the request's outputs and writes nothing of it."""
    T = 4
    w = wl.spec_checkpoints(seed=9, num_reqs=6, T=T, H=2, num_slots=40, num_padding=0,
                            index_stride=5)
    w.index_buf = np.array([[3, -1, 40, 0, 9],
                            [-1, 5, 6, 7, 9],
                            [8, 10, 11, 12, 0],
                            [13, 14, 15, 16, 0],
                            [17, 18, 1 << 30, 19, 0],
                            [20, 21, 22, 23, 0]], np.int32)
    w.num_accepted = np.array([1, 1, 0, 5, 3, 2], np.int32)
    res, dw, out = _run(kda, w, "ckpt slot semantics")
    o = out.float().cpu()
    assert torch.all(o[2 * T:4 * T] == 0) and torch.all(o[4 * T:5 * T] == 0)
    assert int(dw.err.cpu().item()) == ko.ERR_SLOT_OUT_OF_RANGE


def test_checkpoint_rejects_bad_arguments(kda):
    w = wl.spec_checkpoints(seed=10, num_reqs=2, T=4, H=2, num_slots=16, num_padding=0)
    dw = hx.DeviceWorkload(w)
    args = (dw.mixed_qkv, dw.raw_g, dw.raw_beta, dw.A_log, dw.dt_bias, None, dw.pool_view())
    table = dw.index_buf.reshape(2, 4)
    with pytest.raises(ValueError, match="column per token"):
        kda.kda_spec_verify_checkpoints(*args, table[:, :3], 4)
    w17 = wl.spec_checkpoints(seed=10, num_reqs=1, T=17, H=1, num_slots=32, num_padding=0)
    d17 = hx.DeviceWorkload(w17)
    with pytest.raises(ValueError, match="tokens_per_req"):
        kda.kda_spec_verify_checkpoints(d17.mixed_qkv, d17.raw_g, d17.raw_beta, d17.A_log,
                                        d17.dt_bias, None, d17.pool_view(),
                                        d17.index_buf.reshape(1, 17), 17)


def test_checkpoints_graph_replay(kda):
    """Captured once in a CUDA graph, replayed: the same results each replay."""
    w = wl.spec_checkpoints(seed=11, num_reqs=8, T=4, H=4, num_slots=64, num_padding=1)
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
    ref = ko.run_spec_checkpoints(w)
    for _ in range(3):
        dw.reset_pool()
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        hx.check_ckpt(dw, out, ref, label="graph replay")
