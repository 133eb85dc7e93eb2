"""kda_chunk_prefill_no_alloc: the chunked prefill with its records in the library's fixed
device scratch instead of a caller workspace, for callers that cannot allocate device
memory. Checked through the C ABI against kda_chunk_prefill on calls in a row (the second
with other lengths and head counts, so that records the first call left in the shared
array would show if they were read; the third with heads whose units take the pairwise
path, so that their flags sit in the array too), and its size limit, which it enforces on
the host before any CUDA call.

The file name makes pytest collect it last: its first GPU call does the per-device set-up
of the scratch address, and it must pass both alone in a fresh process and after the
other GPU tests."""
import ctypes

import numpy as np
import pytest
import torch

from linear_attention_state_recurrent_gb300 import workloads as wl


@pytest.fixture(scope="module")
def kda():
    from linear_attention_state_recurrent_gb300 import build
    build.build()
    from linear_attention_state_recurrent_gb300 import kda as k
    return k


def test_no_alloc_rejects_oversize_on_the_host(kda):
    """Beyond KDA_NO_ALLOC_SCRATCH_BYTES the call fails with KDA_ERR_WORKSPACE before any
    CUDA call (no pointer below is dereferenced)."""
    fake = ctypes.c_void_p(1 << 20)
    H = 32
    chunks = kda.KDA_NO_ALLOC_SCRATCH_BYTES // (57856 * H) + 1   # one chunk too many at H = 32
    need = chunks * H * 57856 + (chunks * H + 15) // 16 * 16    # records, then their flags
    cu = np.array([0, 64 * chunks], np.int32)
    hd = kda.KdaHeads(H=H, K=128, V=128, A_log=fake.value, dt_bias=None, has_lower_bound=0,
                      lower_bound=0.0, scale=0.1, l2_eps=1e-6)
    st = kda.KdaState(pool=fake.value, num_slots=4, slot_stride=H * 128 * 128, indices=fake.value,
                      index_stride=1, null_slot=-1)
    s = kda.lib.kda_chunk_prefill_no_alloc(fake, 3 * H * 128, fake, H * 128, fake, H, fake,
                                           cu.ctypes.data_as(ctypes.c_void_p), 1, 64,
                                           ctypes.byref(hd), ctypes.byref(st), fake, H * 128,
                                           None, None)
    assert s == kda.KDA_ERR_WORKSPACE
    msg = kda.last_error()
    assert "kda_chunk_prefill_no_alloc" in msg and str(kda.KDA_NO_ALLOC_SCRATCH_BYTES) in msg
    assert str(need) in msg


def _rel_l2(a, b):
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


@pytest.mark.gpu
def test_no_alloc_matches_chunk_prefill_on_calls_in_a_row(kda):
    from tests import kda_harness as hx
    dev = "cuda:0"
    cases = [
        wl.varlen_case([200, 1, 130, 0, 64, 300], 4, 128, 128, seed=71, lower_bound=-5.0),
        wl.varlen_case([129, 65, 7], 2, 128, 128, seed=72, lower_bound=None, index_stride=4),
        wl.varlen_case([333, 64, 1], 2, 64, 64, seed=73, lower_bound=None),
    ]
    cases[2].A_log = np.array([4.0, 0.5], dtype=np.float32)   # marked units: their flags live in the scratch too
    for i, w in enumerate(cases):
        assert 0 < kda.kda_chunk_prefill_workspace_bytes(torch.from_numpy(w.cu_seqlens), w.H, w.K, w.V) \
            <= kda.KDA_NO_ALLOC_SCRATCH_BYTES
        ref = hx.DeviceWorkload(w, dev)    # kda_chunk_prefill with its own workspace
        got = hx.DeviceWorkload(w, dev)    # kda_chunk_prefill_no_alloc
        out_ref = hx.run_gpu(ref, kda)
        out = torch.empty(w.N, w.H * w.V, dtype=torch.bfloat16, device=dev)
        kda.kda_chunk_prefill_no_alloc(got.mixed_qkv, got.raw_g, got.raw_beta, got.A_log,
                                       got.dt_bias, w.lower_bound, got.pool_view(),
                                       got.indices_view(), got.cu, torch.from_numpy(w.cu_seqlens),
                                       out, scale=w.scale, l2_eps=w.eps, null_slot=w.null_slot,
                                       err_flags=got.err)
        torch.cuda.synchronize()
        label = f"call {i + 1}"
        a = hx.bf16_to_f64(out)
        b = hx.bf16_to_f64(out_ref)
        assert np.all(np.isfinite(a)), label
        assert _rel_l2(a, b) <= hx.REL_L2, label
        assert float(np.abs(a - b).max(initial=0.0)) <= hx.MAX_ABS, label
        pa = got.pool_flat.cpu().numpy().astype(np.float64)
        pb = ref.pool_flat.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(pa)), label
        assert _rel_l2(pa, pb) <= hx.REL_L2, label
        assert int(got.err.item()) == int(ref.err.item()) == 0, label


@pytest.mark.gpu
def test_no_alloc_at_its_largest_size_equals_the_workspace_call(kda):
    """The largest call the scratch holds at H = 32 (36 chunks x 32 heads = 1,152 of its
    1,159 chunk-heads; the last sequences ragged): the same kernels as kda_chunk_prefill
    with a caller workspace, so outputs, states and error word are bit-identical."""
    from tests import kda_harness as hx
    dev = "cuda:0"
    w = wl.varlen_case([1000, 1024, 130, 5], 32, 128, 128, seed=74, lower_bound=-5.0)
    assert wl.num_chunks([1000, 1024, 130, 5]) == 36
    nb = kda.kda_chunk_prefill_workspace_bytes(torch.from_numpy(w.cu_seqlens), w.H, w.K, w.V)
    assert nb <= kda.KDA_NO_ALLOC_SCRATCH_BYTES < nb + 57856 * w.H   # one more chunk would not fit
    ref = hx.DeviceWorkload(w, dev)
    got = hx.DeviceWorkload(w, dev)
    out_ref = hx.run_gpu(ref, kda)
    out = torch.empty(w.N, w.H * w.V, dtype=torch.bfloat16, device=dev)
    kda.kda_chunk_prefill_no_alloc(got.mixed_qkv, got.raw_g, got.raw_beta, got.A_log,
                                   got.dt_bias, w.lower_bound, got.pool_view(),
                                   got.indices_view(), got.cu, torch.from_numpy(w.cu_seqlens),
                                   out, scale=w.scale, l2_eps=w.eps, null_slot=w.null_slot,
                                   err_flags=got.err)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))
    assert torch.equal(got.pool_flat, ref.pool_flat)
    assert int(got.err.item()) == int(ref.err.item()) == 0
