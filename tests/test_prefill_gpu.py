"""GPU parity of the chunked varlen prefill and the mixed decode+prefill batch against
the fp64 oracle, through the C ABI. Lengths cover one and several chunks of 64 with
ragged tails, the length-1 sequences that the chunk kernel of vLLM PR #50649 turned
into NaN, and empty sequences."""
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


def _run(kda, w, label, heads=None, nthreads=0):
    dw = hx.DeviceWorkload(w)
    out = hx.run_gpu(dw, kda)
    ref = ko.run(w, heads=heads, nthreads=nthreads)
    return hx.check(dw, out, ref, fp32_path=False, label=label)


@pytest.mark.parametrize("lower_bound", [None, -5.0])
@pytest.mark.parametrize("stride", [1, 8])
def test_prefill_ragged(kda, lower_bound, stride):
    lengths = [1, 2, 63, 64, 65, 127, 129, 300]
    w = wl.varlen_case(lengths, 2, 128, 128, seed=61 + stride, lower_bound=lower_bound,
                       index_stride=stride)
    _run(kda, w, f"prefill lb={lower_bound} s={stride}")


@pytest.mark.parametrize("num_seqs", [1, 8, 32])
def test_prefill_matrix(kda, num_seqs):
    rng = np.random.default_rng(num_seqs)
    lengths = [int(x) for x in rng.integers(1, 200, size=num_seqs)]
    for lb in (-5.0, None):
        for stride in (1, 8):
            w = wl.varlen_case(lengths, 4, 128, 128, seed=num_seqs * 10 + stride, lower_bound=lb,
                               index_stride=stride)
            _run(kda, w, f"prefill n={num_seqs} lb={lb} s={stride}")


@pytest.mark.parametrize("K,V", [(32, 32), (64, 128), (128, 64)])
def test_prefill_dims(kda, K, V):
    w = wl.varlen_case([5, 70, 130], 3, K, V, seed=K * 3 + V)
    _run(kda, w, f"prefill K={K} V={V}")


@pytest.mark.parametrize("K,V", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("lower_bound", [None, -5.0])
def test_prefill_chunked_64_wide(kda, K, V, lower_bound):
    """Heads with K or V of 64 take the tensor-core path on 128 x 128 tiles with the
    channels / columns past the data held at zero: several chunks, ragged tails, an empty
    sequence, length 1, a strided index view."""
    lengths = [1, 63, 64, 65, 0, 200, 129]
    w = wl.varlen_case(lengths, 4, K, V, seed=K + 7 * V + (0 if lower_bound is None else 1),
                       lower_bound=lower_bound, index_stride=3)
    _run(kda, w, f"prefill K={K} V={V} lb={lower_bound}")


def test_prefill_chunked_64_strong_decay(kda):
    """K = V = 64 with heads strong enough to take the pairwise diagonal path."""
    w = wl.varlen_case([40, 150, 333], 4, 64, 64, seed=19)
    w.A_log = np.array([3.0, -1.0, 4.0, 0.5], dtype=np.float32)
    _run(kda, w, "prefill K=V=64 strong decay")


def test_mixed_batch_marked_units(kda):
    """A mixed batch whose prefill heads need the pairwise diagonal path: the prep kernel's
    pass over marked units runs while the decodes wait on the side stream."""
    w = wl.varlen_case([1] * 5 + [300, 129, 64], 4, 128, 128, seed=97, index_stride=2,
                       num_decodes=5, kind="mixed")
    w.A_log = np.array([4.0, -1.0, 3.5, 0.0], dtype=np.float32)
    _run(kda, w, "mixed marked units")


def test_mixed_batch_64_wide(kda):
    w = wl.varlen_case([1] * 6 + [77, 200], 4, 64, 64, seed=95, lower_bound=-5.0, index_stride=2,
                       num_decodes=6, kind="mixed")
    _run(kda, w, "mixed K=V=64")


def test_prefill_empty_and_length_one(kda):
    w = wl.varlen_case([0, 1, 0, 1, 1], 2, 128, 128, seed=5)
    r = _run(kda, w, "empty/len1")
    assert r["out_rel_l2"] < 2e-3


def test_length_one_prefill_equals_decode(kda):
    """The pages' mixed-batch NaN came from length-1 sequences in the chunk kernel."""
    w = wl.varlen_case([1, 1, 1, 1], 4, 128, 128, seed=6)
    dw = hx.DeviceWorkload(w)
    a = hx.run_gpu(dw, kda).clone()
    pa = dw.pool_flat.clone()
    dw.reset_pool()
    d = wl.Workload(**{**w.__dict__, "kind": "decode"})
    dd = hx.DeviceWorkload(d)
    b = hx.run_gpu(dd, kda)
    assert torch.isfinite(a.float()).all()
    ref = ko.run(d)
    hx.check(dd, b, ref, fp32_path=True, label="decode side")
    np.testing.assert_allclose(a.float().cpu().numpy(), b.float().cpu().numpy(), atol=2e-2)


def test_chunked_prefill_config(kda):
    """8 sequences of the seed-1 lengths (33,494 tokens), H=32, K=V=128: every head of every
    sequence against the oracle, element by element (outputs and final states)."""
    w = wl.chunked_prefill(None)
    _run(kda, w, "chunked prefill 8 seqs", heads=(0, 32))


def test_chunked_prefill_config_lower_bound(kda):
    w = wl.chunked_prefill(-5.0)
    _run(kda, w, "chunked prefill lb", heads=(28, 32))


def test_split_prefill_resumes_from_slot(kda):
    """A prompt chunked across two calls equals one call (state carried in the slot)."""
    w = wl.varlen_case([300], 2, 128, 128, seed=8)
    dw = hx.DeviceWorkload(w)
    one = hx.run_gpu(dw, kda).float().cpu().numpy()
    pool_one = dw.pool_flat.clone()
    dw.reset_pool()
    cut = 130
    cu_a = torch.tensor([0, cut], dtype=torch.int32)
    cu_b = torch.tensor([0, 300 - cut], dtype=torch.int32)
    oa, _ = kda.kda_chunk_prefill(dw.mixed_qkv[:cut], dw.raw_g[:cut], dw.raw_beta[:cut], dw.A_log,
                                  dw.dt_bias, None, dw.pool_view(), dw.indices_view(), cu_a.cuda(),
                                  scale=w.scale)
    ob, _ = kda.kda_chunk_prefill(dw.mixed_qkv[cut:], dw.raw_g[cut:], dw.raw_beta[cut:], dw.A_log,
                                  dw.dt_bias, None, dw.pool_view(), dw.indices_view(), cu_b.cuda(),
                                  scale=w.scale)
    two = torch.cat([oa, ob]).float().cpu().numpy()
    assert hx.rel_l2(two, one) < 2e-3
    s = int(w.indices()[0])
    assert hx.rel_l2(dw.pool_flat[s].cpu().numpy(), pool_one[s].cpu().numpy()) < 2e-3


def test_mixed_batch_config(kda):
    """96 length-1 decodes + 4 prefills of 4096, index stride 4: every head of every
    sequence against the oracle, element by element."""
    w = wl.mixed_batch()
    _run(kda, w, "mixed batch", heads=(0, 32))


def test_mixed_batch_rows_after_an_offset(kda):
    """cu_seqlens starting at row 3: three leading rows that no sequence covers (filled with
    other values). The decodes read rows cu_seqlens[0] + d and the prefills their own rows;
    results equal the oracle's on the unshifted batch, and the leading output rows keep
    what they held."""
    off = 3
    lengths = [1] * 5 + [130, 64, 1, 70]
    w = wl.varlen_case(lengths, 2, 128, 128, seed=79, index_stride=2, num_decodes=5, kind="mixed")
    dw = hx.DeviceWorkload(w)
    ref = ko.run(w)

    def shifted(t):   # off rows of other values (the batch's last rows, reversed) in front
        return torch.cat([t[-off:].flip(0), t]).contiguous()
    mq, rg, rb = shifted(dw.mixed_qkv), shifted(dw.raw_g), shifted(dw.raw_beta)
    cu_h = torch.from_numpy(w.cu_seqlens + off)
    out = torch.full((w.N + off, w.H * w.V), 1.0, dtype=torch.bfloat16, device=dw.device)
    kda.kda_mixed_batch(mq, rg, rb, dw.A_log, dw.dt_bias, w.lower_bound, dw.pool_view(),
                        dw.indices_view(), cu_h.to(dw.device), w.num_decodes, cu_seqlens_host=cu_h,
                        scale=w.scale, l2_eps=w.eps, null_slot=w.null_slot, out=out,
                        err_flags=dw.err)
    torch.cuda.synchronize()
    assert torch.equal(out[:off], torch.full_like(out[:off], 1.0))
    hx.check(dw, out[off:], ref, fp32_path=False, label="mixed batch after an offset")


@pytest.mark.parametrize("lower_bound", [-5.0, None])
@pytest.mark.parametrize("stride", [1, 8])
def test_mixed_batch_matrix(kda, lower_bound, stride):
    lengths = [1] * 8 + [1, 77, 200]
    w = wl.varlen_case(lengths, 4, 128, 128, seed=90 + stride, lower_bound=lower_bound,
                       index_stride=stride, num_decodes=8, kind="mixed")
    _run(kda, w, f"mixed lb={lower_bound} s={stride}")


def test_mixed_batch_rejects_long_decode(kda):
    w = wl.varlen_case([1, 2, 5], 2, 128, 128, seed=3, num_decodes=2, kind="mixed")
    dw = hx.DeviceWorkload(w)
    with pytest.raises(ValueError, match="length"):
        hx.run_gpu(dw, kda)


@pytest.mark.parametrize("A_log", [[3.0, -1.0, 0.5, 2.5], [4.0, 4.0, 4.0, 4.0]])
def test_prefill_strong_decay(kda, A_log):
    """Heads whose channels decay by more than 40 nats within 8 rows take the pairwise
    path for the diagonal blocks; the others the tensor-core path. Both match the oracle."""
    w = wl.varlen_case([1, 40, 64, 150, 333], 4, 128, 128, seed=17)
    w.A_log = np.array(A_log, dtype=np.float32)
    _run(kda, w, f"strong decay A_log={A_log}")


def test_prefill_marked_units_over_the_grid(kda):
    """Units whose channel halves need the pairwise path are marked by the first pass and
    redone by a grid of a few CTAs per SM, each taking every G-th marked unit. Here 520
    (chunk, head) units, 5 heads of 8 marked throughout: more marked units than that grid
    has CTAs, so CTAs run several in turn, interleaved with unmarked units."""
    w = wl.varlen_case([3000, 1100, 64, 1], 8, 128, 128, seed=78)
    w.A_log = np.array([4.0, -1.0, 4.0, 0.5, 4.0, 4.0, -2.0, 3.0], dtype=np.float32)
    _run(kda, w, "marked units over the grid")


def test_prefill_more_than_1024_sequences(kda):
    """More sequences than one launch takes (1024): the call splits into two launches
    whose records and unit flags sit at their offsets in one workspace; one head is
    marked everywhere, so both launches redo units."""
    rng = np.random.default_rng(5)
    lengths = [int(x) for x in rng.integers(0, 131, size=1100)]
    w = wl.varlen_case(lengths, 2, 128, 128, seed=77)
    w.A_log = np.array([4.0, -1.0], dtype=np.float32)
    _run(kda, w, "1100 sequences")


def test_prefill_weak_decay_long(kda):
    """Near-unit decay (A_log = -6) over 2000 rows: the state carries information across
    many chunks, so errors in the chain would accumulate."""
    w = wl.varlen_case([2000, 700], 2, 128, 128, seed=19)
    w.A_log = np.full(2, -6.0, dtype=np.float32)
    _run(kda, w, "weak decay long")


def test_prefill_one_long_sequence(kda):
    """One sequence of 65,573 rows (1,025 chunks, the last of 37 rows): a chain sixteen
    times longer than the bench's longest. Head 0 decays weakly (A_log = -6), so the state
    carries every chunk's contribution to the end; head 1 decays at the workloads' rates."""
    w = wl.varlen_case([65573], 2, 128, 128, seed=78)
    w.A_log = np.array([-6.0, 0.3], dtype=np.float32)
    _run(kda, w, "one long sequence")


def test_prefill_repeat_bit_identical(kda):
    w = wl.varlen_case([300, 129, 64], 4, 128, 128, seed=23)
    dw = hx.DeviceWorkload(w)
    first = hx.run_gpu(dw, kda).clone()
    pool_first = dw.pool_flat.clone()
    ref_pool = torch.from_numpy(w.pool).cuda()
    out = torch.empty_like(first)
    for _ in range(20):
        dw.pool_flat.copy_(ref_pool)
        hx.run_gpu(dw, kda, out=out)
        assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    assert torch.equal(dw.pool_flat.view(torch.int32), pool_first.view(torch.int32))


def test_prefill_slot_semantics(kda):
    """The chunk kernel's slot handling: null slot read-only, negative slot from zero,
    out-of-range slot flagged with zero outputs and no state access."""
    w = wl.varlen_case([70, 5, 130, 64, 1], 2, 128, 128, seed=29, num_slots=12)
    w.index_buf = np.array([[3], [-1], [11], [40], [7]], np.int32)
    w.null_slot = 11
    dw = hx.DeviceWorkload(w)
    out = hx.run_gpu(dw, kda)
    ref = ko.run(w)
    assert ref.err_flags == ko.ERR_SLOT_OUT_OF_RANGE
    hx.check(dw, out, ref, fp32_path=False, label="prefill slot semantics")
    o = out.float().cpu()
    assert torch.all(o[205:269] == 0)


def test_mixed_batch_null_slot_padding(kda):
    lengths = [1, 1, 1, 100]
    w = wl.varlen_case(lengths, 2, 128, 128, seed=33, num_decodes=3, kind="mixed", num_slots=10)
    w.index_buf = np.array([[0], [4], [0], [6]], np.int32)
    w.null_slot = 0
    _run(kda, w, "mixed null slot")


@pytest.mark.parametrize("num_decodes,H", [(1, 1), (3, 2), (300, 4)])
def test_mixed_batch_decode_workers(kda, num_decodes, H):
    """At K = V = 128 the decodes of a mixed batch run on worker CTAs of the chunk launch,
    each 128-thread group walking (decode, head, slice) tiles with the next tile staged
    ahead: few tiles (groups with nothing to do) and many (long grid-stride walks)."""
    lengths = [1] * num_decodes + [130, 64]
    w = wl.varlen_case(lengths, H, 128, 128, seed=200 + num_decodes, index_stride=3,
                       num_decodes=num_decodes, kind="mixed", num_slots=2 * len(lengths) + 8)
    _run(kda, w, f"mixed workers d={num_decodes} H={H}")


def test_mixed_batch_decode_worker_slot_semantics(kda):
    """Decode slots out of range (error bit, zero outputs), negative (zero state, no write)
    and the null slot (read, not written) among valid ones, on the worker path."""
    lengths = [1] * 40 + [90]
    w = wl.varlen_case(lengths, 2, 128, 128, seed=210, num_decodes=40, kind="mixed",
                       num_slots=64)
    idx = np.arange(1, 42, dtype=np.int32).reshape(41, 1)
    idx[3] = -1
    idx[7] = 64            # out of range
    idx[11] = 0            # null slot
    idx[12] = 1 << 30      # out of range
    w.index_buf = idx
    w.null_slot = 0
    _run(kda, w, "mixed worker slots")


def test_mixed_batch_repeat_bit_identical(kda):
    w = wl.varlen_case([1] * 50 + [200, 70], 4, 128, 128, seed=220, num_decodes=50, kind="mixed")
    dw = hx.DeviceWorkload(w)
    first = None
    for _ in range(5):
        dw.reset_pool()
        out = hx.run_gpu(dw, kda)
        torch.cuda.synchronize()
        snap = (out.clone(), dw.pool_flat.clone())
        if first is None:
            first = snap
        assert torch.equal(snap[0], first[0]) and torch.equal(snap[1], first[1])


@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (32, 32)])
def test_prefill_empty_sequence_out_of_range_slot(kda, K, V):
    """An empty sequence whose slot is out of range sets the range bit on the chunked path
    (K, V in {64, 128}) and on the token-recurrent one (K or V of 32) alike, and touches
    nothing."""
    w = wl.varlen_case([0, 70, 0, 5], 2, K, V, seed=300 + K, num_slots=8)
    w.index_buf = np.array([[9], [1], [2], [3]], np.int32)
    ref = ko.run(w)
    assert ref.err_flags == ko.ERR_SLOT_OUT_OF_RANGE
    dw = hx.DeviceWorkload(w)
    out = hx.run_gpu(dw, kda)
    hx.check(dw, out, ref, fp32_path=(K == 32), label=f"empty out-of-range K={K}")


def test_prefill_fp16_range_flag(kda):
    """Values of ~1e5 exceed the fp16 range that the chunked path's V - K^G S operand has:
    the call reports it in the error word (bit 2) instead of returning Inf silently."""
    w = wl.varlen_case([70, 40], 2, 128, 128, seed=310)
    HK = w.H * w.K
    v = w.mixed_qkv[:, 2 * HK:].view(np.uint16)
    big = wl.f32_to_bf16_bits(np.float32(1e5) * np.random.default_rng(5).standard_normal(v.shape).astype(np.float32))
    w.mixed_qkv[:, 2 * HK:] = big
    dw = hx.DeviceWorkload(w)
    hx.run_gpu(dw, kda)
    torch.cuda.synchronize()
    err = int(dw.err.cpu().item())
    assert err & 4, f"range bit not set (err = {err})"
