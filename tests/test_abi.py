"""Host-only checks of the C-ABI library: it loads, exports every function that
include/kda.h declares, and rejects bad arguments on the host with the right status
before launching anything (no GPU needed: every call here fails validation first)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def kda():
    from linear_attention_state_recurrent_gb300 import build
    build.build()
    from linear_attention_state_recurrent_gb300 import kda as k
    return k


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("kda_gate", "kda_packed_decode", "kda_spec_verify", "kda_chunk_prefill",
              "kda_mixed_batch", "kda_chunk_prefill_workspace_bytes", "kda_last_error",
              "kda_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(kda):
    lib = ctypes.CDLL(kda._LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"libkda.so does not export {name}"
    assert set(declared_functions()) == set(kda.EXPORTED)


def test_status_strings(kda):
    for code, name in ((0, "KDA_OK"), (1, "KDA_ERR_INVALID_ARGUMENT"), (2, "KDA_ERR_UNSUPPORTED"),
                       (3, "KDA_ERR_WORKSPACE"), (4, "KDA_ERR_CUDA")):
        assert kda.lib.kda_status_string(code).decode() == name


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails before any launch


def _heads(kda, H=2, K=128, V=128, A_log=FAKE, lb=None, scale=0.1, eps=1e-6):
    return kda.KdaHeads(H=H, K=K, V=V, A_log=A_log.value if A_log else None, dt_bias=None,
                        has_lower_bound=int(lb is not None), lower_bound=float(lb or 0.0),
                        scale=scale, l2_eps=eps)


def _state(kda, num_slots=8, slot_stride=2 * 128 * 128, index_stride=1, null_slot=-1, pool=FAKE):
    return kda.KdaState(pool=pool.value if pool else None, num_slots=num_slots,
                        slot_stride=slot_stride, indices=FAKE.value, index_stride=index_stride,
                        null_slot=null_slot)


def _decode(kda, hd, st, N=4, ld_qkv=3 * 2 * 128, ld_out=2 * 128, out=FAKE):
    return kda.lib.kda_packed_decode(FAKE, ld_qkv, FAKE, 2 * 128, FAKE, 2, N, ctypes.byref(hd),
                                     ctypes.byref(st), out, ld_out, None, None)


@pytest.mark.parametrize("case,status,pattern", [
    (dict(index_stride=0), 1, "index_stride"),
    (dict(index_stride=-8), 1, "index_stride"),
    (dict(slot_stride=100), 1, "slot_stride"),
    (dict(slot_stride=2 * 128 * 128 + 2), 1, "multiple of 4"),
    (dict(null_slot=8), 1, "null_slot"),
    (dict(num_slots=0), 1, "num_slots"),
    (dict(pool=None), 1, "pool"),
])
def test_decode_state_validation(kda, case, status, pattern):
    hd = _heads(kda)
    st = _state(kda, **case)
    assert _decode(kda, hd, st) == status
    assert re.search(pattern, kda.last_error())


@pytest.mark.parametrize("case,status,pattern", [
    (dict(K=96), 2, "K and V"),
    (dict(V=256), 2, "K and V"),
    (dict(H=0), 1, "H must"),
    (dict(A_log=None), 1, "A_log"),
    (dict(lb=float("nan")), 1, "lower_bound"),
    (dict(lb=1.0), 1, "lower_bound"),
    (dict(eps=-1.0), 1, "l2_eps"),
    (dict(scale=float("inf")), 1, "scale"),
])
def test_decode_heads_validation(kda, case, status, pattern):
    hd = _heads(kda, **case)
    st = _state(kda, slot_stride=max(2 * 128 * 256, 1))
    assert _decode(kda, hd, st) == status
    assert re.search(pattern, kda.last_error())


def test_decode_row_validation(kda):
    hd, st = _heads(kda), _state(kda)
    assert _decode(kda, hd, st, ld_qkv=100) == 1 and "ld_qkv" in kda.last_error()
    assert _decode(kda, hd, st, ld_out=10) == 1 and "ld_out" in kda.last_error()
    assert _decode(kda, hd, st, out=None) == 1
    assert _decode(kda, hd, st, out=ctypes.c_void_p((1 << 20) + 2)) == 1 and "aligned" in kda.last_error()
    assert _decode(kda, hd, st, N=-1) == 1


def test_zero_sized_calls_are_noops(kda):
    hd, st = _heads(kda), _state(kda)
    assert _decode(kda, hd, st, N=0) == 0
    assert kda.last_error() == ""


def test_spec_verify_width_validation(kda):
    hd, st = _heads(kda), _state(kda)
    for T in (0, 65):
        s = kda.lib.kda_spec_verify(FAKE, 768, FAKE, 256, FAKE, 2, 4, T, ctypes.byref(hd),
                                    ctypes.byref(st), FAKE, 256, None, None)
        assert s == 1 and "tokens_per_req" in kda.last_error()


def test_chunk_prefill_validation(kda):
    hd, st = _heads(kda), _state(kda)
    cu = np.array([0, 5, 3], np.int32)
    args = lambda cuh, cs=64, nd=0, npf=2: (FAKE, 768, FAKE, 256, FAKE, 2, FAKE,  # noqa: E731
                                           cuh.ctypes.data_as(ctypes.c_void_p), nd, npf,
                                           ctypes.byref(hd), ctypes.byref(st), None, 0, FAKE,
                                           256, None, None)
    assert kda.lib.kda_mixed_batch(*args(cu)) == 1 and "non-decreasing" in kda.last_error()
    cu2 = np.array([0, 1, 3, 9], np.int32)
    assert kda.lib.kda_mixed_batch(*args(cu2, nd=2, npf=1)) == 1 and "length 2" in kda.last_error()
    s = kda.lib.kda_chunk_prefill(FAKE, 768, FAKE, 256, FAKE, 2, FAKE,
                                  cu2.ctypes.data_as(ctypes.c_void_p), 3, 32, ctypes.byref(hd),
                                  ctypes.byref(st), None, 0, FAKE, 256, None, None)
    assert s == 2 and "chunk_size" in kda.last_error()


def test_workspace_query_is_host_only(kda):
    cu = np.array([0, 100, 300, 301], np.int32)
    hd = _heads(kda)
    n = kda.lib.kda_chunk_prefill_workspace_bytes(cu.ctypes.data_as(ctypes.c_void_p), 3,
                                                  ctypes.byref(hd), 64)
    # one record per (chunk of 64 rows, head), then one flag byte per record rounded up to 16
    assert n == (2 + 4 + 1) * 2 * 57856 + 16
    for K, V in ((64, 64), (64, 128), (128, 64)):
        hk = _heads(kda, K=K, V=V)
        assert kda.lib.kda_chunk_prefill_workspace_bytes(cu.ctypes.data_as(ctypes.c_void_p), 3,
                                                         ctypes.byref(hk), 64) == n
    h32 = _heads(kda, K=32, V=64)   # the token-recurrent path needs none
    assert kda.lib.kda_chunk_prefill_workspace_bytes(cu.ctypes.data_as(ctypes.c_void_p), 3,
                                                     ctypes.byref(h32), 64) == 0
    assert kda.lib.kda_chunk_prefill_workspace_bytes(cu.ctypes.data_as(ctypes.c_void_p), 3,
                                                     ctypes.byref(hd), 16) == 0
    assert "chunk_size" in kda.last_error()


def test_binding_rejects_2d_indices_without_gpu(kda):
    torch = pytest.importorskip("torch")
    idx = torch.zeros(4, 2, dtype=torch.int32)
    pool = torch.zeros(2, 1, 32, 32)
    with pytest.raises(ValueError, match="one-dimensional"):
        kda.make_state(pool, idx)


def _fused(kda, hd, st, conv=None, norm=None, T=1, N=4, ld_qkv=768, ld_g=256, qkv=FAKE):
    c = ctypes.byref(conv) if conv is not None else None
    n = ctypes.byref(norm) if norm is not None else None
    if T == 1:
        return kda.lib.kda_fused_decode(qkv, ld_qkv, FAKE, ld_g, FAKE, 2, N, ctypes.byref(hd),
                                        ctypes.byref(st), c, n, FAKE, 256, None, None)
    return kda.lib.kda_fused_spec_verify(qkv, ld_qkv, FAKE, ld_g, FAKE, 2, N, T, ctypes.byref(hd),
                                         ctypes.byref(st), c, n, FAKE, 256, None, None)


@pytest.mark.parametrize("conv_kw,pattern", [
    (dict(width=0), "conv width"),
    (dict(width=5), "conv width"),
    (dict(weight=None), "conv weight"),
    (dict(slot_stride=10), "slot_stride"),
    (dict(slot_stride=3 * 768 + 2), "multiple of 4"),
    (dict(state=(1 << 20) + 2), "8-byte aligned"),
])
def test_fused_conv_validation(kda, conv_kw, pattern):
    hd, st = _heads(kda), _state(kda)
    kw = dict(weight=FAKE.value, bias=None, state=FAKE.value, slot_stride=3 * 768, width=4)
    kw.update(conv_kw)
    conv = kda.KdaShortConv(**kw)
    assert _fused(kda, hd, st, conv=conv) == 1
    assert re.search(pattern, kda.last_error())


def test_fused_norm_and_row_validation(kda):
    hd, st = _heads(kda), _state(kda)
    bad_ld = kda.KdaGatedNorm(gate=FAKE.value, ld_gate=255, weight=FAKE.value, eps=1e-5)
    assert _fused(kda, hd, st, norm=bad_ld) == 1 and "ld_gate" in kda.last_error()
    bad_eps = kda.KdaGatedNorm(gate=FAKE.value, ld_gate=256, weight=FAKE.value, eps=-1.0)
    assert _fused(kda, hd, st, norm=bad_eps) == 1 and "eps" in kda.last_error()
    no_w = kda.KdaGatedNorm(gate=FAKE.value, ld_gate=256, weight=None, eps=1e-5)
    assert _fused(kda, hd, st, norm=no_w) == 1 and "weight" in kda.last_error()
    # rows for 8-byte channel loads: pitches multiples of 4, 8-byte aligned pointers
    assert _fused(kda, hd, st, ld_qkv=770) == 1 and "multiples of 4" in kda.last_error()
    assert _fused(kda, hd, st, qkv=ctypes.c_void_p((1 << 20) + 4)) == 1
    for T in (0, 17):
        assert _fused(kda, hd, st, T=T) == 1 and "tokens_per_req" in kda.last_error()
    assert _fused(kda, hd, st, N=0) == 0


def test_spec_checkpoint_validation(kda):
    hd = _heads(kda)
    st = _state(kda, index_stride=4)
    args = lambda T, acc=None: (FAKE, 768, FAKE, 256, FAKE, 2, 4, T, acc, ctypes.byref(hd),  # noqa: E731
                                ctypes.byref(st), FAKE, 256, None, None)
    assert kda.lib.kda_spec_verify_checkpoints(*args(5)) == 1 and "index_stride" in kda.last_error()
    assert kda.lib.kda_spec_verify_checkpoints(*args(17)) == 1 and "tokens_per_req" in kda.last_error()
    assert kda.lib.kda_spec_verify_checkpoints(*args(4, ctypes.c_void_p((1 << 20) + 2))) == 1
    assert "num_accepted" in kda.last_error()


def test_bounded_wait_selftest_needs_an_error_word(kda):
    assert kda.lib.kda_selftest_bounded_wait(None, None) == 1
    assert "err_flags" in kda.last_error()


def test_oversized_batches_are_refused_before_launch(kda):
    """One call is one launch: more entries than a grid can hold (4 CTAs per entry and head,
    at most 2^31 - 1 blocks) is refused with KDA_ERR_UNSUPPORTED instead of being cut short."""
    hd, st = _heads(kda), _state(kda)
    limit = (2 ** 31 - 1) // (4 * hd.H)
    too_many = limit + 1
    assert _decode(kda, hd, st, N=too_many) == 2 and "split the call" in kda.last_error()
    s = kda.lib.kda_spec_verify(FAKE, 768, FAKE, 256, FAKE, 2, too_many, 8, ctypes.byref(hd),
                                ctypes.byref(st), FAKE, 256, None, None)
    assert s == 2 and "split the call" in kda.last_error()
    st8 = _state(kda, index_stride=8)
    s = kda.lib.kda_spec_verify_checkpoints(FAKE, 768, FAKE, 256, FAKE, 2, too_many, 8, None,
                                            ctypes.byref(hd), ctypes.byref(st8), FAKE, 256, None, None)
    assert s == 2 and "split the call" in kda.last_error()
    assert _fused(kda, hd, st, N=too_many) == 2 and "split the call" in kda.last_error()
    for nd, npf in ((too_many, 0), (0, too_many), (limit, 1)):
        s = kda.lib.kda_mixed_batch(FAKE, 768, FAKE, 256, FAKE, 2, FAKE, None, nd, npf,
                                    ctypes.byref(hd), ctypes.byref(st), None, 0, FAKE, 256, None, None)
        assert s == 2 and "split the call" in kda.last_error()
    # at the limit the count itself is accepted (the call then fails on its NULL host cu_seqlens)
    s = kda.lib.kda_chunk_prefill(FAKE, 768, FAKE, 256, FAKE, 2, FAKE, None, limit, 64,
                                  ctypes.byref(hd), ctypes.byref(st), None, 0, FAKE, 256, None, None)
    assert s == 1 and "split the call" not in kda.last_error()


def _varlen_inputs(torch, N=10, H=2, K=128, V=128, S=2, slots=4):
    qkv = torch.zeros(N, 2 * H * K + H * V, dtype=torch.bfloat16)
    g = torch.zeros(N, H * K, dtype=torch.bfloat16)
    b = torch.zeros(N, H, dtype=torch.bfloat16)
    A_log = torch.zeros(H)
    pool = torch.zeros(slots, H, K, V)
    idx = torch.arange(S, dtype=torch.int32)
    cu = torch.tensor([0, 4, N], dtype=torch.int32)
    return qkv, g, b, A_log, pool, idx, cu


def test_binding_refuses_short_varlen_inputs_without_gpu(kda):
    """The C ABI has no row counts; the binding refuses inputs that would be read past
    their end: too few state indices, sequence bounds beyond the rows, short per-token
    tensors and a short caller-passed output."""
    torch = pytest.importorskip("torch")
    qkv, g, b, A_log, pool, idx, cu = _varlen_inputs(torch)
    with pytest.raises(ValueError, match="state_indices"):
        kda.kda_chunk_prefill(qkv, g, b, A_log, None, None, pool, idx[:1], cu)
    with pytest.raises(ValueError, match="end at"):
        kda.kda_chunk_prefill(qkv[:8], g[:8], b[:8], A_log, None, None, pool, idx, cu)
    with pytest.raises(ValueError, match="start at"):
        kda.kda_chunk_prefill(qkv, g, b, A_log, None, None, pool, idx,
                              torch.tensor([-1, 4, 10], dtype=torch.int32))
    with pytest.raises(ValueError, match="raw_g"):
        kda.kda_chunk_prefill(qkv, g[:9], b, A_log, None, None, pool, idx, cu)
    with pytest.raises(ValueError, match="raw_beta"):
        kda.kda_mixed_batch(qkv, g, b[:9], A_log, None, None, pool, idx, cu, 0)
    with pytest.raises(ValueError, match="out"):
        kda.kda_chunk_prefill(qkv, g, b, A_log, None, None, pool, idx, cu,
                              out=torch.zeros(9, 2 * 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="same length"):
        kda.kda_chunk_prefill(qkv, g, b, A_log, None, None, pool, idx, cu,
                              cu_seqlens_host=torch.tensor([0, 10], dtype=torch.int32))


def test_binding_refuses_short_decode_inputs_without_gpu(kda):
    torch = pytest.importorskip("torch")
    qkv, g, b, A_log, pool, idx, _ = _varlen_inputs(torch, N=4, S=4)
    with pytest.raises(ValueError, match="raw_g"):
        kda.kda_packed_decode(qkv, g[:3], b, A_log, None, None, pool, idx)
    with pytest.raises(ValueError, match="raw_beta"):
        kda.kda_spec_verify(qkv, g, b[:3], A_log, None, None, pool, idx[:2], 2)
