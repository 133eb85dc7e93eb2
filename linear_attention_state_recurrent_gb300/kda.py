"""Thin ctypes binding of libkda (include/kda.h). Argument marshalling only: every
step of the computation runs in the library's CUDA kernels.

The functions carry the C names and take torch tensors already on the GPU. As
in vLLM's fused_recurrent_kda_packed_decode (PR #51682), the decode-style calls
return (out, state_pool), with the pool updated in place, and raise ValueError
when an argument is rejected (e.g. a state_indices view that is not 1-D).

Tensor conventions:
  mixed_qkv  bf16 [N, >= 2*H*K + H*V], unit inner stride (row = q | k | v)
  raw_g      bf16 [N, >= H*K];  raw_beta bf16 [N, >= H]
  A_log      fp32 [H];  dt_bias fp32 [H*K] (or [H, K]) or None
  state_pool fp32 [num_slots, H, K, V] with contiguous inner [H, K, V]; any slot stride
  state_indices int32 1-D, any positive stride
  cu_seqlens int32 [num_seqs + 1] on the GPU (a host copy is taken for launch sizing)
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARGUMENT = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_ERRFLAG_SLOT_RANGE = 1
KDA_ERRFLAG_TIMEOUT = 2

EXPORTED = ("kda_last_error", "kda_status_string", "kda_gate", "kda_packed_decode",
            "kda_spec_verify", "kda_spec_verify_checkpoints", "kda_fused_decode",
            "kda_fused_spec_verify", "kda_selftest_bounded_wait", "kda_chunk_prefill_workspace_bytes",
            "kda_chunk_prefill", "kda_mixed_batch", "kda_chunk_prefill_no_alloc")

KDA_NO_ALLOC_SCRATCH_BYTES = 64 * 1024 * 1024   # the fixed scratch of kda_chunk_prefill_no_alloc


class KdaHeads(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
                ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("has_lower_bound", ctypes.c_int32), ("lower_bound", ctypes.c_float),
                ("scale", ctypes.c_float), ("l2_eps", ctypes.c_float)]


class KdaState(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_slots", ctypes.c_int64),
                ("slot_stride", ctypes.c_int64), ("indices", ctypes.c_void_p),
                ("index_stride", ctypes.c_int64), ("null_slot", ctypes.c_int32)]


class KdaShortConv(ctypes.Structure):
    _fields_ = [("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("state", ctypes.c_void_p),
                ("slot_stride", ctypes.c_int64), ("width", ctypes.c_int32)]


class KdaGatedNorm(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("ld_gate", ctypes.c_int64), ("weight", ctypes.c_void_p),
                ("eps", ctypes.c_float)]


class KdaError(RuntimeError):
    pass


def _load():
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"libkda.so is not built ({_LIB_PATH}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    HP, SP = ctypes.POINTER(KdaHeads), ctypes.POINTER(KdaState)
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_last_error.argtypes = []
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_gate.restype = ctypes.c_int
    lib.kda_gate.argtypes = [P, I64, P, I64, I64, HP, P, P, P]
    lib.kda_packed_decode.restype = ctypes.c_int
    lib.kda_packed_decode.argtypes = [P, I64, P, I64, P, I64, I64, HP, SP, P, I64, P, P]
    lib.kda_spec_verify.restype = ctypes.c_int
    lib.kda_spec_verify.argtypes = [P, I64, P, I64, P, I64, I64, I32, HP, SP, P, I64, P, P]
    lib.kda_spec_verify_checkpoints.restype = ctypes.c_int
    lib.kda_spec_verify_checkpoints.argtypes = [P, I64, P, I64, P, I64, I64, I32, P, HP, SP, P, I64,
                                                P, P]
    CP, NP = ctypes.POINTER(KdaShortConv), ctypes.POINTER(KdaGatedNorm)
    lib.kda_fused_decode.restype = ctypes.c_int
    lib.kda_fused_decode.argtypes = [P, I64, P, I64, P, I64, I64, HP, SP, CP, NP, P, I64, P, P]
    lib.kda_fused_spec_verify.restype = ctypes.c_int
    lib.kda_fused_spec_verify.argtypes = [P, I64, P, I64, P, I64, I64, I32, HP, SP, CP, NP, P, I64,
                                          P, P]
    lib.kda_selftest_bounded_wait.restype = ctypes.c_int
    lib.kda_selftest_bounded_wait.argtypes = [P, P]
    lib.kda_chunk_prefill_workspace_bytes.restype = SZ
    lib.kda_chunk_prefill_workspace_bytes.argtypes = [P, I64, HP, I32]
    lib.kda_chunk_prefill.restype = ctypes.c_int
    lib.kda_chunk_prefill.argtypes = [P, I64, P, I64, P, I64, P, P, I64, I32, HP, SP, P, SZ, P,
                                      I64, P, P]
    lib.kda_mixed_batch.restype = ctypes.c_int
    lib.kda_mixed_batch.argtypes = [P, I64, P, I64, P, I64, P, P, I64, I64, HP, SP, P, SZ, P,
                                    I64, P, P]
    lib.kda_chunk_prefill_no_alloc.restype = ctypes.c_int
    lib.kda_chunk_prefill_no_alloc.argtypes = [P, I64, P, I64, P, I64, P, P, I64, I32, HP, SP, P,
                                               I64, P, P]
    return lib


lib = _load()


def last_error() -> str:
    return lib.kda_last_error().decode()


def _check(status: int, what: str):
    if status == KDA_OK:
        return
    msg = f"{what}: {lib.kda_status_string(status).decode()}: {last_error()}"
    if status in (KDA_ERR_INVALID_ARGUMENT, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE):
        raise ValueError(msg)
    raise KdaError(msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _rows(t: torch.Tensor, name: str, dtype=torch.bfloat16):
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with unit inner stride")
    return t.stride(0)


def make_heads(A_log, dt_bias, lower_bound, K, V, scale=None, l2_eps=1e-6):
    """Builds the kda_heads struct; keeps the tensors it points at alive via the return."""
    if A_log.dtype != torch.float32 or not A_log.is_contiguous():
        raise ValueError("A_log must be a contiguous fp32 tensor")
    if dt_bias is not None and (dt_bias.dtype != torch.float32 or not dt_bias.is_contiguous()):
        raise ValueError("dt_bias must be a contiguous fp32 tensor")
    H = A_log.numel()
    hd = KdaHeads(H=H, K=K, V=V, A_log=A_log.data_ptr(),
                  dt_bias=None if dt_bias is None else dt_bias.data_ptr(),
                  has_lower_bound=int(lower_bound is not None),
                  lower_bound=float(lower_bound if lower_bound is not None else 0.0),
                  scale=float(K ** -0.5 if scale is None else scale), l2_eps=float(l2_eps))
    return hd


def make_state(state_pool, state_indices, null_slot=-1):
    if state_indices.dim() != 1:
        raise ValueError("`state_indices` must be one-dimensional.")
    if state_indices.dtype != torch.int32:
        raise ValueError("state_indices must be int32")
    if state_pool.dtype != torch.float32 or state_pool.dim() != 4:
        raise ValueError("state_pool must be fp32 [num_slots, H, K, V]")
    _, H, K, V = state_pool.shape
    if state_pool.stride()[1:] != (K * V, V, 1):
        raise ValueError("state_pool's [H, K, V] part must be contiguous")
    return KdaState(pool=state_pool.data_ptr(), num_slots=state_pool.shape[0],
                    slot_stride=state_pool.stride(0), indices=state_indices.data_ptr(),
                    index_stride=state_indices.stride(0), null_slot=int(null_slot))


def _out(out, N, H, V, device):
    if out is None:
        out = torch.empty(N, H * V, dtype=torch.bfloat16, device=device)
    elif out.dim() != 2 or out.shape[0] < N:
        raise ValueError(f"out must have at least {N} rows")
    return out, _rows(out, "out")


def _need_rows(N, **tensors):
    """Every per-token input must hold at least N rows (the C ABI has no row counts, so a
    short tensor would be read past its end on the device)."""
    for name, t in tensors.items():
        if t is not None and (t.dim() < 1 or t.shape[0] < N):
            raise ValueError(f"{name} must have at least {N} rows (got {tuple(t.shape)})")


def kda_gate(raw_g, raw_beta, A_log, dt_bias=None, lower_bound=None, *, K=None, g_out=None,
             beta_out=None, stream=None):
    """Returns (g fp32 [N, H*K], beta fp32 [N, H])."""
    N = raw_g.shape[0]
    H = A_log.numel()
    K = raw_g.shape[1] // H if K is None else K
    ld_g, ld_b = _rows(raw_g, "raw_g"), _rows(raw_beta, "raw_beta")
    hd = make_heads(A_log, dt_bias, lower_bound, K, K)
    if g_out is None:
        g_out = torch.empty(N, H * K, dtype=torch.float32, device=raw_g.device)
    if beta_out is None:
        beta_out = torch.empty(N, H, dtype=torch.float32, device=raw_g.device)
    _check(lib.kda_gate(_ptr(raw_g), ld_g, _ptr(raw_beta), ld_b, N, ctypes.byref(hd),
                        _ptr(g_out), _ptr(beta_out), _stream(stream)), "kda_gate")
    return g_out, beta_out


def kda_packed_decode(mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound, initial_state,
                      state_indices, *, scale=None, l2_eps=1e-6, null_slot=-1, out=None,
                      err_flags=None, stream=None):
    """One decode token per sequence; returns (out bf16 [N, H*V], initial_state)."""
    _, H, K, V = initial_state.shape
    N = mixed_qkv.shape[0]
    hd = make_heads(A_log, dt_bias, lower_bound, K, V, scale, l2_eps)
    st = make_state(initial_state, state_indices, null_slot)
    if state_indices.shape[0] < N:
        raise ValueError("state_indices has fewer entries than sequences")
    _need_rows(N, raw_g=raw_g, raw_beta=raw_beta)
    out, ld_out = _out(out, N, H, V, mixed_qkv.device)
    _check(lib.kda_packed_decode(_ptr(mixed_qkv), _rows(mixed_qkv, "mixed_qkv"), _ptr(raw_g),
                                 _rows(raw_g, "raw_g"), _ptr(raw_beta), _rows(raw_beta, "raw_beta"),
                                 N, ctypes.byref(hd), ctypes.byref(st), _ptr(out), ld_out,
                                 _ptr(err_flags), _stream(stream)), "kda_packed_decode")
    return out, initial_state


def kda_spec_verify(mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound, initial_state,
                    state_indices, tokens_per_req, *, scale=None, l2_eps=1e-6, null_slot=-1,
                    out=None, err_flags=None, stream=None):
    """Requests of tokens_per_req consecutive rows; returns (out, initial_state)."""
    _, H, K, V = initial_state.shape
    N = mixed_qkv.shape[0]
    if N % tokens_per_req:
        raise ValueError("the row count must be a multiple of tokens_per_req")
    R = N // tokens_per_req
    hd = make_heads(A_log, dt_bias, lower_bound, K, V, scale, l2_eps)
    st = make_state(initial_state, state_indices, null_slot)
    if state_indices.shape[0] < R:
        raise ValueError("state_indices has fewer entries than requests")
    _need_rows(N, raw_g=raw_g, raw_beta=raw_beta)
    out, ld_out = _out(out, N, H, V, mixed_qkv.device)
    _check(lib.kda_spec_verify(_ptr(mixed_qkv), _rows(mixed_qkv, "mixed_qkv"), _ptr(raw_g),
                               _rows(raw_g, "raw_g"), _ptr(raw_beta), _rows(raw_beta, "raw_beta"),
                               R, int(tokens_per_req), ctypes.byref(hd), ctypes.byref(st),
                               _ptr(out), ld_out, _ptr(err_flags), _stream(stream)),
           "kda_spec_verify")
    return out, initial_state


def kda_spec_verify_checkpoints(mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound,
                                state_pool, block_table, tokens_per_req, num_accepted=None, *,
                                scale=None, l2_eps=1e-6, null_slot=-1, out=None, err_flags=None,
                                stream=None):
    """Spec-verify that stores the state after every token: request r reads column
    num_accepted[r] - 1 of block_table row r (int32 [num_reqs, >= tokens_per_req], unit
    inner stride) and writes the state after token t to column t. Returns
    (out, state_pool)."""
    _, H, K, V = state_pool.shape
    N = mixed_qkv.shape[0]
    T = int(tokens_per_req)
    if N % T:
        raise ValueError("the row count must be a multiple of tokens_per_req")
    R = N // T
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be int32 [num_reqs, width] with unit inner stride")
    if block_table.shape[0] < R or block_table.shape[1] < T:
        raise ValueError("block_table must have a row per request and a column per token")
    if num_accepted is not None and (num_accepted.dtype != torch.int32 or num_accepted.numel() < R
                                     or not num_accepted.is_contiguous()):
        raise ValueError("num_accepted must be a contiguous int32 tensor with a count per request")
    hd = make_heads(A_log, dt_bias, lower_bound, K, V, scale, l2_eps)
    st = make_state(state_pool, block_table[:, 0], null_slot)
    _need_rows(N, raw_g=raw_g, raw_beta=raw_beta)
    out, ld_out = _out(out, N, H, V, mixed_qkv.device)
    _check(lib.kda_spec_verify_checkpoints(
        _ptr(mixed_qkv), _rows(mixed_qkv, "mixed_qkv"), _ptr(raw_g), _rows(raw_g, "raw_g"),
        _ptr(raw_beta), _rows(raw_beta, "raw_beta"), R, T, _ptr(num_accepted),
        ctypes.byref(hd), ctypes.byref(st), _ptr(out), ld_out, _ptr(err_flags), _stream(stream)),
        "kda_spec_verify_checkpoints")
    return out, state_pool


def make_conv(weight, bias, conv_state):
    """kda_short_conv from weight bf16 [C, W], bias bf16 [C] or None, and the conv-state
    pool bf16 [num_slots, >= (W-1)*C] (unit inner stride)."""
    if weight.dtype != torch.bfloat16 or weight.dim() != 2 or not weight.is_contiguous():
        raise ValueError("conv weight must be a contiguous bf16 [C, W] tensor")
    if bias is not None and (bias.dtype != torch.bfloat16 or not bias.is_contiguous()):
        raise ValueError("conv bias must be a contiguous bf16 tensor")
    if conv_state.dtype != torch.bfloat16 or conv_state.dim() != 2 or conv_state.stride(1) != 1:
        raise ValueError("conv_state must be bf16 [num_slots, slot] with unit inner stride")
    return KdaShortConv(weight=weight.data_ptr(), bias=None if bias is None else bias.data_ptr(),
                        state=conv_state.data_ptr(), slot_stride=conv_state.stride(0),
                        width=weight.shape[1])


def make_norm(gate, weight, eps=1e-5):
    """kda_gated_norm from gate bf16 [N, >= H*V] and weight fp32 [V]."""
    if weight.dtype != torch.float32 or not weight.is_contiguous():
        raise ValueError("norm weight must be a contiguous fp32 tensor")
    return KdaGatedNorm(gate=gate.data_ptr(), ld_gate=_rows(gate, "gate"), weight=weight.data_ptr(),
                        eps=float(eps))


def _fused(name, mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound, initial_state,
           state_indices, T, conv, norm, scale, l2_eps, null_slot, out, err_flags, stream):
    _, H, K, V = initial_state.shape
    N = mixed_qkv.shape[0]
    if N % T:
        raise ValueError("the row count must be a multiple of tokens_per_req")
    E = N // T
    hd = make_heads(A_log, dt_bias, lower_bound, K, V, scale, l2_eps)
    st = make_state(initial_state, state_indices, null_slot)
    if state_indices.shape[0] < E:
        raise ValueError("state_indices has fewer entries than requests")
    _need_rows(N, raw_g=raw_g, raw_beta=raw_beta)
    if conv is not None and conv[2].shape[0] < initial_state.shape[0]:
        raise ValueError("conv_state must have a slot for every state slot")
    cv = None if conv is None else make_conv(*conv)
    nm = None if norm is None else make_norm(*norm)
    out, ld_out = _out(out, N, H, V, mixed_qkv.device)
    head = (_ptr(mixed_qkv), _rows(mixed_qkv, "mixed_qkv"), _ptr(raw_g), _rows(raw_g, "raw_g"),
            _ptr(raw_beta), _rows(raw_beta, "raw_beta"), E)
    tail = (ctypes.byref(hd), ctypes.byref(st), None if cv is None else ctypes.byref(cv),
            None if nm is None else ctypes.byref(nm), _ptr(out), ld_out, _ptr(err_flags),
            _stream(stream))
    if name == "kda_fused_decode":
        _check(lib.kda_fused_decode(*head, *tail), name)
    else:
        _check(lib.kda_fused_spec_verify(*head, int(T), *tail), name)
    return out, initial_state


def kda_fused_decode(mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound, initial_state,
                     state_indices, *, conv=None, norm=None, scale=None, l2_eps=1e-6,
                     null_slot=-1, out=None, err_flags=None, stream=None):
    """Packed decode with the short conv in front (conv = (weight, bias, conv_state) or None;
    mixed_qkv then holds the conv inputs) and the gated RMSNorm behind (norm = (gate,
    weight, eps) or None). Returns (out, initial_state)."""
    return _fused("kda_fused_decode", mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound,
                  initial_state, state_indices, 1, conv, norm, scale, l2_eps, null_slot, out,
                  err_flags, stream)


def kda_fused_spec_verify(mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound, initial_state,
                          state_indices, tokens_per_req, *, conv=None, norm=None, scale=None,
                          l2_eps=1e-6, null_slot=-1, out=None, err_flags=None, stream=None):
    """Spec-verify of tokens_per_req rows per request with the conv / gated norm of
    kda_fused_decode. Returns (out, initial_state)."""
    return _fused("kda_fused_spec_verify", mixed_qkv, raw_g, raw_beta, A_log, dt_bias,
                  lower_bound, initial_state, state_indices, int(tokens_per_req), conv, norm,
                  scale, l2_eps, null_slot, out, err_flags, stream)


def kda_selftest_bounded_wait(err_flags, stream=None):
    """Runs the bounded-wait self-test; err_flags (int32/uint32 device tensor) receives
    KDA_ERRFLAG_TIMEOUT once the wait has given up (after ~2 s)."""
    _check(lib.kda_selftest_bounded_wait(_ptr(err_flags), _stream(stream)), "kda_selftest_bounded_wait")


def _host_cu(cu_seqlens, cu_seqlens_host):
    """The host copy of cu_seqlens (read from the device when not given; a given copy must
    hold the same values as the device tensor, which the library sizes its launch from)."""
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous 1-D int32 tensor")
    if cu_seqlens_host is None:
        cu_seqlens_host = cu_seqlens.cpu()
    cu = cu_seqlens_host.to(torch.int32).contiguous()
    if cu.numel() != cu_seqlens.numel():
        raise ValueError("cu_seqlens_host and cu_seqlens must have the same length")
    return cu


def _check_varlen(cu_h, N, S, state_indices, **tensors):
    """Sequence bounds inside the N rows, one state index per sequence, N rows everywhere."""
    if S > 0 and (int(cu_h[0]) < 0 or int(cu_h[-1]) > N):
        raise ValueError(f"cu_seqlens must start at >= 0 and end at <= {N} rows "
                         f"(got {int(cu_h[0])} .. {int(cu_h[-1])})")
    if state_indices.shape[0] < S:
        raise ValueError(f"state_indices has fewer entries ({state_indices.shape[0]}) than sequences ({S})")
    _need_rows(N, **tensors)


def kda_chunk_prefill_workspace_bytes(cu_seqlens_host, H, K, V, chunk_size=64, num_seqs=None):
    cu = cu_seqlens_host.to(torch.int32).contiguous()
    n = cu.numel() - 1 if num_seqs is None else num_seqs
    hd = KdaHeads(H=H, K=K, V=V, A_log=1, dt_bias=None, has_lower_bound=0, lower_bound=0.0,
                  scale=1.0, l2_eps=0.0)
    return int(lib.kda_chunk_prefill_workspace_bytes(ctypes.c_void_p(cu.data_ptr()), n,
                                                     ctypes.byref(hd), chunk_size))


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        return None, 0
    if workspace is None or workspace.numel() * workspace.element_size() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def kda_chunk_prefill(mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound, initial_state,
                      state_indices, cu_seqlens, *, cu_seqlens_host=None, chunk_size=64,
                      scale=None, l2_eps=1e-6, null_slot=-1, out=None, workspace=None,
                      err_flags=None, stream=None):
    """Chunked varlen prefill; returns (out, initial_state)."""
    _, H, K, V = initial_state.shape
    N = mixed_qkv.shape[0]
    cu_h = _host_cu(cu_seqlens, cu_seqlens_host)
    S = cu_h.numel() - 1
    hd = make_heads(A_log, dt_bias, lower_bound, K, V, scale, l2_eps)
    st = make_state(initial_state, state_indices, null_slot)
    _check_varlen(cu_h, N, S, state_indices, raw_g=raw_g, raw_beta=raw_beta)
    out, ld_out = _out(out, N, H, V, mixed_qkv.device)
    nb = kda_chunk_prefill_workspace_bytes(cu_h, H, K, V, chunk_size)
    ws, ws_bytes = _workspace(nb, mixed_qkv.device, workspace)
    _check(lib.kda_chunk_prefill(_ptr(mixed_qkv), _rows(mixed_qkv, "mixed_qkv"), _ptr(raw_g),
                                 _rows(raw_g, "raw_g"), _ptr(raw_beta), _rows(raw_beta, "raw_beta"),
                                 _ptr(cu_seqlens), ctypes.c_void_p(cu_h.data_ptr()), S,
                                 int(chunk_size), ctypes.byref(hd), ctypes.byref(st), _ptr(ws),
                                 ws_bytes, _ptr(out), ld_out, _ptr(err_flags), _stream(stream)),
           "kda_chunk_prefill")
    return out, initial_state


def kda_chunk_prefill_no_alloc(mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound,
                               initial_state, state_indices, cu_seqlens, cu_seqlens_host, out, *,
                               chunk_size=64, scale=None, l2_eps=1e-6, null_slot=-1,
                               err_flags=None, stream=None):
    """kda_chunk_prefill for callers that cannot allocate device memory: the library keeps
    its records in a fixed 64 MiB device array (calls beyond it raise KdaError). `out` and
    the host copy of cu_seqlens are required, so this wrapper allocates nothing on the
    device either. The first call on a device should come before any stream capture; calls
    that overlap on the GPU race on the shared array. Returns (out, initial_state)."""
    _, H, K, V = initial_state.shape
    N = mixed_qkv.shape[0]
    if out is None or cu_seqlens_host is None:
        raise ValueError("kda_chunk_prefill_no_alloc needs `out` and `cu_seqlens_host`")
    cu_h = _host_cu(cu_seqlens, cu_seqlens_host)
    S = cu_h.numel() - 1
    hd = make_heads(A_log, dt_bias, lower_bound, K, V, scale, l2_eps)
    st = make_state(initial_state, state_indices, null_slot)
    _check_varlen(cu_h, N, S, state_indices, raw_g=raw_g, raw_beta=raw_beta)
    out, ld_out = _out(out, N, H, V, mixed_qkv.device)
    _check(lib.kda_chunk_prefill_no_alloc(_ptr(mixed_qkv), _rows(mixed_qkv, "mixed_qkv"), _ptr(raw_g),
                                          _rows(raw_g, "raw_g"), _ptr(raw_beta), _rows(raw_beta, "raw_beta"),
                                          _ptr(cu_seqlens), ctypes.c_void_p(cu_h.data_ptr()), S,
                                          int(chunk_size), ctypes.byref(hd), ctypes.byref(st),
                                          _ptr(out), ld_out, _ptr(err_flags), _stream(stream)),
           "kda_chunk_prefill_no_alloc")
    return out, initial_state


def kda_mixed_batch(mixed_qkv, raw_g, raw_beta, A_log, dt_bias, lower_bound, initial_state,
                    state_indices, cu_seqlens, num_decodes, *, cu_seqlens_host=None, scale=None,
                    l2_eps=1e-6, null_slot=-1, out=None, workspace=None, err_flags=None,
                    stream=None):
    """Mixed batch: the first num_decodes sequences (length 1) take the recurrent decode
    path, the rest the chunked prefill path; returns (out, initial_state)."""
    _, H, K, V = initial_state.shape
    N = mixed_qkv.shape[0]
    cu_h = _host_cu(cu_seqlens, cu_seqlens_host)
    S = cu_h.numel() - 1
    P = S - num_decodes
    hd = make_heads(A_log, dt_bias, lower_bound, K, V, scale, l2_eps)
    st = make_state(initial_state, state_indices, null_slot)
    _check_varlen(cu_h, N, S, state_indices, raw_g=raw_g, raw_beta=raw_beta)
    out, ld_out = _out(out, N, H, V, mixed_qkv.device)
    nb = kda_chunk_prefill_workspace_bytes(cu_h[num_decodes:], H, K, V, 64, num_seqs=P)
    ws, ws_bytes = _workspace(nb, mixed_qkv.device, workspace)
    _check(lib.kda_mixed_batch(_ptr(mixed_qkv), _rows(mixed_qkv, "mixed_qkv"), _ptr(raw_g),
                               _rows(raw_g, "raw_g"), _ptr(raw_beta), _rows(raw_beta, "raw_beta"),
                               _ptr(cu_seqlens), ctypes.c_void_p(cu_h.data_ptr()), int(num_decodes),
                               int(P), ctypes.byref(hd), ctypes.byref(st), _ptr(ws), ws_bytes,
                               _ptr(out), ld_out, _ptr(err_flags), _stream(stream)),
           "kda_mixed_batch")
    return out, initial_state
