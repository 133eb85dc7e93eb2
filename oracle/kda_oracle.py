"""Python side of the KDA oracle (TEST INFRASTRUCTURE ONLY).

Only the tests, the smoke check and the bench's CPU-baseline leg may import this
module. It loads the fp64 C oracle (`kda_oracle.c`, compiled by `build()`) and
adds the addressing semantics of the five library calls on top of it:

* the state slot of entry i is index_buf[i * index_stride] (the strided
  `state_indices` view of vLLM PR #51682, section "implementation breakdown",
  item 1: the kernel loads `state_indices + i_n * stride_state_indices`);
* a slot in [0, num_slots) is read as the initial state and the final state is
  written back in place, except for the null slot, which padded requests read
  but never write (PR #60683, section "Refusal and steps", CUDA graphs);
* a negative slot starts from a zero state and writes nothing;
* a slot >= num_slots sets bit 0 of the error word, its rows' outputs are zero
  and nothing is read or written;
* decode rows are one token per sequence, spec-verify rows are grouped by
  request (T consecutive rows each), prefill and mixed batches follow
  cu_seqlens, with the mixed batch's length-1 decodes first (PR #50649,
  section Purpose: decodes of a mixed batch take the recurrent path).

Nothing here is shared with the CUDA path.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lib = None

ERR_SLOT_OUT_OF_RANGE = 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP when available). Returns the library path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        D = ctypes.c_double
        lib.kda_oracle_gate.argtypes = [P, I64, P, I64, I64, I, I, P, P, I, D, P, P]
        lib.kda_oracle_gate.restype = None
        lib.kda_oracle_recurrent.argtypes = [P, I64, P, I64, P, I64, P, P, I64, I, I, I, P, P,
                                             I, D, D, D, P, P, I64, I, I, I]
        lib.kda_oracle_recurrent.restype = None
        lib.kda_oracle_chunked.argtypes = [P, I64, P, I64, P, I64, P, P, I64, I, I, I, P, P,
                                           I, D, D, D, I, P, P, I64, I]
        lib.kda_oracle_chunked.restype = None
        lib.kda_oracle_recurrent_ckpt.argtypes = [P, I64, P, I64, P, I64, P, P, I64, I, I, I, P, P,
                                                  I, D, D, D, P, P, I64, P, I64, I]
        lib.kda_oracle_recurrent_ckpt.restype = None
        lib.kda_oracle_max_threads.argtypes = []
        lib.kda_oracle_max_threads.restype = I
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def gate(raw_g, raw_beta, A_log, dt_bias, lower_bound, H, K):
    """fp64 g [N, H*K] and beta [N, H] from bf16 raw_g / raw_beta bits."""
    lib = _load()
    raw_g = np.ascontiguousarray(raw_g, dtype=np.uint16)
    raw_beta = np.ascontiguousarray(raw_beta, dtype=np.uint16)
    N = raw_g.shape[0]
    A_log = np.ascontiguousarray(A_log, dtype=np.float32)
    dt = None if dt_bias is None else np.ascontiguousarray(dt_bias, dtype=np.float32)
    g = np.empty((N, H * K), dtype=np.float64)
    b = np.empty((N, H), dtype=np.float64)
    lib.kda_oracle_gate(_ptr(raw_g), raw_g.shape[1], _ptr(raw_beta), raw_beta.shape[1], N, H, K,
                        _ptr(A_log), _ptr(dt), int(lower_bound is not None),
                        float(lower_bound or 0.0), _ptr(g), _ptr(b))
    return g, b


@dataclasses.dataclass
class OracleResult:
    out: np.ndarray            # fp64 [N, H*V]; NaN for rows/heads not computed
    final_states: np.ndarray   # fp64 [num_entries, H, K, V]
    slots: np.ndarray          # int64 [num_entries] slot of each entry
    writes: np.ndarray         # bool [num_entries]: final state written back to its slot
    err_flags: int
    heads: tuple               # (head_lo, head_hi) computed

    def expected_pool(self, pool: np.ndarray) -> np.ndarray:
        """fp64 copy of `pool` with the written slots replaced by the final states
        (only meaningful when every head was computed)."""
        exp = pool.astype(np.float64)
        HKV = self.final_states[0].size if len(self.final_states) else 0
        for e in range(len(self.slots)):
            if self.writes[e]:
                exp[self.slots[e], :HKV] = self.final_states[e].reshape(-1)
        return exp


def run(w, *, heads: tuple | None = None, chunked: bool = False, chunk_size: int | None = None,
        nthreads: int = 0, bounds: list | None = None, slots: np.ndarray | None = None) -> OracleResult:
    """Evaluate one library call on a `Workload` (see workloads.py) in fp64.

    `bounds` / `slots` override the rows and slots of each entry (used by the
    tests to compose calls); `heads` restricts the heads computed."""
    lib = _load()
    H, K, V = w.H, w.K, w.V
    h_lo, h_hi = heads if heads is not None else (0, H)
    bounds = w.seq_bounds() if bounds is None else bounds
    slots = w.indices().astype(np.int64) if slots is None else np.asarray(slots, dtype=np.int64)
    E = len(bounds)
    assert len(slots) == E
    N = w.N
    states = np.zeros((E, H, K, V), dtype=np.float64)
    valid = np.ones(E, dtype=bool)
    writes = np.zeros(E, dtype=bool)
    err = 0
    for e in range(E):
        s = int(slots[e])
        if s >= w.num_slots:
            valid[e] = False
            err |= ERR_SLOT_OUT_OF_RANGE
        elif s >= 0:
            states[e] = w.pool[s, : H * K * V].reshape(H, K, V).astype(np.float64)
            writes[e] = s != w.null_slot
    out = np.full((N, H * V), np.nan, dtype=np.float64)
    rb = np.array([b[0] for b, ok in zip(bounds, valid) if ok], dtype=np.int64)
    re = np.array([b[1] for b, ok in zip(bounds, valid) if ok], dtype=np.int64)
    vidx = np.nonzero(valid)[0]
    sub = np.ascontiguousarray(states[vidx])
    qkv = np.ascontiguousarray(w.mixed_qkv, dtype=np.uint16)
    rg = np.ascontiguousarray(w.raw_g, dtype=np.uint16)
    rbeta = np.ascontiguousarray(w.raw_beta, dtype=np.uint16)
    A_log = np.ascontiguousarray(w.A_log, dtype=np.float32)
    dt = None if w.dt_bias is None else np.ascontiguousarray(w.dt_bias, dtype=np.float32)
    lb = w.lower_bound
    if len(vidx):
        if chunked:
            assert heads is None
            C = chunk_size or w.chunk_size
            lib.kda_oracle_chunked(_ptr(qkv), qkv.shape[1], _ptr(rg), rg.shape[1], _ptr(rbeta),
                                   rbeta.shape[1], _ptr(rb), _ptr(re), len(vidx), H, K, V,
                                   _ptr(A_log), _ptr(dt), int(lb is not None), float(lb or 0.0),
                                   float(w.scale), float(w.eps), int(C), _ptr(sub), _ptr(out),
                                   H * V, int(nthreads))
        else:
            lib.kda_oracle_recurrent(_ptr(qkv), qkv.shape[1], _ptr(rg), rg.shape[1], _ptr(rbeta),
                                     rbeta.shape[1], _ptr(rb), _ptr(re), len(vidx), H, K, V,
                                     _ptr(A_log), _ptr(dt), int(lb is not None), float(lb or 0.0),
                                     float(w.scale), float(w.eps), _ptr(sub), _ptr(out), H * V,
                                     int(h_lo), int(h_hi), int(nthreads))
    states[vidx] = sub
    for e in range(E):
        if not valid[e]:
            b0, b1 = bounds[e]
            out[b0:b1, :] = 0.0
    return OracleResult(out=out, final_states=states, slots=slots, writes=writes & valid,
                        err_flags=err, heads=(h_lo, h_hi))


@dataclasses.dataclass
class CheckpointResult:
    out: np.ndarray            # fp64 [N, H*V]
    ckpt: np.ndarray           # fp64 [R, T, H, K, V] state after each token
    slots: np.ndarray          # int64 [R, T] slot of each (request, token) column
    writes: np.ndarray         # bool [R, T] the checkpoint is written to its slot
    err_flags: int

    def expected_pool(self, pool: np.ndarray) -> np.ndarray:
        exp = pool.astype(np.float64)
        R, T = self.slots.shape
        HKV = self.ckpt[0, 0].size if self.ckpt.size else 0
        for r in range(R):
            for t in range(T):
                if self.writes[r, t]:
                    exp[self.slots[r, t], :HKV] = self.ckpt[r, t].reshape(-1)
        return exp


def run_spec_checkpoints(w, nthreads: int = 0) -> CheckpointResult:
    """Spec-verify with per-token state checkpoints, on a spec Workload whose block-table
    rows are at least T wide (index_stride >= tokens_per_req).

    Request r with a_r = num_accepted[r] accepted tokens from the previous step (1 when
    `w.num_accepted` is None) reads its initial state from column a_r - 1 of its row,
    index_buf[r*stride + a_r - 1], and writes the state after its token t to column t,
    index_buf[r*stride + t]: the block table of `1 + num_speculative_blocks` columns
    (vLLM PR #51682, body) with the accepted-token count the padded requests carry (PR
    #60683, section "Refusal and steps", CUDA graphs). Slot rules per column are those of
    `run`: negative -> zero state (column a_r - 1) / no write, the null slot -> read but
    never written, >= num_slots -> bit 0 of the error word and no write; if the read column
    is out of range, or a_r is outside [1, T], the request's outputs are zero and nothing
    of it is read or written (bit 0 set)."""
    lib = _load()
    H, K, V, T = w.H, w.K, w.V, w.tokens_per_req
    R = w.num_entries
    flat = np.asarray(w.index_buf).reshape(-1)
    slots = np.stack([flat[r * w.index_stride: r * w.index_stride + T] for r in range(R)]).astype(np.int64) \
        if R else np.zeros((0, T), np.int64)
    acc = np.ones(R, dtype=np.int64) if w.num_accepted is None else np.asarray(w.num_accepted, np.int64)
    states = np.zeros((R, H, K, V), dtype=np.float64)
    valid = np.ones(R, dtype=bool)
    err = 0
    for r in range(R):
        if not 1 <= acc[r] <= T:
            valid[r] = False
            err |= ERR_SLOT_OUT_OF_RANGE
            continue
        s0 = int(slots[r, acc[r] - 1])
        if s0 >= w.num_slots:
            valid[r] = False
            err |= ERR_SLOT_OUT_OF_RANGE
        elif s0 >= 0:
            states[r] = w.pool[s0, : H * K * V].reshape(H, K, V).astype(np.float64)
    writes = np.zeros((R, T), dtype=bool)
    for r in range(R):
        if not valid[r]:
            continue
        for t in range(T):
            st = int(slots[r, t])
            if st >= w.num_slots:
                err |= ERR_SLOT_OUT_OF_RANGE
            elif st >= 0 and st != w.null_slot:
                writes[r, t] = True
    out = np.zeros((w.N, H * V), dtype=np.float64)
    ckpt = np.zeros((R, T, H, K, V), dtype=np.float64)
    vidx = np.nonzero(valid)[0]
    if len(vidx):
        rb = np.array([r * T for r in vidx], dtype=np.int64)
        re = rb + T
        sub = np.ascontiguousarray(states[vidx])
        subck = np.zeros((len(vidx), T, H, K, V), dtype=np.float64)
        qkv = np.ascontiguousarray(w.mixed_qkv, dtype=np.uint16)
        rg = np.ascontiguousarray(w.raw_g, dtype=np.uint16)
        rbeta = np.ascontiguousarray(w.raw_beta, dtype=np.uint16)
        A_log = np.ascontiguousarray(w.A_log, dtype=np.float32)
        dt = None if w.dt_bias is None else np.ascontiguousarray(w.dt_bias, dtype=np.float32)
        lb = w.lower_bound
        lib.kda_oracle_recurrent_ckpt(_ptr(qkv), qkv.shape[1], _ptr(rg), rg.shape[1], _ptr(rbeta),
                                      rbeta.shape[1], _ptr(rb), _ptr(re), len(vidx), H, K, V,
                                      _ptr(A_log), _ptr(dt), int(lb is not None), float(lb or 0.0),
                                      float(w.scale), float(w.eps), _ptr(sub), _ptr(out), H * V,
                                      _ptr(subck), T, int(nthreads))
        ckpt[vidx] = subck
    return CheckpointResult(out=out, ckpt=ckpt, slots=slots, writes=writes, err_flags=err)
