"""Seeded synthetic inputs for the KDA recurrence, shared by the tests, the bench and smoke().

This module only draws random numbers and lays them out in the packed formats
the library consumes. It holds none of the method's arithmetic (no gate, no
normalisation, no update), so the oracle and the CUDA path can both be fed from
it without sharing any computation.

Formats (all host numpy arrays):
  mixed_qkv  uint16 bf16 bits [N, 3*H*K]   row = [q (H*K) | k (H*K) | v (H*V)], head-major
  raw_g      uint16 bf16 bits [N, H*K]
  raw_beta   uint16 bf16 bits [N, H]
  A_log      float32 [H]
  dt_bias    float32 [H*K]
  pool       float32 [num_slots, slot_stride]; slot s, head h at s*slot_stride + h*K*V,
             row-major [K][V]
  index_buf  int32 buffer; the call's state_indices are index_buf[i*index_stride]
  cu_seqlens int32 [num_seqs+1] (varlen calls only)

The workloads mirror the shapes named on the vLLM pages about Kimi-K3's KDA
path: the packed decode test matrix of PR #51682 (num_seqs in {1, 8, 32},
lower_bound in {-5, None}, state index stride in {1, 8}), a serving decode at
H=32, K=V=128 with state indices taken as column 0 of a block table of width
1 + num_speculative_blocks, spec-verify steps of at most 8 rows per request
(PR #60683), and chunked varlen prefill plus a mixed decode+prefill batch
(PR #50649).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Lengths of the eight prefill sequences: torch.randint(512, 8193, (8,)) drawn
# with torch.Generator().manual_seed(1) (pinned by a CPU test).
PREFILL_LENGTHS_SEED1 = [2372, 4818, 2094, 8025, 7872, 942, 5229, 2142]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 24
    for s in range(0, n, step):
        e = min(n, s + step)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = f32_to_bf16_bits(x)
    return out.reshape(shape)


@dataclasses.dataclass
class Workload:
    """One call's worth of inputs. `kind` is decode | spec | prefill | mixed."""

    name: str
    kind: str
    H: int
    K: int
    V: int
    mixed_qkv: np.ndarray
    raw_g: np.ndarray
    raw_beta: np.ndarray
    A_log: np.ndarray
    dt_bias: np.ndarray | None
    lower_bound: float | None
    scale: float
    eps: float
    pool: np.ndarray
    index_buf: np.ndarray
    index_stride: int
    num_entries: int            # number of state slots addressed (seqs or requests)
    null_slot: int = -1
    cu_seqlens: np.ndarray | None = None
    tokens_per_req: int = 1
    num_decodes: int = 0
    chunk_size: int = 64
    num_accepted: np.ndarray | None = None   # int32 [num_entries], spec checkpoints only
    # fused layer tail (short causal conv in front, gated RMSNorm behind); `fused` routes the
    # call through the fused entry points even when both parts are off
    fused: bool = False
    conv_width: int = 0
    conv_weight: np.ndarray | None = None    # bf16 bits [2HK+HV, conv_width]
    conv_bias: np.ndarray | None = None      # bf16 bits [2HK+HV]
    conv_pool: np.ndarray | None = None      # bf16 bits [num_slots, conv_slot_stride]
    out_gate: np.ndarray | None = None       # bf16 bits [N, H*V]
    norm_weight: np.ndarray | None = None    # fp32 [V]
    norm_eps: float = 1e-5

    @property
    def N(self) -> int:
        return int(self.mixed_qkv.shape[0])

    @property
    def num_slots(self) -> int:
        return int(self.pool.shape[0])

    @property
    def slot_stride(self) -> int:
        return int(self.pool.shape[1])

    def indices(self) -> np.ndarray:
        """The strided view the call reads: index_buf[i*index_stride] for i < num_entries."""
        flat = self.index_buf.reshape(-1)
        return flat[: (self.num_entries - 1) * self.index_stride + 1 : self.index_stride].copy() \
            if self.num_entries > 0 else flat[:0].copy()

    def seq_bounds(self) -> list[tuple[int, int]]:
        """[start, end) rows of each addressed entry, in entry order."""
        if self.kind == "decode":
            return [(n, n + 1) for n in range(self.num_entries)]
        if self.kind in ("spec", "spec_ckpt"):
            T = self.tokens_per_req
            return [(r * T, (r + 1) * T) for r in range(self.num_entries)]
        cu = self.cu_seqlens
        return [(int(cu[i]), int(cu[i + 1])) for i in range(self.num_entries)]

    def state_bytes_per_call(self) -> int:
        """fp32 state bytes read + written, counting each addressed (entry, head) tile
        once each way (the unit of the decode metric); with per-token checkpoints, one
        read and tokens_per_req writes per tile."""
        tile = 4 * self.K * self.V * self.H * self.num_entries
        if self.kind == "spec_ckpt":
            return tile * (1 + self.tokens_per_req)
        return 2 * tile


def _heads(rng, H, K, dt_std=0.1):
    A_log = rng.uniform(-1.0, 1.0, size=H).astype(np.float32)
    dt_bias = (rng.standard_normal(H * K, dtype=np.float32) * np.float32(dt_std)).astype(np.float32)
    return A_log, dt_bias


def _pool(rng, num_slots, slot_elems, std, touched=None, slot_stride=None):
    """fp32 pool; `touched` slots get N(0, std), the rest a cheap uniform filler."""
    slot_stride = slot_elems if slot_stride is None else slot_stride
    pool = np.empty((num_slots, slot_stride), dtype=np.float32)
    touched_set = set(range(num_slots)) if touched is None else set(int(t) for t in touched if 0 <= t < num_slots)
    for s in range(num_slots):
        if s in touched_set:
            pool[s] = rng.standard_normal(slot_stride, dtype=np.float32) * np.float32(std)
        else:
            pool[s] = (rng.random(slot_stride, dtype=np.float32) - np.float32(0.5)) * np.float32(2 * std)
    return pool


def decode_case(num_seqs: int, H: int, K: int, V: int, *, seed: int, lower_bound=None,
                index_stride: int = 1, num_slots: int | None = None, pool_std: float = 0.05,
                scale: float | None = None, eps: float = 1e-6, with_dt_bias: bool = True,
                extra_slot_stride: int = 0, name: str = "decode") -> Workload:
    """Packed decode: one token per sequence. The index buffer is a [num_seqs, index_stride]
    block table of distinct random slots in every column where the pool allows it."""
    assert K == V or True
    rng = np.random.default_rng(seed)
    if num_slots is None:
        num_slots = max(2 * num_seqs * index_stride, 8)
    width = 3 * H * K if K == V else 2 * H * K + H * V
    mixed_qkv = _normal_bf16(rng, (num_seqs, width))
    raw_g = _normal_bf16(rng, (num_seqs, H * K))
    raw_beta = _normal_bf16(rng, (num_seqs, H))
    A_log, dt_bias = _heads(rng, H, K)
    table = _block_table(rng, num_seqs, index_stride, num_slots)
    slot_elems = H * K * V
    pool = _pool(rng, num_slots, slot_elems, pool_std, slot_stride=slot_elems + extra_slot_stride)
    return Workload(name=name, kind="decode", H=H, K=K, V=V, mixed_qkv=mixed_qkv, raw_g=raw_g,
                    raw_beta=raw_beta, A_log=A_log, dt_bias=dt_bias if with_dt_bias else None,
                    lower_bound=lower_bound,
                    scale=(K ** -0.5) if scale is None else scale, eps=eps, pool=pool,
                    index_buf=table, index_stride=index_stride, num_entries=num_seqs)


def with_layer_tail(w: Workload, seed: int, conv_width: int | None = 4, norm: bool = True,
                    conv_bias: bool = True, conv_slot_extra: int = 8) -> Workload:
    """A copy of a decode or spec Workload whose mixed_qkv rows are the inputs of a
    depthwise short causal convolution (width conv_width, None = no convolution) and whose
    outputs go through a gated RMSNorm (norm=True). Conv weights N(0, 0.5), bias N(0, 0.1),
    conv-state pool N(0, 1) (past inputs) with conv_slot_extra spare elements per slot,
    output gate N(0, 1), norm weight 1 + N(0, 0.1), all bf16 except the fp32 norm weight."""
    rng = np.random.default_rng(seed)
    C = 2 * w.H * w.K + w.H * w.V
    kw = dict(w.__dict__)
    kw["fused"] = True
    if conv_width is not None:
        kw["conv_width"] = conv_width
        kw["conv_weight"] = _normal_bf16(rng, (C, conv_width), 0.5)
        kw["conv_bias"] = _normal_bf16(rng, (C,), 0.1) if conv_bias else None
        kw["conv_pool"] = _normal_bf16(rng, (w.num_slots, (conv_width - 1) * C + conv_slot_extra))
    if norm:
        kw["out_gate"] = _normal_bf16(rng, (w.N, w.H * w.V))
        kw["norm_weight"] = (1.0 + 0.1 * rng.standard_normal(w.V)).astype(np.float32)
    return Workload(**kw)


def _block_table(rng, rows, width, num_slots):
    """int32 [rows, width]. Column 0 holds distinct slots; the remaining columns are
    filled from a fresh permutation of the pool so that reading a wrong column lands
    on a valid but different slot."""
    table = np.empty((rows, width), dtype=np.int32)
    perm = rng.permutation(num_slots).astype(np.int32)
    assert rows <= num_slots
    table[:, 0] = perm[:rows]
    if width > 1:
        rest = np.concatenate([perm[rows:], rng.permutation(num_slots).astype(np.int32)])
        while rest.size < rows * (width - 1):
            rest = np.concatenate([rest, rng.permutation(num_slots).astype(np.int32)])
        table[:, 1:] = rest[: rows * (width - 1)].reshape(rows, width - 1)
    return table


def tiny_decode() -> Workload:
    """Tiny packed decode, seed 0: 4 seqs, H=2, K=V=32, pool of 8 slots N(0, 0.1),
    state_indices [5, 2, 7, 0] contiguous, lower_bound None."""
    rng = np.random.default_rng(0)
    N, H, K, V = 4, 2, 32, 32
    mixed_qkv = _normal_bf16(rng, (N, 3 * H * K))
    raw_g = _normal_bf16(rng, (N, H * K))
    raw_beta = _normal_bf16(rng, (N, H))
    A_log, dt_bias = _heads(rng, H, K)
    pool = _pool(rng, 8, H * K * V, 0.1)
    idx = np.array([5, 2, 7, 0], dtype=np.int32)
    return Workload(name="tiny_decode", kind="decode", H=H, K=K, V=V, mixed_qkv=mixed_qkv,
                    raw_g=raw_g, raw_beta=raw_beta, A_log=A_log, dt_bias=dt_bias,
                    lower_bound=None, scale=K ** -0.5, eps=1e-6, pool=pool, index_buf=idx,
                    index_stride=1, num_entries=N)


def serving_decode(lower_bound=-5.0, seed: int = 2) -> Workload:
    """Serving-shape packed decode: 128 seqs, H=32, K=V=128, pool of 512 slots N(0, 0.05)
    (1 GiB), state_indices = column 0 of an int32 [128, 8] block table (stride 8)."""
    w = decode_case(128, 32, 128, 128, seed=seed, lower_bound=lower_bound, index_stride=8,
                    num_slots=512, pool_std=0.05, name="serving_decode")
    return w


def shard_heads(w: Workload, lo: int, hi: int) -> Workload:
    """The same call restricted to heads [lo, hi): what one tensor-parallel rank holds.
    Heads are independent in the recurrence (each has its own state tile, gate and
    normalisation), so the ranks' results together are the unsharded call's."""
    H, K, V, N = w.H, w.K, w.V, w.N
    hs = hi - lo
    q = w.mixed_qkv[:, lo * K:hi * K]
    k = w.mixed_qkv[:, H * K + lo * K:H * K + hi * K]
    v = w.mixed_qkv[:, 2 * H * K + lo * V:2 * H * K + hi * V]
    pool = w.pool[:, :H * K * V].reshape(w.num_slots, H, K * V)[:, lo:hi].reshape(w.num_slots, hs * K * V)
    fields = dict(w.__dict__)
    fields.update(name=f"{w.name}[heads {lo}:{hi}]", H=hs,
                  mixed_qkv=np.ascontiguousarray(np.concatenate([q, k, v], axis=1)),
                  raw_g=np.ascontiguousarray(w.raw_g[:, lo * K:hi * K]),
                  raw_beta=np.ascontiguousarray(w.raw_beta[:, lo:hi]),
                  A_log=np.ascontiguousarray(w.A_log[lo:hi]),
                  dt_bias=None if w.dt_bias is None else np.ascontiguousarray(w.dt_bias[lo * K:hi * K]),
                  pool=np.ascontiguousarray(pool))
    assert not w.fused, "head sharding covers the plain calls"
    return Workload(**fields)


def serving_decode_index_sets(w: Workload, count: int = 4) -> list[np.ndarray]:
    """Disjoint sets of 128 slots (the first is the workload's own column 0), used by the
    bench to rotate which slots a step touches so that no step reads state from L2."""
    used = set(int(s) for s in w.indices())
    rest = [s for s in range(w.num_slots) if s not in used]
    rng = np.random.default_rng(12345)
    rng.shuffle(rest)
    sets = [w.indices().astype(np.int32)]
    n = w.num_entries
    for i in range(count - 1):
        sets.append(np.array(rest[i * n:(i + 1) * n], dtype=np.int32))
    return sets


def spec_verify(seed: int = 3, num_reqs: int = 16, T: int = 8, H: int = 32, K: int = 128,
                V: int = 128, num_slots: int = 256, num_padding: int = 2,
                lower_bound=None, index_stride: int = 1) -> Workload:
    """Spec-verify: num_reqs requests x T tokens (rows grouped by request), pool of 256 slots
    with slot 0 the null slot; the last `num_padding` requests are padding pointing at it."""
    rng = np.random.default_rng(seed)
    N = num_reqs * T
    mixed_qkv = _normal_bf16(rng, (N, 2 * H * K + H * V))
    raw_g = _normal_bf16(rng, (N, H * K))
    raw_beta = _normal_bf16(rng, (N, H))
    A_log, dt_bias = _heads(rng, H, K)
    real = (rng.permutation(num_slots - 1)[: num_reqs - num_padding] + 1).astype(np.int32)
    idx = np.concatenate([real, np.zeros(num_padding, dtype=np.int32)])
    buf = np.full((num_reqs, index_stride), -7, dtype=np.int32)
    buf[:, 0] = idx
    if index_stride > 1:
        buf[:, 1:] = rng.integers(0, num_slots, size=(num_reqs, index_stride - 1), dtype=np.int32)
    pool = _pool(rng, num_slots, H * K * V, 0.05)
    return Workload(name="spec_verify", kind="spec", H=H, K=K, V=V, mixed_qkv=mixed_qkv,
                    raw_g=raw_g, raw_beta=raw_beta, A_log=A_log, dt_bias=dt_bias,
                    lower_bound=lower_bound, scale=K ** -0.5, eps=1e-6, pool=pool,
                    index_buf=buf, index_stride=index_stride, num_entries=num_reqs,
                    null_slot=0, tokens_per_req=T)


def spec_checkpoints(seed: int = 6, num_reqs: int = 16, T: int = 8, H: int = 32, K: int = 128,
                     V: int = 128, num_slots: int = 256, num_padding: int = 2,
                     lower_bound=None, index_stride: int | None = None) -> Workload:
    """Spec-verify with per-token state checkpoints: each real request owns a block-table
    row of T distinct slots (columns beyond T, if index_stride > T, hold other slots) and
    a number of accepted tokens in [1, T] from the previous step; padding requests point
    every column at the null slot 0 with one accepted token."""
    stride = T if index_stride is None else index_stride
    assert stride >= T
    nreal = num_reqs - num_padding
    assert nreal * T <= num_slots - 1
    rng = np.random.default_rng(seed)
    N = num_reqs * T
    mixed_qkv = _normal_bf16(rng, (N, 2 * H * K + H * V))
    raw_g = _normal_bf16(rng, (N, H * K))
    raw_beta = _normal_bf16(rng, (N, H))
    A_log, dt_bias = _heads(rng, H, K)
    buf = np.zeros((num_reqs, stride), dtype=np.int32)
    buf[:nreal, :T] = (rng.permutation(num_slots - 1)[: nreal * T] + 1).reshape(nreal, T)
    if stride > T:
        buf[:, T:] = rng.integers(0, num_slots, size=(num_reqs, stride - T), dtype=np.int32)
    acc = np.ones(num_reqs, dtype=np.int32)
    acc[:nreal] = rng.integers(1, T + 1, size=nreal, dtype=np.int32)
    pool = _pool(rng, num_slots, H * K * V, 0.05)
    return Workload(name="spec_checkpoints", kind="spec_ckpt", H=H, K=K, V=V, mixed_qkv=mixed_qkv,
                    raw_g=raw_g, raw_beta=raw_beta, A_log=A_log, dt_bias=dt_bias,
                    lower_bound=lower_bound, scale=K ** -0.5, eps=1e-6, pool=pool,
                    index_buf=buf, index_stride=stride, num_entries=num_reqs,
                    null_slot=0, tokens_per_req=T, num_accepted=acc)


def varlen_case(lengths, H: int, K: int, V: int, *, seed: int, lower_bound=None,
                index_stride: int = 1, num_slots: int | None = None, pool_std: float = 0.05,
                num_decodes: int = 0, scale: float | None = None, eps: float = 1e-6,
                kind: str = "prefill", name: str = "prefill", chunk_size: int = 64) -> Workload:
    """Varlen prefill (or mixed batch when num_decodes > 0: the first num_decodes
    sequences must have length 1). Initial states N(0, pool_std) from the pool."""
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in lengths]
    S = len(lengths)
    N = int(sum(lengths))
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    mixed_qkv = _normal_bf16(rng, (N, 2 * H * K + H * V))
    raw_g = _normal_bf16(rng, (N, H * K))
    raw_beta = _normal_bf16(rng, (N, H))
    A_log, dt_bias = _heads(rng, H, K)
    if num_slots is None:
        num_slots = max(2 * S * index_stride, 8)
    table = _block_table(rng, S, index_stride, num_slots) if S > 0 else np.zeros((1, index_stride), np.int32)
    touched = table[:, 0] if S > 0 else []
    pool = _pool(rng, num_slots, H * K * V, pool_std, touched=touched)
    return Workload(name=name, kind=kind, H=H, K=K, V=V, mixed_qkv=mixed_qkv, raw_g=raw_g,
                    raw_beta=raw_beta, A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound,
                    scale=(K ** -0.5) if scale is None else scale, eps=eps, pool=pool,
                    index_buf=table, index_stride=index_stride, num_entries=S,
                    cu_seqlens=cu, num_decodes=num_decodes, chunk_size=chunk_size)


def chunked_prefill(lower_bound=None, seed: int = 1) -> Workload:
    """Chunked varlen prefill: 8 sequences with the seed-1 lengths (33,494 tokens),
    H=32, K=V=128, chunk 64, pool of 16 slots (slot stride H*K*V)."""
    return varlen_case(PREFILL_LENGTHS_SEED1, 32, 128, 128, seed=seed, lower_bound=lower_bound,
                       num_slots=16, name="chunked_prefill")


def mixed_batch(seed: int = 5, lower_bound=None) -> Workload:
    """Mixed batch: 96 length-1 decodes then 4 prefills of 4096 tokens, H=32, K=V=128,
    pool of 1024 slots, state indices with stride 4."""
    lengths = [1] * 96 + [4096] * 4
    return varlen_case(lengths, 32, 128, 128, seed=seed, lower_bound=lower_bound,
                       index_stride=4, num_slots=1024, num_decodes=96, kind="mixed",
                       name="mixed_batch")


def num_chunks(lengths, chunk_size: int = 64) -> int:
    return int(sum(math.ceil(int(L) / chunk_size) for L in lengths))


# ---------------------------------------------------------------------------
# Device upload and dispatch of a workload to the matching library call
# (torch is imported lazily so the generators stay importable without it).
# ---------------------------------------------------------------------------

def bf16_tensor(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class DeviceWorkload:
    """A Workload's tensors on a CUDA device, laid out as the library takes them."""

    def __init__(self, w, device="cuda:0"):
        import torch
        self.w = w
        self.device = device
        self.mixed_qkv = bf16_tensor(w.mixed_qkv, device)
        self.raw_g = bf16_tensor(w.raw_g, device)
        self.raw_beta = bf16_tensor(w.raw_beta, device)
        self.A_log = torch.from_numpy(w.A_log).to(device)
        self.dt_bias = None if w.dt_bias is None else torch.from_numpy(w.dt_bias).to(device)
        self.pool_flat = torch.from_numpy(w.pool).to(device)
        self.index_buf = torch.from_numpy(np.ascontiguousarray(w.index_buf)).to(device)
        self.cu = None if w.cu_seqlens is None else torch.from_numpy(w.cu_seqlens).to(device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.conv_weight = None if w.conv_weight is None else bf16_tensor(w.conv_weight, device)
        self.conv_bias = None if w.conv_bias is None else bf16_tensor(w.conv_bias, device)
        self.conv_pool = None if w.conv_pool is None else bf16_tensor(w.conv_pool, device)
        self.out_gate = None if w.out_gate is None else bf16_tensor(w.out_gate, device)
        self.norm_weight = None if w.norm_weight is None else torch.from_numpy(w.norm_weight).to(device)
        self.num_accepted = None if w.num_accepted is None else \
            torch.from_numpy(np.ascontiguousarray(w.num_accepted, dtype=np.int32)).to(device)

    def pool_view(self):
        w = self.w
        return self.pool_flat.as_strided((w.num_slots, w.H, w.K, w.V),
                                         (w.slot_stride, w.K * w.V, w.V, 1))

    def indices_view(self):
        flat = self.index_buf.reshape(-1)
        return flat.as_strided((self.w.num_entries,), (self.w.index_stride,))

    def reset_pool(self):
        import torch
        self.pool_flat.copy_(torch.from_numpy(self.w.pool).to(self.device))
        if self.conv_pool is not None:
            self.conv_pool.copy_(bf16_tensor(self.w.conv_pool, self.device))
        self.err.zero_()


def run_gpu(dw: DeviceWorkload, kda, out=None, stream=None, workspace=None):
    """Runs the library call the workload's kind names; returns the bf16 output tensor."""
    import torch
    w = dw.w
    args = (dw.mixed_qkv, dw.raw_g, dw.raw_beta, dw.A_log, dw.dt_bias, w.lower_bound,
            dw.pool_view(), dw.indices_view())
    kw = dict(scale=w.scale, l2_eps=w.eps, null_slot=w.null_slot, err_flags=dw.err, out=out,
              stream=stream)
    if w.fused:
        conv = None if w.conv_weight is None else (dw.conv_weight, dw.conv_bias, dw.conv_pool)
        norm = None if w.norm_weight is None else (dw.out_gate, dw.norm_weight, w.norm_eps)
        if w.kind == "decode":
            o, _ = kda.kda_fused_decode(*args, conv=conv, norm=norm, **kw)
        else:
            o, _ = kda.kda_fused_spec_verify(*args, w.tokens_per_req, conv=conv, norm=norm, **kw)
    elif w.kind == "decode":
        o, _ = kda.kda_packed_decode(*args, **kw)
    elif w.kind == "spec":
        o, _ = kda.kda_spec_verify(*args, w.tokens_per_req, **kw)
    elif w.kind == "spec_ckpt":
        table = dw.index_buf.reshape(w.num_entries, w.index_stride)
        o, _ = kda.kda_spec_verify_checkpoints(*args[:7], table, w.tokens_per_req,
                                               dw.num_accepted, **kw)
    elif w.kind == "prefill":
        o, _ = kda.kda_chunk_prefill(*args, dw.cu, cu_seqlens_host=torch.from_numpy(w.cu_seqlens),
                                     workspace=workspace, **kw)
    elif w.kind == "mixed":
        o, _ = kda.kda_mixed_batch(*args, dw.cu, w.num_decodes,
                                   cu_seqlens_host=torch.from_numpy(w.cu_seqlens),
                                   workspace=workspace, **kw)
    else:
        raise ValueError(w.kind)
    return o
