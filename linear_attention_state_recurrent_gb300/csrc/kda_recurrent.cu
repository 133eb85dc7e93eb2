// Recurrent (token-by-token) KDA kernels: the standalone gate, packed decode,
// spec-verify and the recurrent path over varlen rows.
//
// One CTA owns one (entry, head, 32-wide V slice) state tile. The value columns
// of S are independent in the update (column j of S_t depends only on column j
// of S_{t-1}; the coupling is only through the K-reductions k^T S and q^T S), so
// a K x V tile splits along V with no communication. The tile is loaded once with
// 128-bit coalesced accesses, advanced over the entry's tokens and stored once: in
// registers for the multi-token modes (recurrent_kernel), in shared memory for the
// single-token decode (decode_kernel), where no register then holds it and more CTAs fit
// on an SM. Gate, beta and the q/k L2 norms are fused in.
#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_pdl.cuh"

namespace kda {

// ---------------------------------------------------------------------------
// Standalone gate: g (fp32 [N, H*K]) and beta (fp32 [N, H]).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gate_kernel(Params p, int K, int64_t N, float *g_out,
                                                   float *beta_out)
{
    const int64_t HK = static_cast<int64_t>(p.H) * K;
    const int64_t total = N * HK;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += stride) {
        const int64_t t = i / HK;
        const int64_t hc = i - t * HK;
        const int h = static_cast<int>(hc / K);
        float x = bf16_to_f32(p.rg[t * p.ld_g + hc]);
        if (p.dt_bias) x += p.dt_bias[hc];
        g_out[i] = gate_log_decay(x, expf(p.A_log[h]), p.has_lb, p.lb);
    }
    const int64_t totb = N * p.H;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < totb;
         i += stride) {
        const int64_t t = i / p.H;
        const int h = static_cast<int>(i - t * p.H);
        beta_out[i] = sigmoid_f(bf16_to_f32(p.rb[t * p.ld_beta + h]));
    }
}

// ---------------------------------------------------------------------------
// Recurrent kernel.
//
// Thread layout (128 threads): cg = tid & 7 picks 4 value columns (one float4),
// rg = tid >> 3 picks rows rg, rg + 16, ... (RPT = K / 16 rows per thread). A warp
// therefore covers 4 rows x 32 columns per float4 load: four 128-byte segments.
//
// Per token:
//   [A] threads c < K compute the gate alpha_c and stash alpha_c, k_c, q_c (raw)
//       in shared memory; each warp sums |q|^2, |k|^2, q.k over its 32 channels.
//   [B] every thread decays its rows (S <- alpha S), accumulates k^T S and q^T S
//       over its rows, reduces over the 4 row groups of its warp by shuffles and
//       writes per-warp partials.
//   [C] every thread sums the 4 warps' partials for its 4 columns and forms
//       u = beta (v - S'^T k^), o = S'^T q^ + (q^.k^) u, then S <- S' + k^ u^T.
// ---------------------------------------------------------------------------
enum RowMode { kRowsDecode = 0, kRowsSpec = 1, kRowsVarlen = 2 };

// 8 CTAs per SM (64 registers per thread): the multi-token modes are bound by how many
// state bytes are in flight, and at 8 resident CTAs each SM keeps 128 KiB of loads
// outstanding. (The single-token decode runs decode_kernel below.)
template <int K, int V>
__global__ void __launch_bounds__(128, 8) recurrent_kernel(Params p, int mode, int T,
                                                        const int32_t *cu, int64_t entry_base)
{
    constexpr int VT = 32;              // value columns per CTA
    constexpr int VS = V / VT;          // V slices per (entry, head)
    constexpr int RPT = K / 16;         // rows per thread
    constexpr int KW = K / 32;          // warps that own channels in [A]

    // s_k is read again in [C], after the second barrier, so it alternates between two
    // buffers by token parity: token t+1's [A] may run while slower warps are still in
    // token t's [C]. The other arrays are last read before the second barrier.
    __shared__ float s_a[K], s_k[2][K], s_q[K];
    __shared__ float s_part[KW][3];
    __shared__ float s_red[4][2][VT];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int cg = tid & 7;
    const int rg = tid >> 3;

    pdl_wait_then_release();   // launched by launch_pdl: no global read before this

    const int64_t b = blockIdx.x;
    const int vs = static_cast<int>(b % VS);
    const int h = static_cast<int>((b / VS) % p.H);
    const int64_t e = b / (static_cast<int64_t>(VS) * p.H) + entry_base;

    int64_t row0, row1;
    if (mode == kRowsDecode) { row0 = e; row1 = e + 1; }
    else if (mode == kRowsSpec) { row0 = e * T; row1 = row0 + T; }
    else { row0 = cu[e]; row1 = cu[e + 1]; }

    const int j0 = vs * VT + cg * 4;                    // first of this thread's 4 columns
    const int64_t slot = load_slot(p, e);

    if (slot >= p.num_slots) {                          // out of range: flag, zero outputs
        if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
        if (rg == 0)
            for (int64_t t = row0; t < row1; t++) {
                uint2 z = make_uint2(0u, 0u);
                *reinterpret_cast<uint2 *>(p.out + t * p.ld_out + static_cast<int64_t>(h) * V + j0) = z;
            }
        return;
    }
    const bool has_state = slot >= 0;
    const bool writable = has_state && slot != p.null_slot;
    float *tile = has_state ? p.pool + slot * p.slot_stride + static_cast<int64_t>(h) * K * V : nullptr;

    // Issue the state loads first so they are in flight during the gate math.
    float4 S[RPT];
    if (has_state) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            S[i] = *reinterpret_cast<const float4 *>(tile + static_cast<int64_t>(rg + 16 * i) * V + j0);
    } else {
#pragma unroll
        for (int i = 0; i < RPT; i++) S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const float expA = expf(__ldg(p.A_log + h));
    const bool chan = tid < K;
    const float dtb = (chan && p.dt_bias) ? __ldg(p.dt_bias + h * K + tid) : 0.f;
    const int64_t HK = static_cast<int64_t>(p.H) * K;

    // Prefetch token row0's inputs.
    float nq = 0.f, nk = 0.f, ng = 0.f, nb = 0.f;
    float4 nv = make_float4(0.f, 0.f, 0.f, 0.f);
    auto fetch = [&](int64_t t) {
        const uint16_t *row = p.qkv + t * p.ld_qkv;
        if (chan) {
            nq = bf16_to_f32(row[h * K + tid]);
            nk = bf16_to_f32(row[HK + h * K + tid]);
            ng = bf16_to_f32(p.rg[t * p.ld_g + h * K + tid]);
        }
        const uint16_t *vp = row + 2 * HK + static_cast<int64_t>(h) * V + j0;
        nv = make_float4(bf16_to_f32(vp[0]), bf16_to_f32(vp[1]), bf16_to_f32(vp[2]), bf16_to_f32(vp[3]));
        nb = bf16_to_f32(p.rb[t * p.ld_beta + h]);
    };
    if (row0 < row1) fetch(row0);

    for (int64_t t = row0; t < row1; t++) {
        const int kb = static_cast<int>((t - row0) & 1);
        // ---- [A] gate + stash ----
        const float4 v = nv;
        const float beta = sigmoid_f(nb);
        if (chan) {
            const float g = gate_log_decay(ng + dtb, expA, p.has_lb, p.lb);
            s_a[tid] = expf(g);
            s_k[kb][tid] = nk;
            s_q[tid] = nq;
            float qq = warp_sum(nq * nq), kk = warp_sum(nk * nk), qk = warp_sum(nq * nk);
            if (lane == 0) { s_part[warp][0] = qq; s_part[warp][1] = kk; s_part[warp][2] = qk; }
        }
        __syncthreads();
        if (t + 1 < row1) fetch(t + 1);

        // ---- [B] decay + partial reductions ----
        float qq = 0.f, kk = 0.f, qk = 0.f;
#pragma unroll
        for (int w = 0; w < KW; w++) { qq += s_part[w][0]; kk += s_part[w][1]; qk += s_part[w][2]; }
        const float rq = p.scale * rsqrtf(qq + p.eps);
        const float rk = rsqrtf(kk + p.eps);
        float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const int r = rg + 16 * i;
            const float a = s_a[r], kr = s_k[kb][r], qr = s_q[r];
            S[i].x *= a; S[i].y *= a; S[i].z *= a; S[i].w *= a;
            pk[0] += kr * S[i].x; pk[1] += kr * S[i].y; pk[2] += kr * S[i].z; pk[3] += kr * S[i].w;
            pq[0] += qr * S[i].x; pq[1] += qr * S[i].y; pq[2] += qr * S[i].z; pq[3] += qr * S[i].w;
        }
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            pk[jj] += __shfl_xor_sync(0xffffffffu, pk[jj], 8);
            pk[jj] += __shfl_xor_sync(0xffffffffu, pk[jj], 16);
            pq[jj] += __shfl_xor_sync(0xffffffffu, pq[jj], 8);
            pq[jj] += __shfl_xor_sync(0xffffffffu, pq[jj], 16);
        }
        if (lane < 8) {
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
                s_red[warp][0][cg * 4 + jj] = pk[jj];
                s_red[warp][1][cg * 4 + jj] = pq[jj];
            }
        }
        __syncthreads();

        // ---- [C] u, o, rank-1 update ----
        float u[4], o[4];
        const float vv[4] = {v.x, v.y, v.z, v.w};
        const float qkh = qk * rq * rk;
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const int c = cg * 4 + jj;
            const float ks = (s_red[0][0][c] + s_red[1][0][c] + s_red[2][0][c] + s_red[3][0][c]) * rk;
            const float qs = (s_red[0][1][c] + s_red[1][1][c] + s_red[2][1][c] + s_red[3][1][c]) * rq;
            u[jj] = beta * (vv[jj] - ks);
            o[jj] = qs + qkh * u[jj];
        }
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const float kh = s_k[kb][rg + 16 * i] * rk;
            S[i].x += kh * u[0]; S[i].y += kh * u[1]; S[i].z += kh * u[2]; S[i].w += kh * u[3];
        }
        if (rg == 0) {
            uint2 packed;
            packed.x = static_cast<uint32_t>(f32_to_bf16(o[0])) | (static_cast<uint32_t>(f32_to_bf16(o[1])) << 16);
            packed.y = static_cast<uint32_t>(f32_to_bf16(o[2])) | (static_cast<uint32_t>(f32_to_bf16(o[3])) << 16);
            *reinterpret_cast<uint2 *>(p.out + t * p.ld_out + static_cast<int64_t>(h) * V + j0) = packed;
        }
    }

    if (writable && row0 < row1) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            *reinterpret_cast<float4 *>(tile + static_cast<int64_t>(rg + 16 * i) * V + j0) = S[i];
    }
}

// ---------------------------------------------------------------------------
// Packed decode: one token per entry, the state slice in shared memory.
//
// recurrent_kernel's thread layout and phases for one token, with the slice (K rows x 32
// columns, 16 KiB at K = 128) copied by cp.async into shared memory and kept there: each
// thread copies, reads twice (the reductions, with the decay folded into k and q, then the
// update) and stores the same RPT float4, so the slice needs no barrier of its own and is
// never written back. No register holds the tile (40 registers a thread),
// and shared memory sets how many CTAs an SM keeps: 12 at K = 128 (192 KiB of state loads
// in flight), where the register-resident tile allowed 8 (128 KiB).
// ---------------------------------------------------------------------------
template <int K, int V>
__global__ void __launch_bounds__(128, K == 128 ? 12 : 8) decode_kernel(Params p, int64_t entry_base, int64_t row_base)
{
    constexpr int VT = 32;              // value columns per CTA
    constexpr int VS = V / VT;          // V slices per (entry, head)
    constexpr int RPT = K / 16;         // rows per thread
    constexpr int CPL = K / 32;         // channels per lane in the norms

    // 18,432 bytes at K = 128: twelve CTAs fill an SM's 228 KiB (with the 1 KiB each
    // reserves). k and q stay in bf16 (their input type: exact); every warp forms the norms
    // itself, so no exchange array is needed for them. A row's alpha, k and q are one 8-byte
    // read, a warp's four partial sums of a phase one 16-byte read.
    __shared__ __align__(16) float4 s_tile[RPT][128];   // [row step][thread]
    __shared__ __align__(8) uint2 s_akq[K];   // per channel: alpha (fp32 bits), bf16 k | q << 16
    __shared__ __align__(16) float4 s_red[4][2][VT / 4];   // [warp][k^T S, q^T S][column group]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int cg = tid & 7;
    const int rg = tid >> 3;

    pdl_wait_then_release();   // launched by launch_pdl: no global read before this

    const int64_t b = blockIdx.x;
    const int vs = static_cast<int>(b % VS);
    const int h = static_cast<int>((b / VS) % p.H);
    const int64_t ei = b / (static_cast<int64_t>(VS) * p.H);
    const int64_t e = ei + entry_base, t = ei + row_base;   // entry (its slot) and row
    const int j0 = vs * VT + cg * 4;                    // first of this thread's 4 columns
    const int64_t slot = load_slot(p, e);
    uint16_t *orow = p.out + t * p.ld_out + static_cast<int64_t>(h) * V + j0;

    if (slot >= p.num_slots) {                          // out of range: flag, zero outputs
        if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
        if (rg == 0) *reinterpret_cast<uint2 *>(orow) = make_uint2(0u, 0u);
        return;
    }
    const bool has_state = slot >= 0;
    const bool writable = has_state && slot != p.null_slot;
    float *tile = has_state ? p.pool + slot * p.slot_stride + static_cast<int64_t>(h) * K * V + j0 : nullptr;

    // the state copies first, so they are in flight during the gate math
    if (has_state) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&s_tile[i][tid])),
                       tile + static_cast<int64_t>(rg + 16 * i) * V, true);
    }
    cp_async_commit();

    const bool chan = tid < K;
    const int64_t HK = static_cast<int64_t>(p.H) * K;
    const uint16_t *row = p.qkv + t * p.ld_qkv;
    // channels lane + 32 c of q and k (every warp: the norms); this thread's own channel is
    // the one with c == warp
    uint16_t qb[CPL], kb[CPL];
#pragma unroll
    for (int c = 0; c < CPL; c++) {
        qb[c] = row[h * K + lane + 32 * c];
        kb[c] = row[HK + h * K + lane + 32 * c];
    }
    float gr = 0.f, dtb = 0.f;
    if (chan) {
        gr = bf16_to_f32(p.rg[t * p.ld_g + h * K + tid]);
        if (p.dt_bias) dtb = __ldg(p.dt_bias + h * K + tid);
    }
    const uint16_t *vp = row + 2 * HK + static_cast<int64_t>(h) * V + j0;
    const float vv[4] = {bf16_to_f32(vp[0]), bf16_to_f32(vp[1]), bf16_to_f32(vp[2]), bf16_to_f32(vp[3])};
    const float beta = sigmoid_f(bf16_to_f32(p.rb[t * p.ld_beta + h]));
    const float expA = expf(__ldg(p.A_log + h));

    // ---- [A] gate + stash ----
    if (chan) {
        const float g = gate_log_decay(gr + dtb, expA, p.has_lb, p.lb);
        uint32_t kq = 0;
#pragma unroll
        for (int c = 0; c < CPL; c++)
            if (c == warp) kq = static_cast<uint32_t>(kb[c]) | (static_cast<uint32_t>(qb[c]) << 16);
        s_akq[tid] = make_uint2(__float_as_uint(expf(g)), kq);
    }
    float qq = 0.f, kk = 0.f, qk = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; c++) {
        const float qf = bf16_to_f32(qb[c]), kf = bf16_to_f32(kb[c]);
        qq += qf * qf; kk += kf * kf; qk += qf * kf;
    }
    qq = warp_sum(qq);
    kk = warp_sum(kk);
    qk = warp_sum(qk);
    cp_async_wait_all();   // this thread's own copies
    __syncthreads();

    // ---- [B] partial reductions over the decayed state (k alpha)^T S, (q alpha)^T S ----
    const float rq = p.scale * rsqrtf(qq + p.eps);
    const float rk = rsqrtf(kk + p.eps);
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < RPT; i++) {
        const int r = rg + 16 * i;
        const uint2 akq = s_akq[r];
        const float a = __uint_as_float(akq.x);
        const float kr = __uint_as_float(akq.y << 16) * a, qr = __uint_as_float(akq.y & 0xffff0000u) * a;
        const float4 S = has_state ? s_tile[i][tid] : make_float4(0.f, 0.f, 0.f, 0.f);
        pk[0] += kr * S.x; pk[1] += kr * S.y; pk[2] += kr * S.z; pk[3] += kr * S.w;
        pq[0] += qr * S.x; pq[1] += qr * S.y; pq[2] += qr * S.z; pq[3] += qr * S.w;
    }
#pragma unroll
    for (int jj = 0; jj < 4; jj++) {
        pk[jj] += __shfl_xor_sync(0xffffffffu, pk[jj], 8);
        pk[jj] += __shfl_xor_sync(0xffffffffu, pk[jj], 16);
        pq[jj] += __shfl_xor_sync(0xffffffffu, pq[jj], 8);
        pq[jj] += __shfl_xor_sync(0xffffffffu, pq[jj], 16);
    }
    if (lane < 8) {
        s_red[warp][0][cg] = make_float4(pk[0], pk[1], pk[2], pk[3]);
        s_red[warp][1][cg] = make_float4(pq[0], pq[1], pq[2], pq[3]);
    }
    __syncthreads();

    // ---- [C] u, o, S <- Diag(alpha) S + k^ u^T, stores ----
    float u[4], o[4];
    const float qkh = qk * rq * rk;
    {
        float4 kw[4], qw[4];
#pragma unroll
        for (int w = 0; w < 4; w++) { kw[w] = s_red[w][0][cg]; qw[w] = s_red[w][1][cg]; }
        const float ks[4] = {(kw[0].x + kw[1].x + kw[2].x + kw[3].x) * rk, (kw[0].y + kw[1].y + kw[2].y + kw[3].y) * rk,
                             (kw[0].z + kw[1].z + kw[2].z + kw[3].z) * rk, (kw[0].w + kw[1].w + kw[2].w + kw[3].w) * rk};
        const float qs[4] = {(qw[0].x + qw[1].x + qw[2].x + qw[3].x) * rq, (qw[0].y + qw[1].y + qw[2].y + qw[3].y) * rq,
                             (qw[0].z + qw[1].z + qw[2].z + qw[3].z) * rq, (qw[0].w + qw[1].w + qw[2].w + qw[3].w) * rq};
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            u[jj] = beta * (vv[jj] - ks[jj]);
            o[jj] = qs[jj] + qkh * u[jj];
        }
    }
    if (rg == 0) {
        uint2 packed;
        packed.x = static_cast<uint32_t>(f32_to_bf16(o[0])) | (static_cast<uint32_t>(f32_to_bf16(o[1])) << 16);
        packed.y = static_cast<uint32_t>(f32_to_bf16(o[2])) | (static_cast<uint32_t>(f32_to_bf16(o[3])) << 16);
        *reinterpret_cast<uint2 *>(orow) = packed;
    }
    if (writable) {
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const int r = rg + 16 * i;
            const uint2 akq = s_akq[r];
            const float a = __uint_as_float(akq.x), kh = __uint_as_float(akq.y << 16) * rk;
            float4 S = s_tile[i][tid];
            S.x = fmaf(S.x, a, kh * u[0]); S.y = fmaf(S.y, a, kh * u[1]);
            S.z = fmaf(S.z, a, kh * u[2]); S.w = fmaf(S.w, a, kh * u[3]);
            *reinterpret_cast<float4 *>(tile + static_cast<int64_t>(r) * V) = S;
        }
    }
}

// ---------------------------------------------------------------------------
// Spec-verify kernel: T <= kSpecMaxT tokens per request. All T tokens' gates, betas
// and q/k norms are computed up front in one parallel pass (their inputs are loaded
// together with the state tile), so the sequential part is only the state update:
// one barrier per token, the reduction buffers double-buffered across tokens.
// Same tile split and thread layout as recurrent_kernel.
// ---------------------------------------------------------------------------
//
// CKPT = true is the checkpointing variant: the request's block-table row holds one slot
// per token; the state is read from column num_accepted[e] - 1 and the state after token
// t is stored to column t (the stores of token t overlap the reductions of token t + 1).
// ---------------------------------------------------------------------------
constexpr int kSpecMaxT = 16;
static_assert(kSpecCkptMaxT <= kSpecMaxT, "checkpointing requests run in the spec kernel");

template <int K, int V, bool CKPT>
__global__ void __launch_bounds__(128, CKPT ? 6 : 7) spec_kernel(Params p, int T, const int32_t *num_accepted)
{
    constexpr int VT = 32, VS = V / VT, RPT = K / 16;
    __shared__ float s_a[kSpecMaxT][K], s_k[kSpecMaxT][K], s_q[kSpecMaxT][K];
    __shared__ float s_tok[kSpecMaxT][4];          // rq, rk, q^.k^, beta
    __shared__ float s_red[2][4][2][VT];
    __shared__ float4 s_v[kSpecMaxT][VT / 4];      // this CTA's value columns of every token
    __shared__ int64_t s_col[CKPT ? kSpecMaxT : 1]; // checkpoint slot of every token

    pdl_wait_then_release();   // launched by launch_pdl: no global read before this
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, cg = tid & 7, rg = tid >> 3;
    const int64_t b = blockIdx.x;
    const int vs = static_cast<int>(b % VS);
    const int h = static_cast<int>((b / VS) % p.H);
    const int64_t e = b / (static_cast<int64_t>(VS) * p.H);
    const int64_t row0 = e * T;
    const int j0 = vs * VT + cg * 4;
    int64_t slot;
    if (CKPT) {
        const int acc = num_accepted ? __ldg(num_accepted + e) : 1;
        slot = (acc >= 1 && acc <= T)
                   ? static_cast<int64_t>(__ldg(p.indices + e * p.index_stride + (acc - 1)))
                   : p.num_slots;                    // a bad count is treated as a bad slot
        if (tid < T) s_col[tid] = static_cast<int64_t>(__ldg(p.indices + e * p.index_stride + tid));
    } else {
        slot = load_slot(p, e);
    }
    if (slot >= p.num_slots) {
        if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
        if (rg == 0)
            for (int t = 0; t < T; t++)
                *reinterpret_cast<uint2 *>(p.out + (row0 + t) * p.ld_out + static_cast<int64_t>(h) * V + j0) = make_uint2(0u, 0u);
        return;
    }
    const bool has_state = slot >= 0;
    const bool writable = has_state && slot != p.null_slot;
    float *tile = has_state ? p.pool + slot * p.slot_stride + static_cast<int64_t>(h) * K * V : nullptr;
    float4 S[RPT];
    if (has_state) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            S[i] = *reinterpret_cast<const float4 *>(tile + static_cast<int64_t>(rg + 16 * i) * V + j0);
    } else {
#pragma unroll
        for (int i = 0; i < RPT; i++) S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int64_t HK = static_cast<int64_t>(p.H) * K;
    uint16_t braw = 0;
    if (tid < T) braw = p.rb[(row0 + tid) * p.ld_beta + h];
    // the CTA's value columns of every token (threads (t, cg))
    if (rg < T) {
        const uint16_t *vp = p.qkv + (row0 + rg) * p.ld_qkv + 2 * HK + static_cast<int64_t>(h) * V + j0;
        s_v[rg][cg] = make_float4(bf16_to_f32(vp[0]), bf16_to_f32(vp[1]), bf16_to_f32(vp[2]), bf16_to_f32(vp[3]));
    }
    // every token's gate and raw q/k (threads c < K, one channel each), in batches of 8
    if (tid < K) {
        const float expA = expf(__ldg(p.A_log + h));
        const float dtb = p.dt_bias ? __ldg(p.dt_bias + h * K + tid) : 0.f;
        for (int t0 = 0; t0 < T; t0 += 8) {
            uint16_t qr[8], kr[8], gr[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                if (t0 + u < T) {
                    const int64_t rr = row0 + t0 + u;
                    const uint16_t *row = p.qkv + rr * p.ld_qkv;
                    qr[u] = row[h * K + tid];
                    kr[u] = row[HK + h * K + tid];
                    gr[u] = p.rg[rr * p.ld_g + h * K + tid];
                }
            }
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int t = t0 + u;
                if (t < T) {
                    const float g = gate_log_decay(bf16_to_f32(gr[u]) + dtb, expA, p.has_lb, p.lb);
                    s_a[t][tid] = expf(g);
                    s_k[t][tid] = bf16_to_f32(kr[u]);
                    s_q[t][tid] = bf16_to_f32(qr[u]);
                }
            }
        }
    }
    __syncthreads();
    // per-token |q|^2, |k|^2, q.k: 128 / kSpecMaxT threads per token, then shuffles
    {
        constexpr int TPT = 128 / kSpecMaxT;          // threads per token (8)
        const int t = tid / TPT, part = tid % TPT;
        float qq = 0.f, kk = 0.f, qk = 0.f;
        if (t < T) {
            for (int c = part; c < K; c += TPT) {
                const float q = s_q[t][c], k = s_k[t][c];
                qq += q * q; kk += k * k; qk += q * k;
            }
        }
#pragma unroll
        for (int o = TPT / 2; o > 0; o >>= 1) {
            qq += __shfl_xor_sync(0xffffffffu, qq, o);
            kk += __shfl_xor_sync(0xffffffffu, kk, o);
            qk += __shfl_xor_sync(0xffffffffu, qk, o);
        }
        if (t < T && part == 0) {
            const float rq = p.scale * rsqrtf(qq + p.eps), rk = rsqrtf(kk + p.eps);
            s_tok[t][0] = rq;
            s_tok[t][1] = rk;
            s_tok[t][2] = qk * rq * rk;
        }
        if (tid < T) s_tok[tid][3] = sigmoid_f(bf16_to_f32(braw));
    }
    __syncthreads();
    // offset of this thread's first state element inside a slot (checkpoint stores)
    const int64_t tile_off = CKPT ? static_cast<int64_t>(h) * K * V + static_cast<int64_t>(rg) * V + j0 : 0;
#pragma unroll(CKPT ? 2 : kSpecMaxT)
    for (int t = 0; t < kSpecMaxT; t++) {
        if (t >= T) break;
        const int bb = t & 1;
        float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const int r = rg + 16 * i;
            const float a = s_a[t][r], kr = s_k[t][r], qr = s_q[t][r];
            S[i].x *= a; S[i].y *= a; S[i].z *= a; S[i].w *= a;
            pk[0] += kr * S[i].x; pk[1] += kr * S[i].y; pk[2] += kr * S[i].z; pk[3] += kr * S[i].w;
            pq[0] += qr * S[i].x; pq[1] += qr * S[i].y; pq[2] += qr * S[i].z; pq[3] += qr * S[i].w;
        }
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            pk[jj] += __shfl_xor_sync(0xffffffffu, pk[jj], 8);
            pk[jj] += __shfl_xor_sync(0xffffffffu, pk[jj], 16);
            pq[jj] += __shfl_xor_sync(0xffffffffu, pq[jj], 8);
            pq[jj] += __shfl_xor_sync(0xffffffffu, pq[jj], 16);
        }
        if (lane < 8) {
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
                s_red[bb][warp][0][cg * 4 + jj] = pk[jj];
                s_red[bb][warp][1][cg * 4 + jj] = pq[jj];
            }
        }
        __syncthreads();
        const float rq = s_tok[t][0], rk = s_tok[t][1], qkh = s_tok[t][2], beta = s_tok[t][3];
        const float4 v4 = s_v[t][cg];
        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
        float u[4], o[4];
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const int c = cg * 4 + jj;
            const float ks = (s_red[bb][0][0][c] + s_red[bb][1][0][c] + s_red[bb][2][0][c] + s_red[bb][3][0][c]) * rk;
            const float qs = (s_red[bb][0][1][c] + s_red[bb][1][1][c] + s_red[bb][2][1][c] + s_red[bb][3][1][c]) * rq;
            u[jj] = beta * (vv[jj] - ks);
            o[jj] = qs + qkh * u[jj];
        }
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const float kh = s_k[t][rg + 16 * i] * rk;
            S[i].x += kh * u[0]; S[i].y += kh * u[1]; S[i].z += kh * u[2]; S[i].w += kh * u[3];
        }
        if (rg == 0) {
            uint2 packed;
            packed.x = static_cast<uint32_t>(f32_to_bf16(o[0])) | (static_cast<uint32_t>(f32_to_bf16(o[1])) << 16);
            packed.y = static_cast<uint32_t>(f32_to_bf16(o[2])) | (static_cast<uint32_t>(f32_to_bf16(o[3])) << 16);
            *reinterpret_cast<uint2 *>(p.out + (row0 + t) * p.ld_out + static_cast<int64_t>(h) * V + j0) = packed;
        }
        if (CKPT) {
            const int64_t cs = s_col[t];
            if (cs >= p.num_slots) {
                if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
            } else if (cs >= 0 && cs != p.null_slot) {
                float *ct = p.pool + cs * p.slot_stride + tile_off;
#pragma unroll
                for (int i = 0; i < RPT; i++)
                    *reinterpret_cast<float4 *>(ct + 16 * i * V) = S[i];
            }
        }
    }
    if (!CKPT && writable) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            *reinterpret_cast<float4 *>(tile + static_cast<int64_t>(rg + 16 * i) * V + j0) = S[i];
    }
}

template <int K, int V, bool CKPT>
static cudaError_t launch_spec_kv(const Params &p, int T, int64_t num_reqs,
                                  const int32_t *num_accepted, cudaStream_t stream)
{
    const int64_t grid = num_reqs * p.H * (V / 32);
    return launch_pdl(spec_kernel<K, V, CKPT>, dim3(static_cast<unsigned>(grid)), dim3(128), 0, stream, p, T,
                      num_accepted);
}

template <bool CKPT>
static cudaError_t launch_spec_dims(const Params &p, int K, int V, int T, int64_t num_reqs,
                                    const int32_t *num_accepted, cudaStream_t stream)
{
#define KDA_SPEC_CASE(KK, VV) \
    if (K == KK && V == VV) return launch_spec_kv<KK, VV, CKPT>(p, T, num_reqs, num_accepted, stream);
    KDA_SPEC_CASE(32, 32) KDA_SPEC_CASE(32, 64) KDA_SPEC_CASE(32, 128)
    KDA_SPEC_CASE(64, 32) KDA_SPEC_CASE(64, 64) KDA_SPEC_CASE(64, 128)
    KDA_SPEC_CASE(128, 32) KDA_SPEC_CASE(128, 64) KDA_SPEC_CASE(128, 128)
#undef KDA_SPEC_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_spec(const Params &p, int K, int V, int T, int64_t num_reqs, cudaStream_t stream)
{
    if (num_reqs <= 0) return cudaSuccess;
    if (T > kSpecMaxT)  // longer requests take the token-streaming recurrent kernel
        return launch_recurrent(p, K, V, kRowsSpec, T, nullptr, 0, num_reqs, stream);
    return launch_spec_dims<false>(p, K, V, T, num_reqs, nullptr, stream);
}

cudaError_t launch_spec_checkpoints(const Params &p, int K, int V, int T, int64_t num_reqs,
                                    const int32_t *num_accepted, cudaStream_t stream)
{
    if (num_reqs <= 0) return cudaSuccess;
    if (T < 1 || T > kSpecCkptMaxT) return cudaErrorInvalidValue;
    return launch_spec_dims<true>(p, K, V, T, num_reqs, num_accepted, stream);
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
cudaError_t launch_gate(const Params &p, int K, int64_t N, float *g_out, float *beta_out,
                        cudaStream_t stream)
{
    const int64_t total = N * p.H * static_cast<int64_t>(K);
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    gate_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p, K, N, g_out, beta_out);
    return cudaGetLastError();
}

template <int K, int V>
static cudaError_t launch_rec_kv(const Params &p, int mode, int T, const int32_t *cu,
                                 int64_t entry_base, int64_t num_entries, cudaStream_t stream)
{
    const int64_t grid = num_entries * p.H * (V / 32);
    const dim3 g(static_cast<unsigned>(grid)), blk(128);
    if (mode == kRowsDecode)   // row e for entry e
        return launch_pdl(decode_kernel<K, V>, g, blk, 0, stream, p, entry_base, entry_base);
    return launch_pdl(recurrent_kernel<K, V>, g, blk, 0, stream, p, mode, T, cu, entry_base);
}

template <int K, int V>
static cudaError_t launch_dec_kv(const Params &p, int64_t row_base, int64_t num_entries, cudaStream_t stream)
{
    const dim3 g(static_cast<unsigned>(num_entries * p.H * (V / 32))), blk(128);
    return launch_pdl(decode_kernel<K, V>, g, blk, 0, stream, p, static_cast<int64_t>(0), row_base);
}

cudaError_t launch_decode(const Params &p, int K, int V, int64_t row_base, int64_t num_entries,
                          cudaStream_t stream)
{
    if (num_entries <= 0) return cudaSuccess;
#define KDA_DEC_CASE(KK, VV) \
    if (K == KK && V == VV) return launch_dec_kv<KK, VV>(p, row_base, num_entries, stream);
    KDA_DEC_CASE(32, 32) KDA_DEC_CASE(32, 64) KDA_DEC_CASE(32, 128)
    KDA_DEC_CASE(64, 32) KDA_DEC_CASE(64, 64) KDA_DEC_CASE(64, 128)
    KDA_DEC_CASE(128, 32) KDA_DEC_CASE(128, 64) KDA_DEC_CASE(128, 128)
#undef KDA_DEC_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_recurrent(const Params &p, int K, int V, int mode, int T, const int32_t *cu,
                             int64_t entry_base, int64_t num_entries, cudaStream_t stream)
{
    if (num_entries <= 0) return cudaSuccess;
#define KDA_REC_CASE(KK, VV) \
    if (K == KK && V == VV) return launch_rec_kv<KK, VV>(p, mode, T, cu, entry_base, num_entries, stream);
    KDA_REC_CASE(32, 32) KDA_REC_CASE(32, 64) KDA_REC_CASE(32, 128)
    KDA_REC_CASE(64, 32) KDA_REC_CASE(64, 64) KDA_REC_CASE(64, 128)
    KDA_REC_CASE(128, 32) KDA_REC_CASE(128, 64) KDA_REC_CASE(128, 128)
#undef KDA_REC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
