// Fused layer tail for decode and spec-verify: short causal convolution -> KDA
// recurrence -> gated RMSNorm, in one kernel (the "spec conv, KDA recurrence, gated
// RMSNorm" run of the Kimi-K3 decode layer, vLLM PR #60683, section Purpose).
//
// The state tiles split along V exactly as in the recurrent kernel: one CTA of 128
// threads per (entry, head, 32-column slice), thread (rg, cg) holding rows rg, rg + 16, ...
// of columns 4cg .. 4cg + 3, up to eight CTAs per SM so that each SM keeps its share of
// the state stream in flight. The V / 32 slices of one (entry, head) form a thread-block
// cluster, which is what the two ends of the fusion need:
//   - every slice convolves the head's q and k channels (it needs all of them for k^T S
//     and q^T S) and its own v columns; the v conv state is written by its slice, the q/k
//     conv state by slice 0 after a cluster barrier, i.e. after every slice has read it;
//   - the RMS of o over V sums one partial per slice, read from the other slices' shared
//     memory (distributed shared memory) after the same barrier.
// All T tokens' convolutions, gates, betas and q/k norms are computed up front in one
// parallel pass; the sequential part is the state update with one barrier per token; the
// gated norm and the bf16 stores run once at the end over the slice's T x 32 outputs.
// Every cluster barrier is reached by all CTAs of the cluster: the conditions that guard
// them depend only on kernel arguments and on the (entry, head), which the slices share.
#include <cooperative_groups.h>

#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {

namespace {

namespace cgx = cooperative_groups;

constexpr int kFusedMaxT = 16;

// Fast-math activations (hardware exp2 and reciprocal): ~1e-6 relative error, far inside
// the bf16 output spacing. For y -> -inf the divisor overflows to inf and the result is 0.
__device__ __forceinline__ float silu_fast(float y) { return __fdividef(y, 1.f + __expf(-y)); }
__device__ __forceinline__ float sigmoid_fast(float y) { return __fdividef(1.f, 1.f + __expf(-y)); }

// Cluster barrier halves, in the forms that may sit in divergent code (the waits of one
// phase are reached at different places by different threads of a warp). Every thread
// pairs each arrive with one wait. arrive.release orders this thread's earlier memory
// accesses before the other CTAs' accesses after their wait; arrive.relaxed orders nothing.
__device__ __forceinline__ void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

// four bf16 values (8 bytes) to fp32
__device__ __forceinline__ void bf16x4(uint2 u, float f[4])
{
    f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
}

// MAXT: the most tokens per entry this instance takes (1 for decode, 8 or 16 for spec).
template <int K, int V, int MAXT>
__global__ void __cluster_dims__(V / 32, 1, 1) __launch_bounds__(128, MAXT == 1 ? 8 : 5)
fused_kernel(Params p, TailParams tp, int T)
{
    constexpr int VS = V / 32, VT = 32, RPT = K / 16;
    constexpr int NQK = K / 2, NCV = NQK + VT / 4, NI = NCV + K / 4;   // channel items
    static_assert(NI <= 128, "one channel item per thread");
    // every array below is read or written with 8- or 16-byte accesses somewhere
    __shared__ __align__(16) float s_a[MAXT][K];      // alpha = e^g
    __shared__ __align__(16) float s_k[MAXT][K];      // conv'd k, raw
    __shared__ __align__(16) float s_q[MAXT][K];      // conv'd q, raw
    __shared__ __align__(16) float s_v[MAXT][VT];     // conv'd v of the slice's columns
    __shared__ __align__(16) float s_o[MAXT][VT];     // o before the norm
    __shared__ __align__(16) float s_gw[MAXT][VT];    // norm weight * sigmoid(gate)
    __shared__ float s_tok[MAXT][4];                  // rq, rk, q^.k^, beta
    __shared__ float s_red[2][4][2][VT];              // per-warp partials of k^T S, q^T S
    __shared__ float s_ss[MAXT];                      // this slice's sum of o^2 per token
    __shared__ __align__(16) uint16_t s_cnew[3][2 * K + VT];   // new conv state: q|k, v
    // The state tile streams into shared memory during the channel pass (no registers held
    // meanwhile); each thread copies the elements it will hold, so it alone reads them back.
    // The 16-token instance loads straight into registers (its shared memory is full).
    constexpr bool kStage = MAXT <= 8;
    __shared__ __align__(16) float4 s_stage[kStage ? RPT : 1][128];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, cg = tid & 7, rg = tid >> 3;
    const uint32_t hv = blockIdx.x / VS;             // 32-bit index math (the grid is < 2^31)
    const int vs = static_cast<int>(blockIdx.x % VS);
    const int h = static_cast<int>(hv % static_cast<uint32_t>(p.H));
    const int64_t e = hv / static_cast<uint32_t>(p.H);
    const int64_t row0 = e * T;
    const int j0 = vs * VT + cg * 4;
    const int64_t slot = load_slot(p, e);
    if (slot >= p.num_slots) {                       // out of range (the whole cluster): zero outputs
        if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
        if (rg == 0)
            for (int t = 0; t < T; t++)
                *reinterpret_cast<uint2 *>(p.out + (row0 + t) * p.ld_out + static_cast<int64_t>(h) * V + j0) =
                    make_uint2(0u, 0u);
        return;
    }
    const bool has_state = slot >= 0;
    const bool writable = has_state && slot != p.null_slot;
    float *tile = has_state ? p.pool + slot * p.slot_stride + static_cast<int64_t>(h) * K * V : nullptr;
    float4 S[RPT];
    if (kStage && has_state) {
        const uint32_t st = static_cast<uint32_t>(__cvta_generic_to_shared(&s_stage[0][tid]));
#pragma unroll
        for (int i = 0; i < RPT; i++)
            cp_async16(st + i * 128 * 16, tile + static_cast<int64_t>(rg + 16 * i) * V + j0, true);
        cp_async_commit();
    } else if (!kStage) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            S[i] = has_state ? *reinterpret_cast<const float4 *>(tile + static_cast<int64_t>(rg + 16 * i) * V + j0)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // ---- channel pass, one item of 4 channels per thread, loads issued up front:
    //      [0, K/2): the head's q|k channels (conv; every slice needs all of them),
    //      [K/2, K/2 + 8): the slice's v columns (conv), [.., NI): gates, the rest: the
    //      norm's weight * sigmoid(gate) ----
    const int64_t HK = static_cast<int64_t>(p.H) * K;
    const int64_t C = 2 * HK + static_cast<int64_t>(p.H) * V;
    const int W = tp.conv_width;
    uint16_t *cstate = (W > 1 && has_state) ? tp.conv_state + slot * tp.conv_slot_stride : nullptr;
    const bool cwrite = W > 1 && writable;
    if (tid < NCV) {
        const int i = tid < NQK ? 4 * tid : 2 * K + 4 * (tid - NQK);   // head-local channel
        const int64_t gc = i < K ? h * K + i
                         : i < 2 * K ? HK + h * K + (i - K)
                                     : 2 * HK + static_cast<int64_t>(h) * V + vs * VT + (i - 2 * K);
        // taps front-padded to 4 (oldest first) and the 3 previous inputs a[.][0..2]
        float wt[4][4], a[4][3], bias[4] = {0.f, 0.f, 0.f, 0.f};
        if (W == 4) {   // one 8-byte load per channel
#pragma unroll
            for (int m = 0; m < 4; m++) {
                float f[4];
                bf16x4(__ldg(reinterpret_cast<const uint2 *>(tp.conv_w + (gc + m) * 4)), f);
#pragma unroll
                for (int k = 0; k < 4; k++) wt[m][k] = f[k];
            }
        } else {
#pragma unroll
            for (int m = 0; m < 4; m++)
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int src = k - (4 - W);
                    wt[m][k] = (W > 0 && src >= 0) ? bf16_to_f32(tp.conv_w[(gc + m) * W + src]) : 0.f;
                }
        }
#pragma unroll
        for (int m = 0; m < 4; m++)
#pragma unroll
            for (int r = 0; r < 3; r++) a[m][r] = 0.f;
        if (W > 0 && tp.conv_b) bf16x4(*reinterpret_cast<const uint2 *>(tp.conv_b + gc), bias);
        if (cstate) {
#pragma unroll
            for (int r = 0; r < 3; r++) {
                const int src = r - (4 - W);
                if (src >= 0) {
                    float f[4];
                    bf16x4(*reinterpret_cast<const uint2 *>(cstate + src * C + gc), f);
#pragma unroll
                    for (int m = 0; m < 4; m++) a[m][r] = f[m];
                }
            }
        }
        float *dst = i < K ? &s_q[0][i] : i < 2 * K ? &s_k[0][i - K] : &s_v[0][i - 2 * K];
        const int pitch = i < 2 * K ? K : VT;
        constexpr int XB = MAXT < 4 ? MAXT : 4;   // tokens whose inputs load together
        for (int t0 = 0; t0 < T; t0 += XB) {
            uint2 xr[XB];
#pragma unroll
            for (int u = 0; u < XB; u++)
                xr[u] = (t0 + u < T) ? *reinterpret_cast<const uint2 *>(p.qkv + (row0 + t0 + u) * p.ld_qkv + gc)
                                     : make_uint2(0u, 0u);
#pragma unroll
            for (int u = 0; u < XB; u++) {
                if (t0 + u < T) {
                    float x[4], y[4];
                    bf16x4(xr[u], x);
#pragma unroll
                    for (int m = 0; m < 4; m++) {
                        y[m] = x[m];
                        if (W > 0) {
                            y[m] = silu_fast(fmaf(wt[m][0], a[m][0], fmaf(wt[m][1], a[m][1],
                                             fmaf(wt[m][2], a[m][2], fmaf(wt[m][3], x[m], bias[m])))));
                            a[m][0] = a[m][1]; a[m][1] = a[m][2]; a[m][2] = x[m];
                        }
                    }
                    *reinterpret_cast<float4 *>(dst + (t0 + u) * pitch) = make_float4(y[0], y[1], y[2], y[3]);
                }
            }
        }
        if (cwrite) {   // the last W - 1 inputs, bit-exact (they are bf16 values)
#pragma unroll
            for (int r = 0; r < 3; r++) {
                const int d = r - (4 - W);
                if (d < 0) continue;
                uint2 bits;
                bits.x = (__float_as_uint(a[0][r]) >> 16) | (__float_as_uint(a[1][r]) & 0xffff0000u);
                bits.y = (__float_as_uint(a[2][r]) >> 16) | (__float_as_uint(a[3][r]) & 0xffff0000u);
                *reinterpret_cast<uint2 *>(&s_cnew[d][i]) = bits;   // stored after the cluster barrier
            }
        }
    } else if (tid < NI) {
        const int c = 4 * (tid - NCV);
        const float expA = expf(__ldg(p.A_log + h));
        const float4 dtb = p.dt_bias ? __ldg(reinterpret_cast<const float4 *>(p.dt_bias + h * K + c))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int t = 0; t < T; t++) {
            float gr[4];
            bf16x4(*reinterpret_cast<const uint2 *>(p.rg + (row0 + t) * p.ld_g + h * K + c), gr);
            *reinterpret_cast<float4 *>(&s_a[t][c]) = make_float4(
                __expf(gate_log_decay_fast(gr[0] + dtb.x, expA, p.has_lb, p.lb)),
                __expf(gate_log_decay_fast(gr[1] + dtb.y, expA, p.has_lb, p.lb)),
                __expf(gate_log_decay_fast(gr[2] + dtb.z, expA, p.has_lb, p.lb)),
                __expf(gate_log_decay_fast(gr[3] + dtb.w, expA, p.has_lb, p.lb)));
        }
    } else if (tp.gate != nullptr) {
#pragma unroll 4
        for (int idx = tid - NI; idx < T * VT; idx += 128 - NI) {
            const int t = idx / VT, j = idx - t * VT;
            const float gv = bf16_to_f32(tp.gate[(row0 + t) * tp.ld_gate + static_cast<int64_t>(h) * V + vs * VT + j]);
            s_gw[t][j] = __ldg(tp.norm_w + vs * VT + j) * sigmoid_fast(gv);
        }
    }
    if (kStage) {
        cp_async_wait_all();
#pragma unroll
        for (int i = 0; i < RPT; i++) S[i] = has_state ? s_stage[i][tid] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    // ---- per-token |q|^2, |k|^2, q.k (one warp per token), beta ----
    for (int t = warp; t < T; t += 4) {
        float qq = 0.f, kk = 0.f, qk = 0.f;
        for (int c = lane; c < K; c += 32) {
            const float q = s_q[t][c], k = s_k[t][c];
            qq += q * q; kk += k * k; qk += q * k;
        }
        qq = warp_sum(qq); kk = warp_sum(kk); qk = warp_sum(qk);
        if (lane == 0) {
            const float rq = p.scale * rsqrtf(qq + p.eps), rk = rsqrtf(kk + p.eps);
            s_tok[t][0] = rq;
            s_tok[t][1] = rk;
            s_tok[t][2] = qk * rq * rk;
            s_tok[t][3] = sigmoid_f(bf16_to_f32(p.rb[(row0 + t) * p.ld_beta + h]));
        }
    }
    __syncthreads();
    // ---- the recurrence, token by token ----
    const bool norm = tp.gate != nullptr;
#pragma unroll(MAXT == 1 ? 1 : 2)
    for (int t = 0; t < T; t++) {
        const int bb = t & 1;
        float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const int r = rg + 16 * i;
            const float al = s_a[t][r], kr = s_k[t][r], qr = s_q[t][r];
            S[i].x *= al; S[i].y *= al; S[i].z *= al; S[i].w *= al;
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
        float u[4], o[4];
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const int c = cg * 4 + jj;
            const float ks = (s_red[bb][0][0][c] + s_red[bb][1][0][c] + s_red[bb][2][0][c] + s_red[bb][3][0][c]) * rk;
            const float qs = (s_red[bb][0][1][c] + s_red[bb][1][1][c] + s_red[bb][2][1][c] + s_red[bb][3][1][c]) * rq;
            u[jj] = beta * (s_v[t][c] - ks);
            o[jj] = qs + qkh * u[jj];
        }
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const float kh = s_k[t][rg + 16 * i] * rk;
            S[i].x += kh * u[0]; S[i].y += kh * u[1]; S[i].z += kh * u[2]; S[i].w += kh * u[3];
        }
        if (rg == 0) {   // lanes 0..7 of warp 0
            *reinterpret_cast<float4 *>(&s_o[t][cg * 4]) = make_float4(o[0], o[1], o[2], o[3]);
            float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
            ss += __shfl_xor_sync(0xffu, ss, 1);
            ss += __shfl_xor_sync(0xffu, ss, 2);
            ss += __shfl_xor_sync(0xffu, ss, 4);
            if (cg == 0) s_ss[t] = ss;
        }
    }
    // ---- cluster barrier: every slice has read the q/k conv state and posted s_ss. The
    //      arrive releases only shared-memory writes and completed loads; the state stores
    //      go out between arrive and wait, so the release does not wait for them. ----
    const bool csync = VS > 1 && (norm || W > 1);
    if (csync) cluster_arrive_release();
    if (writable) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            *reinterpret_cast<float4 *>(tile + static_cast<int64_t>(rg + 16 * i) * V + j0) = S[i];
    }
    if (csync) cluster_wait();
    else __syncthreads();
    // ---- gated RMSNorm and bf16 stores of the slice's T x 32 outputs, two per thread ----
    for (int idx = tid; idx < T * (VT / 2); idx += 128) {
        const int t = idx / (VT / 2), j = 2 * (idx - t * (VT / 2));
        float o0 = s_o[t][j], o1 = s_o[t][j + 1];
        if (norm) {
            float ss = 0.f;
            if (VS > 1) {
                cgx::cluster_group cl = cgx::this_cluster();
#pragma unroll
                for (int r = 0; r < VS; r++) ss += cl.map_shared_rank(&s_ss[0], r)[t];
            } else {
                ss = s_ss[t];
            }
            const float rn = rsqrtf(ss * (1.f / V) + tp.norm_eps);
            o0 *= rn * s_gw[t][j];
            o1 *= rn * s_gw[t][j + 1];
        }
        *reinterpret_cast<uint32_t *>(p.out + (row0 + t) * p.ld_out + static_cast<int64_t>(h) * V + vs * VT + j) =
            pack_bf16x2(o0, o1);
    }
    // the new conv state: the q/k part by slice 0 (every slice has read the old one), the
    // slice's own v columns by the slice; 4 channels (8 bytes) per store
    if (cwrite) {
        constexpr int CW4 = (2 * K + VT) / 4, QK4 = 2 * K / 4;
        const int first = vs == 0 ? 0 : QK4;
        for (int d = 0; d < W - 1; d++) {
            for (int i4 = first + tid; i4 < CW4; i4 += 128) {
                const int i = 4 * i4;
                const int64_t gc = i < K ? h * K + i
                                 : i < 2 * K ? HK + h * K + (i - K)
                                             : 2 * HK + static_cast<int64_t>(h) * V + vs * VT + (i - 2 * K);
                *reinterpret_cast<uint2 *>(cstate + d * C + gc) = *reinterpret_cast<const uint2 *>(&s_cnew[d][i]);
            }
        }
    }
    // keep s_ss alive until every slice of the cluster has read it (the reads have returned
    // their values by now, so a relaxed arrive suffices)
    if (csync && norm) {
        cluster_arrive_relaxed();
        cluster_wait();
    }
}

template <int K, int V, int MAXT>
cudaError_t launch_fused_kv(const Params &p, const TailParams &tp, int T, int64_t num_entries,
                            cudaStream_t stream)
{
    const int64_t grid = num_entries * p.H * (V / 32);
    fused_kernel<K, V, MAXT><<<static_cast<unsigned>(grid), 128, 0, stream>>>(p, tp, T);
    return cudaGetLastError();
}

template <int K, int V>
cudaError_t launch_fused_t(const Params &p, const TailParams &tp, int T, int64_t num_entries,
                           cudaStream_t stream)
{
    if (T == 1) return launch_fused_kv<K, V, 1>(p, tp, T, num_entries, stream);
    if (T <= 8) return launch_fused_kv<K, V, 8>(p, tp, T, num_entries, stream);
    return launch_fused_kv<K, V, kFusedMaxT>(p, tp, T, num_entries, stream);
}

}  // namespace

cudaError_t launch_fused(const Params &p, const TailParams &tp, int K, int V, int T,
                         int64_t num_entries, cudaStream_t stream)
{
    if (num_entries <= 0) return cudaSuccess;
    if (T < 1 || T > kFusedMaxT) return cudaErrorInvalidValue;
#define KDA_FUSED_CASE(KK, VV) \
    if (K == KK && V == VV) return launch_fused_t<KK, VV>(p, tp, T, num_entries, stream);
    KDA_FUSED_CASE(32, 32) KDA_FUSED_CASE(32, 64) KDA_FUSED_CASE(32, 128)
    KDA_FUSED_CASE(64, 32) KDA_FUSED_CASE(64, 64) KDA_FUSED_CASE(64, 128)
    KDA_FUSED_CASE(128, 32) KDA_FUSED_CASE(128, 64) KDA_FUSED_CASE(128, 128)
#undef KDA_FUSED_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
