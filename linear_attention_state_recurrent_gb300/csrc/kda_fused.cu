// Fused layer tail for decode and spec-verify: short causal convolution -> KDA
// recurrence -> gated RMSNorm, in one kernel (the "spec conv, KDA recurrence, gated
// RMSNorm" run of the Kimi-K3 decode layer, vLLM PR #60683, section Purpose).
//
// One CTA owns one (entry, head) and all V columns of its state: VS = V / 32 groups of 128
// threads, each group the same 32-column tile layout as the recurrent kernel (thread
// (rg, cg) holds rows rg, rg + 16, ... of columns 4cg .. 4cg + 3). Owning the whole head in
// one CTA is what makes both ends local:
//   - the convolution of the head's q, k, v channels and the update of their conv state
//     happen in the one CTA that reads that state (no other CTA reads it);
//   - the RMS of o over V is a reduction across the CTA's groups.
// All T tokens' convolutions, gates, betas and q/k norms are computed up front in one
// parallel pass; the sequential part is the state update with one barrier per token; the
// gated norm and the bf16 stores run once at the end over all T x V outputs.
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {

namespace {

constexpr int kFusedMaxT = 16;

__device__ __forceinline__ float silu_f(float y) { return y / (1.f + expf(-y)); }

template <int K, int V>
struct __align__(16) FusedSmem {
    static constexpr int VS = V / 32;
    static constexpr int QW = K > V ? K : V;     // s_q rows also hold o (V values)
    float a[kFusedMaxT][K];                      // alpha = e^g of every token
    float k[kFusedMaxT][K];                      // conv'd k (raw, before the L2 norm)
    float q[kFusedMaxT][QW];                     // conv'd q, then o of the token
    float v[kFusedMaxT][V];                      // conv'd v
    float tok[kFusedMaxT][4];                    // rq, rk, q^.k^, beta
    float red[2][VS][4][2][32];                  // per-group warp partials of k^T S, q^T S
    float ss[kFusedMaxT][VS];                    // per-group sum of o^2
};

template <int K, int V>
__global__ void __launch_bounds__(128 * (V / 32), (V == 128 ? 2 : 1))
fused_kernel(Params p, TailParams tp, int T)
{
    constexpr int VS = V / 32, NT = 128 * VS, RPT = K / 16;
    __shared__ FusedSmem<K, V> sm;

    const int tid = threadIdx.x, lane = tid & 31;
    const int g = tid >> 7, gt = tid & 127, gwarp = gt >> 5, cg = gt & 7, rg = gt >> 3;
    const int h = static_cast<int>(blockIdx.x % p.H);
    const int64_t e = blockIdx.x / p.H;
    const int64_t row0 = e * T;
    const int j0 = g * 32 + cg * 4;
    const int64_t slot = load_slot(p, e);
    if (slot >= p.num_slots) {                        // out of range: flag, zero outputs
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
    if (has_state) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            S[i] = *reinterpret_cast<const float4 *>(tile + static_cast<int64_t>(rg + 16 * i) * V + j0);
    } else {
#pragma unroll
        for (int i = 0; i < RPT; i++) S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // ---- channel pass: conv of every q, k, v channel of the head, and every gate ----
    const int64_t HK = static_cast<int64_t>(p.H) * K;
    const int64_t C = 2 * HK + static_cast<int64_t>(p.H) * V;
    const int W = tp.conv_width;
    uint16_t *cstate = (W > 1 && has_state) ? tp.conv_state + slot * tp.conv_slot_stride : nullptr;
    const bool cwrite = W > 1 && writable;
    for (int i = tid; i < 3 * K + V; i += NT) {
        if (i < 2 * K + V) {
            const int64_t gc = i < K ? h * K + i
                             : i < 2 * K ? HK + h * K + (i - K)
                                         : 2 * HK + static_cast<int64_t>(h) * V + (i - 2 * K);
            // taps front-padded to 4 (oldest first) and the 3 previous inputs a[0..2]
            float wt[4] = {0.f, 0.f, 0.f, 0.f}, a[3] = {0.f, 0.f, 0.f}, bias = 0.f;
            if (W > 0) {
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int src = k - (4 - W);
                    if (src >= 0) wt[k] = bf16_to_f32(tp.conv_w[gc * W + src]);
                }
                if (tp.conv_b) bias = bf16_to_f32(tp.conv_b[gc]);
                if (cstate) {
#pragma unroll
                    for (int r = 0; r < 3; r++) {
                        const int src = r - (4 - W);
                        if (src >= 0) a[r] = bf16_to_f32(cstate[src * C + gc]);
                    }
                }
            }
            float *dst = i < K ? &sm.q[0][i] : i < 2 * K ? &sm.k[0][i - K] : &sm.v[0][i - 2 * K];
            const int pitch = i < K ? FusedSmem<K, V>::QW : i < 2 * K ? K : V;
            for (int t0 = 0; t0 < T; t0 += 4) {
                float x[4];
#pragma unroll
                for (int u = 0; u < 4; u++)
                    x[u] = (t0 + u < T) ? bf16_to_f32(p.qkv[(row0 + t0 + u) * p.ld_qkv + gc]) : 0.f;
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    if (t0 + u < T) {
                        float y = x[u];
                        if (W > 0) {
                            y = fmaf(wt[0], a[0], fmaf(wt[1], a[1], fmaf(wt[2], a[2], fmaf(wt[3], x[u], bias))));
                            y = silu_f(y);
                            a[0] = a[1]; a[1] = a[2]; a[2] = x[u];
                        }
                        dst[(t0 + u) * pitch] = y;
                    }
                }
            }
            if (cwrite) {   // the last W - 1 inputs, bit-exact (they are bf16 values)
#pragma unroll
                for (int r = 0; r < 3; r++) {
                    const int d = r - (4 - W);
                    if (d >= 0) cstate[d * C + gc] = static_cast<uint16_t>(__float_as_uint(a[r]) >> 16);
                }
            }
        } else {
            const int c = i - (2 * K + V);
            const float expA = expf(__ldg(p.A_log + h));
            const float dtb = p.dt_bias ? __ldg(p.dt_bias + h * K + c) : 0.f;
            for (int t = 0; t < T; t++) {
                const float graw = bf16_to_f32(p.rg[(row0 + t) * p.ld_g + h * K + c]);
                sm.a[t][c] = expf(gate_log_decay(graw + dtb, expA, p.has_lb, p.lb));
            }
        }
    }
    __syncthreads();
    // ---- per-token |q|^2, |k|^2, q.k (NT / kFusedMaxT threads per token), beta ----
    {
        constexpr int TPT = NT / kFusedMaxT;
        const int t = tid / TPT, part = tid % TPT;
        float qq = 0.f, kk = 0.f, qk = 0.f;
        if (t < T) {
            for (int c = part; c < K; c += TPT) {
                const float q = sm.q[t][c], k = sm.k[t][c];
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
            sm.tok[t][0] = rq;
            sm.tok[t][1] = rk;
            sm.tok[t][2] = qk * rq * rk;
        }
        if (tid < T) sm.tok[tid][3] = sigmoid_f(bf16_to_f32(p.rb[(row0 + tid) * p.ld_beta + h]));
    }
    __syncthreads();
    // ---- the recurrence, token by token ----
    const bool norm = tp.gate != nullptr;
    for (int t = 0; t < T; t++) {
        const int bb = t & 1;
        float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const int r = rg + 16 * i;
            const float al = sm.a[t][r], kr = sm.k[t][r], qr = sm.q[t][r];
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
                sm.red[bb][g][gwarp][0][cg * 4 + jj] = pk[jj];
                sm.red[bb][g][gwarp][1][cg * 4 + jj] = pq[jj];
            }
        }
        __syncthreads();
        const float rq = sm.tok[t][0], rk = sm.tok[t][1], qkh = sm.tok[t][2], beta = sm.tok[t][3];
        float u[4], o[4];
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const int c = cg * 4 + jj;
            const float ks = (sm.red[bb][g][0][0][c] + sm.red[bb][g][1][0][c] +
                              sm.red[bb][g][2][0][c] + sm.red[bb][g][3][0][c]) * rk;
            const float qs = (sm.red[bb][g][0][1][c] + sm.red[bb][g][1][1][c] +
                              sm.red[bb][g][2][1][c] + sm.red[bb][g][3][1][c]) * rq;
            u[jj] = beta * (sm.v[t][j0 + jj] - ks);
            o[jj] = qs + qkh * u[jj];
        }
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const float kh = sm.k[t][rg + 16 * i] * rk;
            S[i].x += kh * u[0]; S[i].y += kh * u[1]; S[i].z += kh * u[2]; S[i].w += kh * u[3];
        }
        if (rg == 0) {   // lanes 0..7 of the group's first warp
            *reinterpret_cast<float4 *>(&sm.q[t][j0]) = make_float4(o[0], o[1], o[2], o[3]);
            if (norm) {
                float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
                ss += __shfl_xor_sync(0xffu, ss, 1);
                ss += __shfl_xor_sync(0xffu, ss, 2);
                ss += __shfl_xor_sync(0xffu, ss, 4);
                if (cg == 0) sm.ss[t][g] = ss;
            }
        }
    }
    if (writable) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            *reinterpret_cast<float4 *>(tile + static_cast<int64_t>(rg + 16 * i) * V + j0) = S[i];
    }
    __syncthreads();
    // ---- gated RMSNorm and bf16 stores of all T x V outputs, two columns per thread ----
    for (int idx = tid; idx < T * (V / 2); idx += NT) {
        const int t = idx / (V / 2), j = 2 * (idx - t * (V / 2));
        float o0 = sm.q[t][j], o1 = sm.q[t][j + 1];
        if (norm) {
            float ss = 0.f;
#pragma unroll
            for (int gg = 0; gg < VS; gg++) ss += sm.ss[t][gg];
            const float r = rsqrtf(ss * (1.f / V) + tp.norm_eps);
            const uint32_t gb = *reinterpret_cast<const uint32_t *>(
                tp.gate + (row0 + t) * tp.ld_gate + static_cast<int64_t>(h) * V + j);
            o0 *= r * __ldg(tp.norm_w + j) * sigmoid_f(bf16_to_f32(static_cast<uint16_t>(gb & 0xffffu)));
            o1 *= r * __ldg(tp.norm_w + j + 1) * sigmoid_f(bf16_to_f32(static_cast<uint16_t>(gb >> 16)));
        }
        *reinterpret_cast<uint32_t *>(p.out + (row0 + t) * p.ld_out + static_cast<int64_t>(h) * V + j) =
            static_cast<uint32_t>(f32_to_bf16(o0)) | (static_cast<uint32_t>(f32_to_bf16(o1)) << 16);
    }
}

template <int K, int V>
cudaError_t launch_fused_kv(const Params &p, const TailParams &tp, int T, int64_t num_entries,
                            cudaStream_t stream)
{
    const int64_t grid = num_entries * p.H;
    fused_kernel<K, V><<<static_cast<unsigned>(grid), 128 * (V / 32), 0, stream>>>(p, tp, T);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused(const Params &p, const TailParams &tp, int K, int V, int T,
                         int64_t num_entries, cudaStream_t stream)
{
    if (num_entries <= 0) return cudaSuccess;
    if (T < 1 || T > kFusedMaxT) return cudaErrorInvalidValue;
#define KDA_FUSED_CASE(KK, VV) \
    if (K == KK && V == VV) return launch_fused_kv<KK, VV>(p, tp, T, num_entries, stream);
    KDA_FUSED_CASE(32, 32) KDA_FUSED_CASE(32, 64) KDA_FUSED_CASE(32, 128)
    KDA_FUSED_CASE(64, 32) KDA_FUSED_CASE(64, 64) KDA_FUSED_CASE(64, 128)
    KDA_FUSED_CASE(128, 32) KDA_FUSED_CASE(128, 64) KDA_FUSED_CASE(128, 128)
#undef KDA_FUSED_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
