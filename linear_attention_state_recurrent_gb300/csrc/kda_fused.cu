// Fused layer tail for decode and spec-verify: short causal convolution -> KDA
// recurrence -> gated RMSNorm, in one kernel (the "spec conv, KDA recurrence, gated
// RMSNorm" run of the Kimi-K3 decode layer, vLLM PR #60683, section Purpose).
//
// One CTA of 128 threads owns one (entry, head) and its whole K x V state, in registers
// (see head_kernel). Owning the head makes both ends of the fusion local: the CTA is the
// only reader and writer of the head's conv state, and the RMS of o over V is a
// reduction inside the CTA. All T tokens' convolutions, gates, betas and q/k norms are
// computed up front in one parallel pass, whose loads are issued before the state copies;
// the sequential part is the state update with one barrier per token; the gated norm and
// the bf16 stores run once at the end over all T x V outputs.
#include "kda_common.cuh"
#include "kda_f32x2.cuh"
#include "kda_launch.h"
#include "kda_pdl.cuh"

namespace kda {

namespace {

constexpr int kFusedMaxT = 16;

// Fast-math activations (hardware exp2 and reciprocal): ~1e-6 relative error, far inside
// the bf16 output spacing. For y -> -inf the divisor overflows to inf and the result is 0.
__device__ __forceinline__ float silu_fast(float y) { return __fdividef(y, 1.f + __expf(-y)); }
__device__ __forceinline__ float sigmoid_fast(float y) { return __fdividef(1.f, 1.f + __expf(-y)); }

// four bf16 values (8 bytes) to fp32
__device__ __forceinline__ void bf16x4(uint2 u, float f[4])
{
    f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
}

// ---------------------------------------------------------------------------
// One CTA of 128 threads per (entry, head), the whole K x V state in registers: thread
// (rgp, cg) holds rows rgp*RPT .. rgp*RPT + RPT - 1 of columns 4cg .. 4cg + 3 (CG = V / 4
// column groups, NRG = 128 / CG row groups). At K = V = 128 that is 128 state registers
// per thread and three CTAs per SM, i.e. 192 KiB of state in flight per SM, with the
// convolution done once per head and the RMS of o summed inside the CTA. The state tile is
// staged in shared memory by cp.async while the channel pass runs.
// ---------------------------------------------------------------------------
// RB consecutive floats from shared memory (one 16-byte access when RB = 4)
template <int RB>
__device__ __forceinline__ void load_rows(const float *src, float *dst)
{
    if constexpr (RB == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(src);
        dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
    } else {
#pragma unroll
        for (int m = 0; m < RB; m++) dst[m] = src[m];
    }
}

template <int K, int V, int MAXT>
struct HeadSmem {
    static constexpr int CG = V / 4, NRG = 128 / CG;
    float a[MAXT][K];                 // alpha = e^g
    float k[MAXT][K];                 // conv'd k, raw; then k^ (normalised)
    float q[MAXT][K];                 // conv'd q, raw; then alpha q^
    float ka[MAXT][K];                // alpha k^
    float v[MAXT][V];                 // conv'd v
    float gw[MAXT][V];                // norm weight * sigmoid(gate)
    float o[MAXT][V];                 // o before the norm
    float red[MAXT == 1 ? 1 : 2][NRG][2][V];   // row-group partials of k^T S, q^T S
    float tok[MAXT][4];               // rq, rk, q^.k^, beta
    float ss[MAXT];                   // sum of o^2
};

template <int K, int V, int MAXT>
constexpr size_t head_smem_bytes()
{
    return (sizeof(HeadSmem<K, V, MAXT>) + 15) / 16 * 16 + static_cast<size_t>(K) * V * 4;
}

template <int K, int V, int MAXT>
__global__ void __launch_bounds__(128, MAXT == 1 ? 3 : (MAXT <= 8 ? 2 : 1))
head_kernel(Params p, TailParams tp, int T)
{
    constexpr int CG = V / 4, NRG = 128 / CG, RPT = K / NRG;
    constexpr int RB = RPT < 4 ? RPT : 4;   // rows read per shared-memory access
    static_assert(RPT % RB == 0, "row blocks");
    extern __shared__ __align__(16) unsigned char head_dsm[];
    HeadSmem<K, V, MAXT> &sm = *reinterpret_cast<HeadSmem<K, V, MAXT> *>(head_dsm);
    float4 *stage = reinterpret_cast<float4 *>(head_dsm + (sizeof(HeadSmem<K, V, MAXT>) + 15) / 16 * 16);

    pdl_wait_then_release();   // launched by launch_pdl: no global read before this
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % CG, rgp = tid / CG, r0 = rgp * RPT, j0 = 4 * cg;
    const int h = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.H));
    const int64_t e = blockIdx.x / static_cast<uint32_t>(p.H);
    const int64_t row0 = e * T;
    const int64_t slot = load_slot(p, e);
    if (slot >= p.num_slots) {                       // out of range: flag, zero outputs
        if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
        for (int idx = tid; idx < T * (V / 2); idx += 128) {
            const int t = idx / (V / 2), j = 2 * (idx - t * (V / 2));
            *reinterpret_cast<uint32_t *>(p.out + (row0 + t) * p.ld_out + static_cast<int64_t>(h) * V + j) = 0u;
        }
        return;
    }
    const bool has_state = slot >= 0;
    const bool writable = has_state && slot != p.null_slot;
    float *tile = has_state ? p.pool + slot * p.slot_stride + static_cast<int64_t>(h) * K * V : nullptr;
    // ---- channel pass: one item of 4 channels per thread: [0, K/2) q|k, [K/2, K/2 + V/4)
    //      v (conv; this CTA is the only reader of these channels' conv state), then the
    //      gates; afterwards every thread helps with norm weight * sigmoid(gate). The
    //      item's own loads are issued before the state copies, so they do not queue
    //      behind 64 KiB of state ----
    constexpr int NQK = K / 2, NCV = NQK + V / 4, NI = NCV + K / 4;
    static_assert(NI <= 128, "one channel item per thread");
    const int64_t HK = static_cast<int64_t>(p.H) * K;
    const int64_t C = 2 * HK + static_cast<int64_t>(p.H) * V;
    const int W = tp.conv_width;
    uint16_t *cstate = (W > 1 && has_state) ? tp.conv_state + slot * tp.conv_slot_stride : nullptr;
    const bool cwrite = W > 1 && writable;
    constexpr int XB = MAXT < 4 ? MAXT : 4;   // tokens whose inputs load together
    const int i = 4 * tid;                   // conv items: head-local channel in [0, 2K + V)
    const int64_t gc = i < K ? h * K + i
                     : i < 2 * K ? HK + h * K + (i - K)
                                 : 2 * HK + static_cast<int64_t>(h) * V + (i - 2 * K);
    const int c = 4 * (tid - NCV);           // gate items: first channel
    float wt[4][4], a[4][3], bias[4] = {0.f, 0.f, 0.f, 0.f};
    uint2 xr[XB];
    float4 dtb = make_float4(0.f, 0.f, 0.f, 0.f);
    float expA = 0.f;
    if (tid < NCV) {
        if (W == 4) {
#pragma unroll
            for (int m = 0; m < 4; m++) {
                float f[4];
                bf16x4(__ldg(reinterpret_cast<const uint2 *>(tp.conv_w + (gc + m) * 4)), f);
#pragma unroll
                for (int kk = 0; kk < 4; kk++) wt[m][kk] = f[kk];
            }
        } else {
#pragma unroll
            for (int m = 0; m < 4; m++)
#pragma unroll
                for (int kk = 0; kk < 4; kk++) {
                    const int src = kk - (4 - W);
                    wt[m][kk] = (W > 0 && src >= 0) ? bf16_to_f32(tp.conv_w[(gc + m) * W + src]) : 0.f;
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
#pragma unroll
        for (int u = 0; u < XB; u++)
            xr[u] = (u < T) ? *reinterpret_cast<const uint2 *>(p.qkv + (row0 + u) * p.ld_qkv + gc) : make_uint2(0u, 0u);
    } else if (tid < NI) {
        expA = expf(__ldg(p.A_log + h));
        if (p.dt_bias) dtb = __ldg(reinterpret_cast<const float4 *>(p.dt_bias + h * K + c));
#pragma unroll
        for (int u = 0; u < XB; u++)
            xr[u] = (u < T) ? *reinterpret_cast<const uint2 *>(p.rg + (row0 + u) * p.ld_g + h * K + c) : make_uint2(0u, 0u);
    }
    // the norm's gate values of this thread's outputs idx = tid + 128 m (a handful of
    // registers), also ahead of the state copies
    const bool norm = tp.gate != nullptr;
    constexpr int NGV = (MAXT * V + 127) / 128;
    uint16_t gbits[NGV];
    if (norm) {
#pragma unroll
        for (int m = 0; m < NGV; m++) {
            const int idx = tid + 128 * m, t = idx / V, j = idx - t * V;
            gbits[m] = (t < T) ? tp.gate[(row0 + t) * tp.ld_gate + static_cast<int64_t>(h) * V + j] : 0;
        }
    }
    if (has_state) {   // stage the tile: thread-private slots [RPT][128]
        const uint32_t st = static_cast<uint32_t>(__cvta_generic_to_shared(stage + tid));
#pragma unroll
        for (int ii = 0; ii < RPT; ii++)
            cp_async16(st + ii * 128 * 16, tile + static_cast<int64_t>(r0 + ii) * V + j0, true);
        cp_async_commit();
    }
    if (tid < NCV) {
        float *dst = i < K ? &sm.q[0][i] : i < 2 * K ? &sm.k[0][i - K] : &sm.v[0][i - 2 * K];
        const int pitch = i < 2 * K ? K : V;
        for (int t0 = 0; t0 < T; t0 += XB) {
            if (t0 > 0) {
#pragma unroll
                for (int u = 0; u < XB; u++)
                    xr[u] = (t0 + u < T) ? *reinterpret_cast<const uint2 *>(p.qkv + (row0 + t0 + u) * p.ld_qkv + gc)
                                         : make_uint2(0u, 0u);
            }
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
                *reinterpret_cast<uint2 *>(cstate + d * C + gc) = bits;
            }
        }
    } else if (tid < NI) {
        for (int t0 = 0; t0 < T; t0 += XB) {
            if (t0 > 0) {
#pragma unroll
                for (int u = 0; u < XB; u++)
                    xr[u] = (t0 + u < T) ? *reinterpret_cast<const uint2 *>(p.rg + (row0 + t0 + u) * p.ld_g + h * K + c)
                                         : make_uint2(0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < XB; u++) {
                if (t0 + u < T) {
                    float gr[4];
                    bf16x4(xr[u], gr);
                    *reinterpret_cast<float4 *>(&sm.a[t0 + u][c]) = make_float4(
                        __expf(gate_log_decay_fast(gr[0] + dtb.x, expA, p.has_lb, p.lb)),
                        __expf(gate_log_decay_fast(gr[1] + dtb.y, expA, p.has_lb, p.lb)),
                        __expf(gate_log_decay_fast(gr[2] + dtb.z, expA, p.has_lb, p.lb)),
                        __expf(gate_log_decay_fast(gr[3] + dtb.w, expA, p.has_lb, p.lb)));
                }
            }
        }
    }
    if (norm) {
#pragma unroll
        for (int m = 0; m < NGV; m++) {
            const int idx = tid + 128 * m, t = idx / V, j = idx - t * V;
            if (t < T) sm.gw[t][j] = __ldg(tp.norm_w + j) * sigmoid_fast(bf16_to_f32(gbits[m]));
        }
    }
    __syncthreads();
    // ---- per-token |q|^2, |k|^2, q.k (one warp per token), beta ----
    for (int t = warp; t < T; t += 4) {
        float qq = 0.f, kk = 0.f, qk = 0.f;
        for (int c = lane; c < K; c += 32) {
            const float q = sm.q[t][c], k = sm.k[t][c];
            qq += q * q; kk += k * k; qk += q * k;
        }
        qq = warp_sum(qq); kk = warp_sum(kk); qk = warp_sum(qk);
        if (lane == 0) {
            const float rq = p.scale * rsqrtf(qq + p.eps), rk = rsqrtf(kk + p.eps);
            sm.tok[t][0] = rq;
            sm.tok[t][1] = rk;
            sm.tok[t][2] = qk * rq * rk;
            sm.tok[t][3] = sigmoid_f(bf16_to_f32(p.rb[(row0 + t) * p.ld_beta + h]));
        }
    }
    __syncthreads();
    // ---- per-token row scalars of the state passes: k^ = k rk, alpha k^ and alpha q^ (the
    //      decayed key and query against the state before the token's decay) ----
    for (int idx = tid; idx < T * (K / 4); idx += 128) {
        const int t = idx / (K / 4), c = 4 * (idx - t * (K / 4));
        const float rq = sm.tok[t][0], rk = sm.tok[t][1];
        const float4 al = *reinterpret_cast<const float4 *>(&sm.a[t][c]);
        const float4 kr = *reinterpret_cast<const float4 *>(&sm.k[t][c]);
        const float4 qr = *reinterpret_cast<const float4 *>(&sm.q[t][c]);
        const float4 kh = make_float4(kr.x * rk, kr.y * rk, kr.z * rk, kr.w * rk);
        *reinterpret_cast<float4 *>(&sm.k[t][c]) = kh;
        *reinterpret_cast<float4 *>(&sm.ka[t][c]) = make_float4(kh.x * al.x, kh.y * al.y, kh.z * al.z, kh.w * al.w);
        *reinterpret_cast<float4 *>(&sm.q[t][c]) =
            make_float4(qr.x * rq * al.x, qr.y * rq * al.y, qr.z * rq * al.z, qr.w * rq * al.w);
    }
    float4 S[RPT];
    if (has_state) {
        cp_async_wait_all();
#pragma unroll
        for (int i = 0; i < RPT; i++) S[i] = stage[i * 128 + tid];
    } else {
#pragma unroll
        for (int i = 0; i < RPT; i++) S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    // ---- the recurrence, token by token (one barrier per token) ----
    for (int t = 0; t < T; t++) {
        const int bb = MAXT == 1 ? 0 : (t & 1);
        // partial (alpha k^)^T S and (alpha q^)^T S over this thread's rows, packed pairs of
        // columns, two accumulator sets (even and odd rows) to halve the dependency chains
        float2 ak[2][2], aq[2][2];
#pragma unroll
        for (int e2 = 0; e2 < 2; e2++)
#pragma unroll
            for (int hh = 0; hh < 2; hh++) { ak[e2][hh] = make_float2(0.f, 0.f); aq[e2][hh] = make_float2(0.f, 0.f); }
#pragma unroll
        for (int i4 = 0; i4 < RPT; i4 += RB) {
            float kav[4], qav[4];
            load_rows<RB>(&sm.ka[t][r0 + i4], kav);
            load_rows<RB>(&sm.q[t][r0 + i4], qav);
#pragma unroll
            for (int m = 0; m < RB; m++) {
                const float4 Sv = S[i4 + m];
                const float2 kk = make_float2(kav[m], kav[m]), qq = make_float2(qav[m], qav[m]);
                const int e2 = m & 1;
                ak[e2][0] = ffma2(kk, make_float2(Sv.x, Sv.y), ak[e2][0]);
                ak[e2][1] = ffma2(kk, make_float2(Sv.z, Sv.w), ak[e2][1]);
                aq[e2][0] = ffma2(qq, make_float2(Sv.x, Sv.y), aq[e2][0]);
                aq[e2][1] = ffma2(qq, make_float2(Sv.z, Sv.w), aq[e2][1]);
            }
        }
        const float2 pk01 = fadd2(ak[0][0], ak[1][0]), pk23 = fadd2(ak[0][1], ak[1][1]);
        const float2 pq01 = fadd2(aq[0][0], aq[1][0]), pq23 = fadd2(aq[0][1], aq[1][1]);
        const float4 pk = make_float4(pk01.x, pk01.y, pk23.x, pk23.y), pq = make_float4(pq01.x, pq01.y, pq23.x, pq23.y);
        *reinterpret_cast<float4 *>(&sm.red[bb][rgp][0][j0]) = pk;
        *reinterpret_cast<float4 *>(&sm.red[bb][rgp][1][j0]) = pq;
        __syncthreads();
        const float qkh = sm.tok[t][2], beta = sm.tok[t][3];
        float4 ks = make_float4(0.f, 0.f, 0.f, 0.f), qs = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int gI = 0; gI < NRG; gI++) {
            const float4 a = *reinterpret_cast<const float4 *>(&sm.red[bb][gI][0][j0]);
            const float4 b = *reinterpret_cast<const float4 *>(&sm.red[bb][gI][1][j0]);
            ks.x += a.x; ks.y += a.y; ks.z += a.z; ks.w += a.w;
            qs.x += b.x; qs.y += b.y; qs.z += b.z; qs.w += b.w;
        }
        const float4 v4 = *reinterpret_cast<const float4 *>(&sm.v[t][j0]);
        const float u0 = beta * (v4.x - ks.x), u1 = beta * (v4.y - ks.y);
        const float u2 = beta * (v4.z - ks.z), u3 = beta * (v4.w - ks.w);
        // S <- Diag(alpha) S + k^ u^T, packed pairs of columns
        const float2 u01 = make_float2(u0, u1), u23 = make_float2(u2, u3);
#pragma unroll
        for (int i4 = 0; i4 < RPT; i4 += RB) {
            float alv[4], khv[4];
            load_rows<RB>(&sm.a[t][r0 + i4], alv);
            load_rows<RB>(&sm.k[t][r0 + i4], khv);
#pragma unroll
            for (int m = 0; m < RB; m++) {
                float4 &Sv = S[i4 + m];
                const float2 aa = make_float2(alv[m], alv[m]), kk = make_float2(khv[m], khv[m]);
                const float2 lo = ffma2(aa, make_float2(Sv.x, Sv.y), fmul2(kk, u01));
                const float2 hi = ffma2(aa, make_float2(Sv.z, Sv.w), fmul2(kk, u23));
                Sv = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        if (rgp == 0) {   // the first CG threads (lanes of warp 0) own the outputs
            const float o0 = qs.x + qkh * u0, o1 = qs.y + qkh * u1;
            const float o2 = qs.z + qkh * u2, o3 = qs.w + qkh * u3;
            *reinterpret_cast<float4 *>(&sm.o[t][j0]) = make_float4(o0, o1, o2, o3);
            if (norm) {
                float ss = o0 * o0 + o1 * o1 + o2 * o2 + o3 * o3;
#pragma unroll
                for (int d = CG / 2; d > 0; d >>= 1)
                    ss += __shfl_xor_sync(CG == 32 ? 0xffffffffu : ((1u << CG) - 1u), ss, d);
                if (cg == 0) sm.ss[t] = ss;
            }
        }
    }
    if (writable) {
#pragma unroll
        for (int i = 0; i < RPT; i++)
            *reinterpret_cast<float4 *>(tile + static_cast<int64_t>(r0 + i) * V + j0) = S[i];
    }
    __syncthreads();
    // ---- gated RMSNorm and bf16 stores of all T x V outputs, two per thread ----
    for (int idx = tid; idx < T * (V / 2); idx += 128) {
        const int t = idx / (V / 2), j = 2 * (idx - t * (V / 2));
        float o0 = sm.o[t][j], o1 = sm.o[t][j + 1];
        if (norm) {
            const float rn = rsqrtf(sm.ss[t] * (1.f / V) + tp.norm_eps);
            o0 *= rn * sm.gw[t][j];
            o1 *= rn * sm.gw[t][j + 1];
        }
        *reinterpret_cast<uint32_t *>(p.out + (row0 + t) * p.ld_out + static_cast<int64_t>(h) * V + j) =
            pack_bf16x2(o0, o1);
    }
}

template <int K, int V, int MAXT>
cudaError_t launch_head_kv(const Params &p, const TailParams &tp, int T, int64_t num_entries,
                           cudaStream_t stream)
{
    constexpr size_t smem = head_smem_bytes<K, V, MAXT>();
    cudaError_t err = cudaFuncSetAttribute(head_kernel<K, V, MAXT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const int64_t grid = num_entries * p.H;
    return launch_pdl(head_kernel<K, V, MAXT>, dim3(static_cast<unsigned>(grid)), dim3(128), smem, stream, p, tp, T);
}

template <int K, int V>
cudaError_t launch_fused_t(const Params &p, const TailParams &tp, int T, int64_t num_entries,
                           cudaStream_t stream)
{
    if (T == 1) return launch_head_kv<K, V, 1>(p, tp, T, num_entries, stream);
    if (T <= 8) return launch_head_kv<K, V, 8>(p, tp, T, num_entries, stream);
    return launch_head_kv<K, V, kFusedMaxT>(p, tp, T, num_entries, stream);
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
