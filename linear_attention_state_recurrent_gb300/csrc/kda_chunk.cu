// Chunked varlen prefill on tcgen05 tensor cores (K = V = 128, chunk C = 64).
//
// The chunked (WY) form of the gated delta rule (chunk_kda_with_fused_gate with its
// recompute_w_u step, vLLM PR #50649, section Purpose). For one (sequence, head) and a
// chunk of n <= 64 rows with in-chunk cumulative log-decay b_r = sum_{i<=r} g_i
// (per channel) and Gamma_r = e^{b_r}:
//   A[r,i]   = beta_r sum_c k^_r k^_i e^{b_r - b_i}   (i < r)    T = (I + A)^-1
//   Aqk[r,i] = sum_c q^_r k^_i e^{b_r - b_i}          (i <= r)
//   U   = T diag(beta) (V - (K^ * Gamma) S0)
//   O   = (Q^ * Gamma) S0 + Aqk U
//   S_C = Diag(e^{b_last}) S0 + (K^ * e^{b_last - b})^T U
// (U = U~ - W S0 with W = T diag(beta)(K^ * Gamma) and U~ = T diag(beta) V, folded into
// one product.) The state is kept transposed in tensor memory (lane = value column j,
// column = key channel c), so every product has the 128-long V dimension as MMA M:
//   P    = S^T [K^G; Q^G]^T            M=128 N=128 K=128  fp16   -> (K^G S)^T | (Q^G S)^T
//   U^T  = (beta Y)^T T^T,  Y = V - K^G S   M=128 N=64  K=64   fp16
//   [O^T | S^T] += U^T [Aqk; Kd^T]^T   M=128 N=192 K=64   fp16   (S^T pre-scaled by e^{b_last})
// The decay-weighted Gram matrices are split into 16-row blocks. Off-diagonal blocks
// use the start of the row block as reference point (both factors <= 1, fp16):
//   X_off = [K^e; Q^e] [B_1; B_2; B_3]^T     M=128 N=96 K=128 fp16
// and the diagonal blocks use the middle row of the block, whose factors can reach
// e^{40}, in tf32:
//   X_diag = [K^L; Q^L] (K^R)^T              M=128 N=64 K=128 tf32
// A chunk in which some channel decays by more than 40 nats within half a block
// (8 rows) computes its diagonal blocks pairwise on CUDA cores instead.
//
// fp16 (11-bit significand, round to nearest) carries the same precision as tf32
// with round to nearest; bf16 operands would exceed the 2e-3 relative error bar.
//
// One CTA (256 threads) owns one (sequence, head) chain; CTAs are ordered longest
// sequence first.
#include <algorithm>
#include <numeric>
#include <vector>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_tc.cuh"

namespace kda {
namespace chunk {

constexpr int C = 64;
constexpr int KD = 128;
constexpr int VD = 128;
constexpr int NT = 256;
constexpr float kHalfSpan = 40.f;   // largest in-half-block decay served by the tf32 path
constexpr int kMaxOrder = 1024;

// ---- shared memory map (bytes) ----
constexpr uint32_t SM_OFFA = 0;            // fp16 [128 x 128] K^e rows 0..63, Q^e rows 64..127
constexpr uint32_t SM_OFFB = 32768;        // fp16 [96 x 128]  B_1 (16 rows), B_2 (32), B_3 (48)
constexpr uint32_t SM_DIAGA = 57344;       // tf32 [128 x 128] K^L, Q^L
constexpr uint32_t SM_DIAGB = 122880;      // tf32 [64 x 128]  K^R
constexpr uint32_t SM_PB = 155648;         // fp16 [128 x 128] K^G rows 0..63, Q^G rows 64..127
constexpr uint32_t SM_TB = 188416;         // fp16 [64 x 64]   T
constexpr uint32_t SM_SB = 196608;         // fp16 [192 x 64]  Aqk rows 0..63, Kd^T rows 64..191
constexpr uint32_t SM_SB_KD = SM_SB + 8192;
constexpr uint32_t SM_TAB = SM_TB;         // phase A only: per (block, channel) constants (14336 B)
constexpr uint32_t SM_TOT = 221184;        // fp32 [8][128] per-warp sums of g, then prefixes P_w
constexpr uint32_t SM_GC = SM_TOT + 4096;  // fp32 [128] e^{b_last}
constexpr uint32_t SM_BLAST = SM_GC + 512; // fp32 [128] b_last
constexpr uint32_t SM_BETA = SM_BLAST + 512;  // fp32 [64]
constexpr uint32_t SM_DTB = SM_BETA + 256;    // fp32 [128] dt_bias of this head
constexpr uint32_t SM_MBAR = SM_DTB + 512;
constexpr uint32_t SM_TMEMP = SM_MBAR + 8;
constexpr uint32_t SMEM_BYTES = SM_TMEMP + 8;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(SM_TAB + 4 * 7 * 128 * 4 <= SM_SB_KD, "constants table overlaps Kd^T");
// phase C aliases
constexpr uint32_t SM_AMAT = SM_OFFA;          // fp32 [64][68]
constexpr uint32_t SM_XTMP = SM_OFFA + 17408;  // fp32 scratch (<= 15360 B)
constexpr uint32_t SM_TMAT = SM_OFFB;          // fp32 [64][68]
constexpr int AP = 68;                         // fp32 row pitch of AMAT / TMAT
// phase D aliases
constexpr uint32_t SM_SA = SM_DIAGA;           // fp16 [128 x 128] S^T
constexpr uint32_t SM_YA = SM_DIAGA + 32768;   // fp16 [128 x 64]  (beta Y)^T
constexpr uint32_t SM_UA = SM_DIAGA + 49152;   // fp16 [128 x 64]  U^T
// flagged-chunk stash (fp32 [64][128] each)
constexpr uint32_t SM_STK = SM_DIAGA;
constexpr uint32_t SM_STQ = SM_DIAGA + 32768;
constexpr uint32_t SM_STB = SM_DIAGB;

// ---- tensor memory columns ----
constexpr uint32_t TM_P = 0;      // [0,64) K^G S -> U ; [64,128) O
constexpr uint32_t TM_S = 128;    // S^T (128 columns)
constexpr uint32_t TM_XOFF = 256; // 96 columns
constexpr uint32_t TM_XDIAG = 352;// 64 columns

// stride byte offsets of the operand tiles
constexpr uint32_t SBO128_F16 = 128 * 2 * 8;  // K = 128 fp16
constexpr uint32_t SBO128_TF32 = 128 * 4 * 8; // K = 128 tf32
constexpr uint32_t SBO64_F16 = 64 * 2 * 8;    // K = 64 fp16

struct Args {
    Params p;
    const int32_t *cu;
    int64_t entry_base;
    int32_t num_seqs;
    int32_t order_n;
    int32_t order[kMaxOrder];
};

// constants table entry (block s, constant k, channel c), laid out so that the four
// 32-channel quarters of one 4-channel group are adjacent (conflict-free LDS.128)
__device__ __forceinline__ uint32_t tab_off(int s, int k, int c)
{
    const int q = c >> 5, g = (c & 31) >> 2, e = c & 3;
    return static_cast<uint32_t>(((((s * 7 + k) * 8 + g) * 4 + q) * 4 + e) * 4);
}

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" :: "r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint16_t f16_bits(float x)
{
    uint16_t h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return h;
}

__device__ __forceinline__ void unpack_bf16x8(uint4 u, float *f)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// 8 floats -> 8 fp16 in one 16-byte chunk
__device__ __forceinline__ uint4 pack8_f16(const float *v)
{
    return make_uint4(tc::pack_f16x2(v[0], v[1]), tc::pack_f16x2(v[2], v[3]),
                      tc::pack_f16x2(v[4], v[5]), tc::pack_f16x2(v[6], v[7]));
}

__device__ __forceinline__ uint4 pack4_tf32(const float *v)
{
    return make_uint4(tc::to_tf32(v[0]), tc::to_tf32(v[1]), tc::to_tf32(v[2]), tc::to_tf32(v[3]));
}

// ---------------------------------------------------------------------------
// Phase C: T = (I + A)^-1 for the strictly lower 64x64 A in AMAT (fp32, pitch AP),
// by 16x16 diagonal-block inverses and two levels of block doubling.
// ---------------------------------------------------------------------------
__device__ void solve_T(unsigned char *smem, int tid)
{
    float *A = reinterpret_cast<float *>(smem + SM_AMAT);
    float *T = reinterpret_cast<float *>(smem + SM_TMAT);
    float *X = reinterpret_cast<float *>(smem + SM_XTMP);
    // level 1: columns of the four 16x16 diagonal inverses
    if (tid < 64) {
        const int s = tid >> 4, j = tid & 15, o = 16 * s;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < r; m++) acc -= A[(o + r) * AP + o + m] * t[m];
            t[r] = (r < j) ? 0.f : acc;
        }
#pragma unroll
        for (int r = 0; r < 16; r++) T[(o + r) * AP + o + j] = t[r];
    }
    __syncthreads();
    // level 2: within each 32-block p, X = A_10 T_00 then T_10 = -T_11 X (16x16)
    {
        const int p = tid >> 7, r = (tid >> 3) & 15, j = (tid & 7) * 2, o = 32 * p;
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m++) {
            const float a = A[(o + 16 + r) * AP + o + m];
            x0 += a * T[(o + m) * AP + o + j];
            x1 += a * T[(o + m) * AP + o + j + 1];
        }
        X[(p * 16 + r) * 17 + j] = x0;
        X[(p * 16 + r) * 17 + j + 1] = x1;
    }
    __syncthreads();
    {
        const int p = tid >> 7, r = (tid >> 3) & 15, j = (tid & 7) * 2, o = 32 * p;
        float y0 = 0.f, y1 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m++) {
            const float t = (m <= r) ? T[(o + 16 + r) * AP + o + 16 + m] : 0.f;
            y0 += t * X[(p * 16 + m) * 17 + j];
            y1 += t * X[(p * 16 + m) * 17 + j + 1];
        }
        T[(o + 16 + r) * AP + o + j] = -y0;
        T[(o + 16 + r) * AP + o + j + 1] = -y1;
    }
    __syncthreads();
    // level 3: X = A_ba T_a (32x32), T_ba = -T_b X
    {
        const int r = tid >> 3, j = (tid & 7) * 4;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int m = 0; m < 32; m++) {
            const float a = A[(32 + r) * AP + m];
#pragma unroll
            for (int u = 0; u < 4; u++) x[u] += (m >= j + u) ? a * T[m * AP + j + u] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; u++) X[r * 36 + j + u] = x[u];
    }
    __syncthreads();
    {
        const int r = tid >> 3, j = (tid & 7) * 4;
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int m = 0; m < 32; m++) {
            const float t = (m <= r) ? T[(32 + r) * AP + 32 + m] : 0.f;
#pragma unroll
            for (int u = 0; u < 4; u++) y[u] += t * X[m * 36 + j + u];
        }
#pragma unroll
        for (int u = 0; u < 4; u++) T[(32 + r) * AP + j + u] = -y[u];
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// Phase C1 helper: assemble one row of A (K rows) or Aqk (Q rows) from the off-
// diagonal and diagonal TMEM results. HALF 0: rows 0..31, HALF 1: rows 32..63.
// ---------------------------------------------------------------------------
template <int HALF>
__device__ void assemble_rows(unsigned char *smem, uint32_t tmem_lane, int warp, int lane,
                              bool flagged)
{
    constexpr int NXO = HALF == 0 ? 16 : 80;         // off-diagonal columns this warp reads
    constexpr int XO0 = HALF == 0 ? 0 : 16;          // first off-diagonal column
    const bool qpart = warp >= 2;
    const int r = 32 * HALF + lane;                  // chunk row
    const int s = r >> 4;                            // row block
    float xo[NXO], xd[32];
#pragma unroll
    for (int cc = 0; cc < NXO; cc += 16) {
        float v[16];
        tc::tmem_ld16(tmem_lane + TM_XOFF + XO0 + cc, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; u++) xo[cc + u] = v[u];
    }
    if (!flagged) {
#pragma unroll
        for (int cc = 0; cc < 32; cc += 16) {
            float v[16];
            tc::tmem_ld16(tmem_lane + TM_XDIAG + 32 * HALF + cc, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; u++) xd[cc + u] = v[u];
        }
    } else {
        // pairwise in fp32 from the stash: xd[i - 32*HALF] for i in row r's block
        const float *stk = reinterpret_cast<const float *>(smem + SM_STK);
        const float *stq = reinterpret_cast<const float *>(smem + SM_STQ);
        const float *stb = reinterpret_cast<const float *>(smem + SM_STB);
        const float *xr = (qpart ? stq : stk) + r * KD;
        const float *br = stb + r * KD;
#pragma unroll
        for (int u = 0; u < 32; u++) {
            const int i = 32 * HALF + u;
            float acc = 0.f;
            if ((i >> 4) == s && i <= r) {
                const float *ki = stk + i * KD;
                const float *bi = stb + i * KD;
                for (int c = 0; c < KD; c++) acc += xr[c] * ki[c] * __expf(br[c] - bi[c]);
            }
            xd[u] = acc;
        }
    }
    const float beta = reinterpret_cast<const float *>(smem + SM_BETA)[r];
    float a[64];
#pragma unroll
    for (int i = 0; i < 64; i++) {
        float v = 0.f;
        const bool diag_ok = qpart ? (i <= r) : (i < r);
        if (HALF == 0) {
            if (i < 16) v = (s == 1) ? xo[i] : (diag_ok ? xd[i] : 0.f);
            else if (i < 32) v = (s == 1 && diag_ok) ? xd[i] : 0.f;
        } else {
            if (i < 32) v = (s == 2) ? xo[i] : xo[32 + i];
            else if (i < 48) v = (s == 3) ? xo[32 + i] : (diag_ok ? xd[i - 32] : 0.f);
            else v = (s == 3 && diag_ok) ? xd[i - 32] : 0.f;
        }
        a[i] = qpart ? v : v * beta;
    }
    if (!qpart) {
        float *Arow = reinterpret_cast<float *>(smem + SM_AMAT) + r * AP;
#pragma unroll
        for (int i = 0; i < 64; i += 4) *reinterpret_cast<float4 *>(Arow + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
    } else {
        const uint32_t base = tc::smem_addr(smem + SM_SB);
#pragma unroll
        for (int i = 0; i < 64; i += 8) st_shared_u4(base + tc::core_offset(r, i, 64, 2), pack8_f16(a + i));
    }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 1) chunk_kernel(const __grid_constant__ Args args)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    const Params &p = args.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int rank = blockIdx.x / H, h = blockIdx.x % H;
    const int sidx = args.order_n ? args.order[rank] : rank;
    const int64_t e = args.entry_base + sidx;
    const int64_t row0 = args.cu[e], row1 = args.cu[e + 1];
    if (row1 <= row0) return;
    const int64_t slot = load_slot(p, e);
    if (slot >= p.num_slots) {
        if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
        for (int64_t t = row0 + (tid >> 6); t < row1; t += NT / 64) {
            uint32_t *o = reinterpret_cast<uint32_t *>(p.out + t * p.ld_out + static_cast<int64_t>(h) * VD);
            o[tid & 63] = 0u;
        }
        return;
    }
    const bool has_state = slot >= 0;
    const bool writable = has_state && slot != p.null_slot;
    float *tile = has_state ? p.pool + slot * p.slot_stride + static_cast<int64_t>(h) * KD * VD : nullptr;
    const int64_t HK = static_cast<int64_t>(H) * KD;

    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t mbar = sbase + SM_MBAR;
    if (tid == 0) tc::mbar_init(mbar, 1);
    if (tid < KD) reinterpret_cast<float *>(smem + SM_DTB)[tid] = p.dt_bias ? p.dt_bias[h * KD + tid] : 0.f;
    if (warp == 0) tc::tmem_alloc<512>(sbase + SM_TMEMP);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TMEMP);
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);  // this warp's lanes
    uint32_t phase = 0;
    bool ok = true;

    // thread roles
    const int jv = 32 * (warp & 3) + lane;   // phase D: value column (TMEM lane)
    const int hv = warp >> 2;                // phase D: which half of the columns / rows
    const int ir = lane & 7, iq = lane >> 3; // phase A: row within warp, channel quarter
    const int ra = 8 * warp + ir;            // phase A: chunk row

    // ---- S0 -> TMEM (S^T: lane j, column c) ----
    {
#pragma unroll
        for (int cc = 0; cc < 64; cc += 16) {
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; u++)
                v[u] = has_state ? tile[static_cast<int64_t>(64 * hv + cc + u) * VD + jv] : 0.f;
            tc::tmem_st16(tlane + TM_S + 64 * hv + cc, v);
        }
        tc::tmem_st_wait();
    }

    const float expA = __expf(p.A_log[h]);
    const float *dtb_s = reinterpret_cast<const float *>(smem + SM_DTB);

    for (int64_t c0 = row0; c0 < row1; c0 += C) {
        const int n = static_cast<int>((row1 - c0) < C ? (row1 - c0) : C);

        // ================= Phase A: gate, norms, cumulative decay, operands =================
        float qv[32], kv[32], bv[32];
        float beta_r = 0.f;
        const bool valid = ra < n;
        {
            const int64_t row = c0 + ra;
            if (valid) {
                const uint4 *qp = reinterpret_cast<const uint4 *>(p.qkv + row * p.ld_qkv + h * KD + 32 * iq);
                const uint4 *kp = reinterpret_cast<const uint4 *>(p.qkv + row * p.ld_qkv + HK + h * KD + 32 * iq);
                const uint4 *gp = reinterpret_cast<const uint4 *>(p.rg + row * p.ld_g + h * KD + 32 * iq);
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    unpack_bf16x8(qp[u], qv + 8 * u);
                    unpack_bf16x8(kp[u], kv + 8 * u);
                    unpack_bf16x8(gp[u], bv + 8 * u);
                }
                beta_r = sigmoid_f(bf16_to_f32(p.rb[row * p.ld_beta + h]));
            } else {
#pragma unroll
                for (int u = 0; u < 32; u++) { qv[u] = 0.f; kv[u] = 0.f; bv[u] = 0.f; }
            }
        }
        // gate (g <= 0; zero on padding rows) and row norms
        float qq = 0.f, kk = 0.f;
#pragma unroll
        for (int u = 0; u < 32; u++) {
            bv[u] = valid ? gate_log_decay(bv[u] + dtb_s[32 * iq + u], expA, p.has_lb, p.lb) : 0.f;
            qq += qv[u] * qv[u];
            kk += kv[u] * kv[u];
        }
        qq += __shfl_xor_sync(0xffffffffu, qq, 8);
        qq += __shfl_xor_sync(0xffffffffu, qq, 16);
        kk += __shfl_xor_sync(0xffffffffu, kk, 8);
        kk += __shfl_xor_sync(0xffffffffu, kk, 16);
        {
            const float rq = p.scale * rsqrtf(qq + p.eps), rk = rsqrtf(kk + p.eps);
#pragma unroll
            for (int u = 0; u < 32; u++) { qv[u] *= rq; kv[u] *= rk; }
        }
        // in-warp inclusive scan over the 8 rows (lanes ir = 0..7 of the same quarter)
#pragma unroll
        for (int u = 0; u < 32; u++) {
            float v = bv[u];
#pragma unroll
            for (int d = 1; d < 8; d <<= 1) {
                const float t = __shfl_up_sync(0xffffffffu, v, d, 8);
                if (ir >= d) v += t;
            }
            bv[u] = v;
        }
        float *tot = reinterpret_cast<float *>(smem + SM_TOT);
        if (ir == 7) {
#pragma unroll
            for (int u = 0; u < 32; u += 4)
                *reinterpret_cast<float4 *>(tot + warp * KD + 32 * iq + u) = make_float4(bv[u], bv[u + 1], bv[u + 2], bv[u + 3]);
        }
        if (iq == 0) reinterpret_cast<float *>(smem + SM_BETA)[ra] = beta_r;
        __syncthreads();

        // per-channel constants (threads 0..127, one channel each)
        int flag = 0;
        if (tid < KD) {
            const int c = tid;
            float T[8], E[8], P[9];
            P[0] = 0.f;
#pragma unroll
            for (int w = 0; w < 8; w++) {
                T[w] = tot[w * KD + c];
                P[w + 1] = P[w] + T[w];
                E[w] = __expf(T[w]);
                flag |= (T[w] < -kHalfSpan) ? 1 : 0;
            }
#pragma unroll
            for (int s = 0; s < 4; s++) {
                float G = 1.f, Hh = 1.f;
#pragma unroll
                for (int w = 0; w < 8; w++) {
                    if (w < 2 * s) G *= E[w];
                    if (w >= 2 * s + 2) Hh *= E[w];
                }
                const float D1 = (s <= 2) ? E[2 * s + 2] * E[2 * s + 3] : 0.f;
                const float D12 = (s <= 1) ? D1 * E[2 * s + 4] * E[2 * s + 5] : 0.f;
                const float vals[7] = {T[2 * s], E[2 * s], E[2 * s + 1], G, Hh, D1, D12};
#pragma unroll
                for (int k = 0; k < 7; k++) *reinterpret_cast<float *>(smem + SM_TAB + tab_off(s, k, c)) = vals[k];
            }
            float gc = 1.f;
#pragma unroll
            for (int w = 0; w < 8; w++) gc *= E[w];
            reinterpret_cast<float *>(smem + SM_GC)[c] = gc;
            reinterpret_cast<float *>(smem + SM_BLAST)[c] = P[8];
#pragma unroll
            for (int w = 0; w < 8; w++) tot[w * KD + c] = P[w];  // prefixes replace the sums
        }
        const bool flagged = __syncthreads_or(flag) != 0;

        {
            const int s = warp >> 1, hf = warp & 1;
            const uint32_t offa = sbase + SM_OFFA, offb = sbase + SM_OFFB, diaga = sbase + SM_DIAGA,
                           diagb = sbase + SM_DIAGB, pb = sbase + SM_PB, sbkd = sbase + SM_SB_KD;
            const float *Pw = reinterpret_cast<const float *>(smem + SM_TOT);
            const float *blast = reinterpret_cast<const float *>(smem + SM_BLAST);
#pragma unroll
            for (int g8 = 0; g8 < 4; g8++) {          // 8 channels at a time
                float ek[8], eq[8], pk[8], pq[8], lk[8], lq[8], rkv[8], kd[8], ob[3][8];
#pragma unroll
                for (int half4 = 0; half4 < 2; half4++) {
                    const int cbase = 32 * iq + 8 * g8 + 4 * half4;   // first of 4 channels
                    const float4 sh = ld_shared_f4(sbase + SM_TAB + tab_off(s, 0, cbase));
                    const float4 X = ld_shared_f4(sbase + SM_TAB + tab_off(s, 1, cbase));
                    const float4 Y = ld_shared_f4(sbase + SM_TAB + tab_off(s, 2, cbase));
                    const float4 G = ld_shared_f4(sbase + SM_TAB + tab_off(s, 3, cbase));
                    const float4 Hh = ld_shared_f4(sbase + SM_TAB + tab_off(s, 4, cbase));
                    const float4 D1 = ld_shared_f4(sbase + SM_TAB + tab_off(s, 5, cbase));
                    const float4 D12 = ld_shared_f4(sbase + SM_TAB + tab_off(s, 6, cbase));
                    const float shv[4] = {sh.x, sh.y, sh.z, sh.w}, Xv[4] = {X.x, X.y, X.z, X.w},
                                Yv[4] = {Y.x, Y.y, Y.z, Y.w}, Gv[4] = {G.x, G.y, G.z, G.w},
                                Hv[4] = {Hh.x, Hh.y, Hh.z, Hh.w}, D1v[4] = {D1.x, D1.y, D1.z, D1.w},
                                D12v[4] = {D12.x, D12.y, D12.z, D12.w};
#pragma unroll
                    for (int e4 = 0; e4 < 4; e4++) {
                        const int u = 8 * g8 + 4 * half4 + e4;   // index into this thread's 32 channels
                        const int o = 4 * half4 + e4;            // index within the 8-channel group
                        const float bl = bv[u], kh = kv[u], qh = qv[u];
                        float L, R, eloc, F, Gam, Kdf;
                        if (!flagged) {
                            L = __expf(bl - (hf ? 0.f : shv[e4]));
                            R = __fdividef(1.f, L);
                            eloc = L * Xv[e4];
                            F = R * Yv[e4];
                            Gam = eloc * Gv[e4];
                            Kdf = F * Hv[e4];
                        } else {
                            const int c = cbase + e4;
                            const float pw = Pw[warp * KD + c];
                            const float babs = pw + bl;
                            const float pstart = Pw[(2 * s) * KD + c];
                            const float pend = (s < 3) ? Pw[(2 * s + 2) * KD + c] : blast[c];
                            eloc = __expf(babs - pstart);
                            F = __expf(pend - babs);
                            Gam = __expf(babs);
                            Kdf = __expf(blast[c] - babs);
                            L = 0.f; R = 0.f;
                            // stash for the pairwise diagonal blocks
                            reinterpret_cast<float *>(smem + SM_STK)[ra * KD + c] = kh;
                            reinterpret_cast<float *>(smem + SM_STQ)[ra * KD + c] = qh;
                            reinterpret_cast<float *>(smem + SM_STB)[ra * KD + c] = babs;
                        }
                        ek[o] = kh * eloc; eq[o] = qh * eloc;
                        pk[o] = kh * Gam;  pq[o] = qh * Gam;
                        lk[o] = kh * L;    lq[o] = qh * L;   rkv[o] = kh * R;
                        kd[o] = kh * Kdf;
                        ob[0][o] = kh * F; ob[1][o] = kh * F * D1v[e4]; ob[2][o] = kh * F * D12v[e4];
                    }
                }
                const int k0 = 32 * iq + 8 * g8;     // first channel of the 8
                st_shared_u4(offa + tc::core_offset(ra, k0, KD, 2), pack8_f16(ek));
                st_shared_u4(offa + tc::core_offset(64 + ra, k0, KD, 2), pack8_f16(eq));
                st_shared_u4(pb + tc::core_offset(ra, k0, KD, 2), pack8_f16(pk));
                st_shared_u4(pb + tc::core_offset(64 + ra, k0, KD, 2), pack8_f16(pq));
                if (!flagged) {
                    st_shared_u4(diaga + tc::core_offset(ra, k0, KD, 4), pack4_tf32(lk));
                    st_shared_u4(diaga + tc::core_offset(ra, k0 + 4, KD, 4), pack4_tf32(lk + 4));
                    st_shared_u4(diaga + tc::core_offset(64 + ra, k0, KD, 4), pack4_tf32(lq));
                    st_shared_u4(diaga + tc::core_offset(64 + ra, k0 + 4, KD, 4), pack4_tf32(lq + 4));
                    st_shared_u4(diagb + tc::core_offset(ra, k0, KD, 4), pack4_tf32(rkv));
                    st_shared_u4(diagb + tc::core_offset(ra, k0 + 4, KD, 4), pack4_tf32(rkv + 4));
                }
                // rows of B_R for the later row blocks R = s+1 .. 3
                if (s == 0) {
                    st_shared_u4(offb + tc::core_offset(0 + ra, k0, KD, 2), pack8_f16(ob[0]));
                    st_shared_u4(offb + tc::core_offset(16 + ra, k0, KD, 2), pack8_f16(ob[1]));
                    st_shared_u4(offb + tc::core_offset(48 + ra, k0, KD, 2), pack8_f16(ob[2]));
                } else if (s == 1) {
                    st_shared_u4(offb + tc::core_offset(16 + ra, k0, KD, 2), pack8_f16(ob[0]));
                    st_shared_u4(offb + tc::core_offset(48 + ra, k0, KD, 2), pack8_f16(ob[1]));
                } else if (s == 2) {
                    st_shared_u4(offb + tc::core_offset(48 + ra, k0, KD, 2), pack8_f16(ob[0]));
                }
#pragma unroll
                for (int o = 0; o < 8; o++)
                    st_shared_u16(sbkd + tc::core_offset(k0 + o, ra, 64, 2), f16_bits(kd[o]));
            }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();

        // ================= Phase B: decay-weighted Gram blocks =================
        if (tid == 0) {
            tc::fence_after_sync();
            tc::gemm<0, 96, 128>(tmem + TM_XOFF, sbase + SM_OFFA, SBO128_F16, sbase + SM_OFFB, SBO128_F16, false);
            if (!flagged)
                tc::gemm<2, 64, 128>(tmem + TM_XDIAG, sbase + SM_DIAGA, SBO128_TF32, sbase + SM_DIAGB, SBO128_TF32, false);
            tc::commit(mbar);
        }
        ok &= tc::mbar_wait(mbar, phase);
        phase ^= 1;
        tc::fence_after_sync();

        // ================= Phase C: A, Aqk, T =================
        if (warp < 4) {
            if ((warp & 1) == 0) assemble_rows<0>(smem, tlane, warp, lane, flagged);
            else assemble_rows<1>(smem, tlane, warp, lane, flagged);
        }
        tc::fence_before_sync();
        __syncthreads();
        solve_T(smem, tid);
        {
            // T (fp32, lower, unit diagonal) -> TB fp16 rows r, K = i
            const float *Tm = reinterpret_cast<const float *>(smem + SM_TMAT);
            const int r = tid >> 2, i0 = (tid & 3) * 16;
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; u++) {
                const int i = i0 + u;
                v[u] = (i < r) ? Tm[r * AP + i] : (i == r ? 1.f : 0.f);
            }
            st_shared_u4(sbase + SM_TB + tc::core_offset(r, i0, 64, 2), pack8_f16(v));
            st_shared_u4(sbase + SM_TB + tc::core_offset(r, i0 + 8, 64, 2), pack8_f16(v + 8));
        }

        // ================= Phase D: the chain step =================
        // V values of this thread's column and row half (issued early)
        float vv[32];
        {
            const uint16_t *vp = p.qkv + c0 * p.ld_qkv + 2 * HK + static_cast<int64_t>(h) * VD + jv;
#pragma unroll
            for (int u = 0; u < 32; u++) {
                const int r = 32 * hv + u;
                vv[u] = (r < n) ? bf16_to_f32(vp[static_cast<int64_t>(r) * p.ld_qkv]) : 0.f;
            }
        }
        // D1: S^T -> fp16 operand; TMEM S^T <- S^T Diag(e^{b_last})
        {
            const float *gc = reinterpret_cast<const float *>(smem + SM_GC);
#pragma unroll
            for (int cc = 0; cc < 64; cc += 16) {
                float v[16];
                const int c = 64 * hv + cc;
                tc::tmem_ld16(tlane + TM_S + c, v);
                tc::tmem_ld_wait();
                st_shared_u4(sbase + SM_SA + tc::core_offset(jv, c, KD, 2), pack8_f16(v));
                st_shared_u4(sbase + SM_SA + tc::core_offset(jv, c + 8, KD, 2), pack8_f16(v + 8));
#pragma unroll
                for (int u = 0; u < 16; u++) v[u] *= gc[c + u];
                tc::tmem_st16(tlane + TM_S + c, v);
            }
            tc::tmem_st_wait();
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            tc::gemm<0, 128, 128>(tmem + TM_P, sbase + SM_SA, SBO128_F16, sbase + SM_PB, SBO128_F16, false);
            tc::commit(mbar);
        }
        ok &= tc::mbar_wait(mbar, phase);
        phase ^= 1;
        tc::fence_after_sync();
        // D3: (beta Y)^T = beta (V - K^G S)^T -> fp16 operand
        {
            const float *bet = reinterpret_cast<const float *>(smem + SM_BETA);
#pragma unroll
            for (int cc = 0; cc < 32; cc += 16) {
                float v[16];
                const int r0 = 32 * hv + cc;
                tc::tmem_ld16(tlane + TM_P + r0, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; u++) v[u] = bet[r0 + u] * (vv[cc + u] - v[u]);
                st_shared_u4(sbase + SM_YA + tc::core_offset(jv, r0, 64, 2), pack8_f16(v));
                st_shared_u4(sbase + SM_YA + tc::core_offset(jv, r0 + 8, 64, 2), pack8_f16(v + 8));
            }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            tc::gemm<0, 64, 64>(tmem + TM_P, sbase + SM_YA, SBO64_F16, sbase + SM_TB, SBO64_F16, false);
            tc::commit(mbar);
        }
        ok &= tc::mbar_wait(mbar, phase);
        phase ^= 1;
        tc::fence_after_sync();
        // D5: U^T -> fp16 operand
#pragma unroll
        for (int cc = 0; cc < 32; cc += 16) {
            float v[16];
            const int r0 = 32 * hv + cc;
            tc::tmem_ld16(tlane + TM_P + r0, v);
            tc::tmem_ld_wait();
            st_shared_u4(sbase + SM_UA + tc::core_offset(jv, r0, 64, 2), pack8_f16(v));
            st_shared_u4(sbase + SM_UA + tc::core_offset(jv, r0 + 8, 64, 2), pack8_f16(v + 8));
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            tc::gemm<0, 192, 64>(tmem + TM_P + 64, sbase + SM_UA, SBO64_F16, sbase + SM_SB, SBO64_F16, true);
            tc::commit(mbar);
        }
        ok &= tc::mbar_wait(mbar, phase);
        phase ^= 1;
        tc::fence_after_sync();
        // D7: O^T -> bf16 output rows
        {
            uint16_t *op = p.out + c0 * p.ld_out + static_cast<int64_t>(h) * VD + jv;
#pragma unroll
            for (int cc = 0; cc < 32; cc += 16) {
                float v[16];
                const int r0 = 32 * hv + cc;
                tc::tmem_ld16(tlane + TM_P + 64 + r0, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; u++)
                    if (r0 + u < n) op[static_cast<int64_t>(r0 + u) * p.ld_out] = f32_to_bf16(v[u]);
            }
        }
        tc::fence_before_sync();
        if (__syncthreads_or(ok ? 0 : 1)) {
            ok = false;
            break;
        }
    }

    // ---- final state -> pool ----
    if (ok && writable) {
#pragma unroll
        for (int cc = 0; cc < 64; cc += 16) {
            float v[16];
            const int c = 64 * hv + cc;
            tc::tmem_ld16(tlane + TM_S + c, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; u++) tile[static_cast<int64_t>(c + u) * VD + jv] = v[u];
        }
    }
    if (!ok && tid == 0 && p.err) atomicOr(p.err, kErrTimeout);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc<512>(tmem);
}

}  // namespace chunk

size_t chunk_workspace_bytes(const int32_t *, int64_t, int, int, int, int) { return 0; }

cudaError_t launch_chunk_prefill(const Params &p, int K, int V, const int32_t *cu,
                                 const int32_t *cu_host, int64_t entry_base, int64_t num_seqs,
                                 int, void *, size_t, cudaStream_t stream)
{
    if (num_seqs <= 0) return cudaSuccess;
    if (K != chunk::KD || V != chunk::VD)  // other head sizes take the token-recurrent kernel
        return launch_recurrent(p, K, V, 2, 1, cu, entry_base, num_seqs, stream);
    cudaError_t err = cudaFuncSetAttribute(chunk::chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(chunk::SMEM_BYTES));
    if (err != cudaSuccess) return err;
    chunk::Args a;
    a.p = p;
    a.cu = cu;
    a.entry_base = entry_base;
    a.num_seqs = static_cast<int32_t>(num_seqs);
    a.order_n = 0;
    if (num_seqs <= chunk::kMaxOrder) {
        // longest sequence first, so the longest chains start in the first wave
        std::vector<int32_t> ord(static_cast<size_t>(num_seqs));
        std::iota(ord.begin(), ord.end(), 0);
        const int32_t *cuh = cu_host + entry_base;
        std::stable_sort(ord.begin(), ord.end(), [cuh](int32_t x, int32_t y) {
            return (cuh[x + 1] - cuh[x]) > (cuh[y + 1] - cuh[y]);
        });
        for (int64_t i = 0; i < num_seqs; i++) a.order[i] = ord[static_cast<size_t>(i)];
        a.order_n = static_cast<int32_t>(num_seqs);
    }
    const int64_t grid = num_seqs * p.H;
    chunk::chunk_kernel<<<static_cast<unsigned>(grid), chunk::NT, chunk::SMEM_BYTES, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
