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
// one product.) U only enters through Aqk U and Kd^T U, so T is applied to those two
// instead, off the chain: with Y = V - K^G S,
//   O   = (Q^ * Gamma) S0 + (Aqk T) diag(beta) Y,   S_C = ... + (Kd^T T) diag(beta) Y.
// The state is kept transposed in tensor memory (lane = value column j, column = key
// channel c), so the chain's products have the 128-long V dimension as MMA M:
//   P    = S^T [K^G; Q^G]^T            M=128 N=128 K=128  fp16   -> (K^G S)^T | (Q^G S)^T
//   [O^T | S^T] += (beta Y)^T [Aqk T; Kd^T T]^T   M=128 N=192 K=64 fp16 (S^T pre-scaled by e^{b_last})
// and [Aqk T; Kd^T T] = [Aqk; Kd^T] T is two M=128 N=64 K=64 fp16 products (rows 0..127
// and 64..191) issued right after the triangular solve.
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
// One CTA (512 threads) owns one (sequence, head) chain; CTAs are ordered longest
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
constexpr int NT = 512;
constexpr float kHalfSpan = 40.f;   // largest in-half-block decay served by the tf32 path
constexpr int kMaxOrder = 1024;

// ---- shared memory map (bytes) ----
constexpr uint32_t SM_OFFA = 0;            // fp16 [128 x 128] K^e rows 0..63, Q^e rows 64..127
constexpr uint32_t SM_OFFB = 32768;        // fp16 [96 x 128]  B_1 (16 rows), B_2 (32), B_3 (48)
constexpr uint32_t SM_DIAGA = 57344;       // tf32 [128 x 128] K^L, Q^L
constexpr uint32_t SM_DIAGB = 122880;      // tf32 [64 x 128]  K^R
constexpr uint32_t SM_PB = 155648;         // fp16 [128 x 128] K^G rows 0..63, Q^G rows 64..127
constexpr uint32_t SM_TB = 188416;         // fp16 [64 x 64]   T^T (row m, K = k holds T[k][m])
constexpr uint32_t SM_SB = 196608;         // fp16 [192 x 64]  Aqk rows 0..63, Kd^T rows 64..191,
                                           // then Aqk T and Kd^T T in place
// SB's 8-row core-matrix blocks sit SBO_SB = 1040 bytes apart (16 bytes of padding per
// block): the transposed Kd^T stores of a warp's four 16-channel groups land 2 blocks
// apart, which with a 1024-byte stride would put them in the same banks
constexpr uint32_t SBO_SB = 64 * 2 * 8 + 16;
constexpr uint32_t SM_SB_KD = SM_SB + 8 * SBO_SB;
constexpr uint32_t SM_TAB = SM_TB;         // phase A only: per (block, channel) constants (14336 B)
constexpr uint32_t SM_TOT = SM_SB + 24 * SBO_SB;   // fp32 [8][128] per-warp sums of g, then prefixes P_w
constexpr uint32_t SM_GC = SM_TOT + 4096;  // fp32 [128] e^{b_last}
constexpr uint32_t SM_BLAST = SM_GC + 512; // fp32 [128] b_last
constexpr uint32_t SM_BETA = SM_BLAST + 512;  // fp32 [64]
constexpr uint32_t SM_DTB = SM_BETA + 256;    // fp32 [128] dt_bias of this head
constexpr uint32_t SM_NRM = SM_DTB + 512;     // fp32 [2][64][2] half-row |q|^2, |k|^2
constexpr uint32_t SM_MBAR = SM_NRM + 1024;    // mbarrier of the Gram-block MMAs
constexpr uint32_t SM_MBARC = SM_MBAR + 8;     // mbarrier of the chain MMAs
constexpr uint32_t SM_TMEMP = SM_MBARC + 8;
constexpr uint32_t SM_WAITOK = SM_TMEMP + 4;
constexpr uint32_t SM_MBARW = SM_WAITOK + 4;   // mbarrier of the [Aqk; Kd^T] T products
constexpr uint32_t SMEM_BYTES = SM_MBARW + 8;
static_assert(SM_MBARW % 8 == 0, "mbarrier alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(SM_TAB + 4 * 7 * 128 * 4 <= SM_SB_KD, "constants table overlaps Kd^T");
// phase C aliases
constexpr uint32_t SM_AMAT = SM_OFFA;          // fp32 [64][68]
constexpr uint32_t SM_XTMP = SM_OFFA + 17408;  // fp32 scratch (<= 15360 B)
constexpr uint32_t SM_TMAT = SM_OFFB;          // fp32 [64][68]
constexpr int AP = 68;                         // fp32 row pitch of AMAT / TMAT
// input staging (bf16 [64 rows][128], 16-byte chunks XOR-swizzled by row):
// the next chunk's q, k, raw_g are copied during this chunk's chain step, this
// chunk's V rows during its triangular solve
constexpr uint32_t SM_QST = SM_OFFA;
constexpr uint32_t SM_KST = SM_OFFA + 16384;
constexpr uint32_t SM_VST = SM_DIAGB;
constexpr uint32_t SM_GST = SM_DIAGB + 16384;
// flagged-chunk stash (fp32 [64][128] each)
constexpr uint32_t SM_STK = SM_DIAGA;
constexpr uint32_t SM_STQ = SM_DIAGA + 32768;
constexpr uint32_t SM_STB = SM_DIAGB;

// ---- tensor memory columns ----
constexpr uint32_t TM_P = 0;      // [0,64) K^G S -> U ; [64,128) O
constexpr uint32_t TM_S = 128;    // S^T (128 columns)
constexpr uint32_t TM_XOFF = 256; // 96 columns
constexpr uint32_t TM_XDIAG = 352;// 64 columns
constexpr uint32_t TM_A = 416;    // A operands of the chain MMAs, fp16 packed in pairs:
                                  // S^T (64 columns), then (beta Y)^T at +0
constexpr uint32_t TM_W = TM_XOFF;// [Aqk; Kd^T] T: rows 0..127 (64 columns), rows 64..191 (64)
constexpr uint32_t TM_XDIAG2 = TM_P;  // the diagonal product's channels 64..127 (P is issued after assembly)

// stride byte offsets of the operand tiles
constexpr uint32_t SBO128_F16 = 128 * 2 * 8;  // K = 128 fp16
constexpr uint32_t SBO128_TF32 = 128 * 4 * 8; // K = 128 tf32
constexpr uint32_t SBO64_F16 = 64 * 2 * 8;    // K = 64 fp16

// byte offset of fp16 element (row, k) of SB (K = 64, padded block stride SBO_SB)
__device__ __forceinline__ uint32_t sb_offset(int row, int k)
{
    return static_cast<uint32_t>((row >> 3) * SBO_SB + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// Packs 2*n fp32 values into n fp16 pairs (element 2i in the low half).
template <int n>
__device__ __forceinline__ void pack_pairs(const float *v, uint32_t (&o)[n])
{
#pragma unroll
    for (int i = 0; i < n; i++) o[i] = tc::pack_f16x2(v[2 * i], v[2 * i + 1]);
}

struct Args {
    Params p;
    const int32_t *cu;
    int64_t entry_base;
    int32_t num_seqs;
    int32_t n_chunk;       // CTAs [0, n_chunk) run prefill chains; the rest are decode workers
    int32_t num_decodes;   // mixed batch: entries [0, num_decodes) are length-1 decodes
    int32_t order_n;
    int32_t order[kMaxOrder];
};

// constants table entry (block s, constant k, channel c). A phase-A warp covers one
// 64-channel half; its four 16-channel groups read the same relative 4-channel slot,
// so those four slots sit side by side (one conflict-free LDS.128 per warp).
__device__ __forceinline__ uint32_t tab_off(int s, int k, int c)
{
    const int ch = c >> 6, grp = (c >> 4) & 3, g8 = (c >> 3) & 1, h4 = (c >> 2) & 1, e = c & 3;
    return static_cast<uint32_t>((((((s * 7 + k) * 2 + ch) * 2 + g8) * 2 + h4) * 4 + grp) * 16 + e * 4);
}

__device__ __forceinline__ uint32_t off_b_base(int R) { return R == 1 ? 0 : (R == 2 ? 16 : 48); }

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" :: "r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
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
// by 16x16 diagonal-block inverses and two levels of block doubling (512 threads). Each
// level also writes its final entries of T, transposed and in fp16, to the T^T operand
// tile (row m, K = k holds T[k][m]; at shared address tbt), and the six zero blocks of
// T^T are written during the first level, so the tile is complete (and fenced for the
// async proxy) when the solve returns. The fp32 T keeps only what later levels read.
// ---------------------------------------------------------------------------
__device__ void solve_T(unsigned char *smem, int tid, uint32_t tbt)
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
        // column j of the block is row o + j of T^T, K = o .. o + 15
        st_shared_u4(tbt + tc::core_offset(o + j, o, 64, 2), pack8_f16(t));
        st_shared_u4(tbt + tc::core_offset(o + j, o + 8, 64, 2), pack8_f16(t + 8));
    } else if (tid < 64 + 192) {
        // T^T is zero where the K block precedes the row block: blocks (bm, bk) = (1, 0),
        // (2, 0), (2, 1), (3, 0), (3, 1), (3, 2); 16 rows x two 16-byte chunks each
        const int z = tid - 64, blk = z >> 5, rr = (z >> 1) & 15, hf = z & 1;
        const int bm = blk < 1 ? 1 : (blk < 3 ? 2 : 3), bk = blk - bm * (bm - 1) / 2;
        st_shared_u4(tbt + tc::core_offset(16 * bm + rr, 16 * bk + 8 * hf, 64, 2), make_uint4(0u, 0u, 0u, 0u));
    }
    __syncthreads();
    // level 2: within each 32-block p, X = A_10 T_00 then T_10 = -T_11 X (16x16)
    {
        const int p = tid >> 8, r = (tid >> 4) & 15, j = tid & 15, o = 32 * p;
        float x = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m++) x += A[(o + 16 + r) * AP + o + m] * T[(o + m) * AP + o + j];
        X[(p * 16 + r) * 17 + j] = x;
    }
    __syncthreads();
    {
        const int p = tid >> 8, r = (tid >> 4) & 15, j = tid & 15, o = 32 * p;
        float y = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m++)
            if (m <= r) y += T[(o + 16 + r) * AP + o + 16 + m] * X[(p * 16 + m) * 17 + j];
        T[(o + 16 + r) * AP + o + j] = -y;
        st_shared_u16(tbt + tc::core_offset(o + j, o + 16 + r, 64, 2), f16_bits(-y));
    }
    __syncthreads();
    // level 3: X = A_ba T_a (32x32), T_ba = -T_b X; 2x2 output tiles on 256 threads
    if (tid < 256) {
        const int r = (tid >> 4) * 2, j = (tid & 15) * 2;
        float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;
        for (int m = j; m < 32; m++) {           // T_a is lower triangular: m >= j
            const float a0 = A[(32 + r) * AP + m], a1 = A[(33 + r) * AP + m];
            const float2 t = *reinterpret_cast<const float2 *>(T + m * AP + j);
            const float t1 = (m >= j + 1) ? t.y : 0.f;
            x00 += a0 * t.x; x01 += a0 * t1;
            x10 += a1 * t.x; x11 += a1 * t1;
        }
        *reinterpret_cast<float2 *>(X + r * 36 + j) = make_float2(x00, x01);
        *reinterpret_cast<float2 *>(X + (r + 1) * 36 + j) = make_float2(x10, x11);
    }
    __syncthreads();
    if (tid < 256) {
        const int r = (tid >> 4) * 2, j = (tid & 15) * 2;
        float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
        for (int m = 0; m <= r + 1; m++) {       // T_b is lower triangular: m <= row
            const float t0 = (m <= r) ? T[(32 + r) * AP + 32 + m] : 0.f;
            const float t1 = T[(33 + r) * AP + 32 + m];
            const float2 x = *reinterpret_cast<const float2 *>(X + m * 36 + j);
            y00 += t0 * x.x; y01 += t0 * x.y;
            y10 += t1 * x.x; y11 += t1 * x.y;
        }
        // T_ba is final and read by no later level: only its fp16 transpose is stored, the
        // rows 32 + r, 33 + r of columns j, j + 1 as K pairs of T^T rows j, j + 1
        st_shared_u32(tbt + tc::core_offset(j, 32 + r, 64, 2), tc::pack_f16x2(-y00, -y10));
        st_shared_u32(tbt + tc::core_offset(j + 1, 32 + r, 64, 2), tc::pack_f16x2(-y01, -y11));
    }
    tc::fence_proxy_async();   // T^T is read by the products issued after the barrier
    __syncthreads();
}

// ---------------------------------------------------------------------------
// Phase C0 (flagged chunks only): the diagonal 16x16 blocks of A (before beta) and of Aqk,
// pairwise in fp32 from the stash: one warp per (row r, column i <= r) pair of a block, 4
// channels per lane and a warp reduction; e^{b_r - b_i} is evaluated once for both
// products. Results: dgK / dgQ [64 rows][16] in the phase-C scratch.
// ---------------------------------------------------------------------------
__device__ void flagged_diag(unsigned char *smem, int warp, int lane)
{
    const float *stk = reinterpret_cast<const float *>(smem + SM_STK);
    const float *stq = reinterpret_cast<const float *>(smem + SM_STQ);
    const float *stb = reinterpret_cast<const float *>(smem + SM_STB);
    float *dgK = reinterpret_cast<float *>(smem + SM_XTMP);
    float *dgQ = dgK + 64 * 16;
    const int c = 4 * lane;
    for (int pidx = warp; pidx < 4 * 136; pidx += NT / 32) {
        const int s = pidx / 136, q = pidx - s * 136;   // block s, pair q = rl (rl + 1) / 2 + il
        int rl = static_cast<int>((sqrtf(8.f * q + 1.f) - 1.f) * 0.5f);
        if ((rl + 1) * (rl + 2) / 2 <= q) rl++;
        if (rl * (rl + 1) / 2 > q) rl--;
        const int il = q - rl * (rl + 1) / 2;
        const int r = 16 * s + rl, i = 16 * s + il;
        const float4 kr = *reinterpret_cast<const float4 *>(stk + r * KD + c);
        const float4 qr = *reinterpret_cast<const float4 *>(stq + r * KD + c);
        const float4 br = *reinterpret_cast<const float4 *>(stb + r * KD + c);
        const float4 ki = *reinterpret_cast<const float4 *>(stk + i * KD + c);
        const float4 bi = *reinterpret_cast<const float4 *>(stb + i * KD + c);
        const float e0 = __expf(br.x - bi.x) * ki.x, e1 = __expf(br.y - bi.y) * ki.y;
        const float e2 = __expf(br.z - bi.z) * ki.z, e3 = __expf(br.w - bi.w) * ki.w;
        float a = kr.x * e0 + kr.y * e1 + kr.z * e2 + kr.w * e3;
        float aq = qr.x * e0 + qr.y * e1 + qr.z * e2 + qr.w * e3;
        a = warp_sum(a);
        aq = warp_sum(aq);
        if (lane == 0) {
            dgK[r * 16 + il] = a;
            dgQ[r * 16 + il] = aq;
        }
    }
}

// ---------------------------------------------------------------------------
// Phase C1: one 16-column slice of one row of A (K rows, scaled by beta_r) or Aqk
// (Q rows), from the off-diagonal and diagonal Gram results in TMEM. Thread roles:
// TMEM lane quarter qd = warp & 3 (lanes 0..63 are the K rows, 64..127 the Q rows),
// column slice k4 = warp >> 2.
// ---------------------------------------------------------------------------
__device__ void assemble_slice(unsigned char *smem, uint32_t tlane, int warp, int lane, bool flagged)
{
    const int qd = warp & 3, k4 = warp >> 2;
    const bool qpart = qd >= 2;
    const int r = 32 * (qd & 1) + lane;   // chunk row
    const int s = r >> 4;                 // row block of this lane
    const int s0 = 2 * (qd & 1);          // row blocks of this warp: s0, s0 + 1
    const int i0 = 16 * k4;               // first output column
    float off0[16], off1[16], dg[16];
    // warp-collective loads: every lane loads the same columns, then keeps its own. All
    // three are loaded unconditionally (columns a lane does not need hold values it
    // ignores) so that the arrays stay in registers.
    tc::tmem_ld16(tlane + TM_XOFF + (k4 < s0 ? off_b_base(s0) + i0 : 0), off0);
    tc::tmem_ld16(tlane + TM_XOFF + (k4 < s0 + 1 ? off_b_base(s0 + 1) + i0 : 0), off1);
    tc::tmem_ld16(tlane + TM_XDIAG + i0, dg);
    {
        float dg2[16];   // the diagonal product's second channel half
        tc::tmem_ld16(tlane + TM_XDIAG2 + i0, dg2);
        tc::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; u++) dg[u] += dg2[u];
    }
    if (flagged && k4 == s) {
        // the diagonal block, computed pairwise by flagged_diag (entries i > r are not
        // written there and are masked below)
        const float4 *src = reinterpret_cast<const float4 *>(smem + SM_XTMP) + ((qpart ? 64 : 0) + r) * 4;
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const float4 v = src[u];
            dg[4 * u] = v.x; dg[4 * u + 1] = v.y; dg[4 * u + 2] = v.z; dg[4 * u + 3] = v.w;
        }
    }
    const float beta = qpart ? 1.f : reinterpret_cast<const float *>(smem + SM_BETA)[r];
    float a[16];
#pragma unroll
    for (int u = 0; u < 16; u++) {
        const int i = i0 + u;
        float v = 0.f;
        if (k4 < s) v = (s == s0) ? off0[u] : off1[u];
        else if (k4 == s) v = (qpart ? (i <= r) : (i < r)) ? dg[u] : 0.f;
        a[u] = v * beta;
    }
    if (!qpart) {
        float *Arow = reinterpret_cast<float *>(smem + SM_AMAT) + r * AP + i0;
#pragma unroll
        for (int u = 0; u < 16; u += 4) *reinterpret_cast<float4 *>(Arow + u) = make_float4(a[u], a[u + 1], a[u + 2], a[u + 3]);
    } else {
        const uint32_t base = tc::smem_addr(smem + SM_SB);
        st_shared_u4(base + sb_offset(r, i0), pack8_f16(a));
        st_shared_u4(base + sb_offset(r, i0 + 8), pack8_f16(a + 8));
    }
}

// Waits for the MMAs tracked by `mbar`: warp 0 polls the mbarrier, the other warps park
// on the CTA barrier instead of spinning. Returns false (on every thread) if the wait
// gave up.
__device__ __forceinline__ bool wait_mma(uint32_t mbar, uint32_t parity, int warp, unsigned char *smem)
{
    volatile int *flag = reinterpret_cast<volatile int *>(smem + SM_WAITOK);
    if (warp == 0) {
        const bool ok = tc::mbar_wait(mbar, parity);
        if ((threadIdx.x & 31) == 0) *flag = ok ? 1 : 0;
    }
    __syncthreads();
    const bool ok = *flag != 0;
    tc::fence_after_sync();
    return ok;
}

// As wait_mma for two mbarriers (warp 0 polls both, then one CTA barrier).
__device__ __forceinline__ bool wait_mma2(uint32_t mbar0, uint32_t parity0, uint32_t mbar1, uint32_t parity1,
                                          int warp, unsigned char *smem)
{
    volatile int *flag = reinterpret_cast<volatile int *>(smem + SM_WAITOK);
    if (warp == 0) {
        const bool ok = tc::mbar_wait(mbar0, parity0) && tc::mbar_wait(mbar1, parity1);
        if ((threadIdx.x & 31) == 0) *flag = ok ? 1 : 0;
    }
    __syncthreads();
    const bool ok = *flag != 0;
    tc::fence_after_sync();
    return ok;
}

// byte offset of 16-byte chunk `ch` (0..15) of row r in a staged [64][128] bf16 tile
__device__ __forceinline__ uint32_t st_off(int r, int ch) { return static_cast<uint32_t>(r * 256 + ((ch ^ (r & 7)) << 4)); }

// Copies rows [c0, c0 + 64) of one 128-wide bf16 column block (base + row*ld) into a
// staged tile; rows at or past `nrows` are zero-filled (their source is not read).
__device__ __forceinline__ void stage_rows(uint32_t tile, const uint16_t *base, int64_t ld, int nrows, int tid)
{
#pragma unroll
    for (int x = 0; x < 2; x++) {
        const int id = tid + NT * x, r = id >> 4, ch = id & 15;
        const bool ok = r < nrows;
        const uint16_t *src = base + (ok ? static_cast<int64_t>(r) * ld : 0) + 8 * ch;
        cp_async16(tile + st_off(r, ch), src, ok);
    }
}

// raw phase-A inputs of one thread: 16 channels of q, k and raw_g for one row
struct RowIn {
    uint4 q[2], k[2], g[2];
};

__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// this thread's row r and channels cb .. cb+15 from the staged q, k, raw_g tiles
__device__ __forceinline__ void load_row_inputs(uint32_t sbase, int r, int cb, RowIn &in)
{
    const int ch = cb >> 3;
    in.q[0] = ld_shared_u4(sbase + SM_QST + st_off(r, ch));
    in.q[1] = ld_shared_u4(sbase + SM_QST + st_off(r, ch + 1));
    in.k[0] = ld_shared_u4(sbase + SM_KST + st_off(r, ch));
    in.k[1] = ld_shared_u4(sbase + SM_KST + st_off(r, ch + 1));
    in.g[0] = ld_shared_u4(sbase + SM_GST + st_off(r, ch));
    in.g[1] = ld_shared_u4(sbase + SM_GST + st_off(r, ch + 1));
}

// ---------------------------------------------------------------------------
// The kernel (512 threads, one (sequence, head) chain per CTA)
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// Decode workers of a mixed batch: the CTAs after the prefill chains. Each of the four
// 128-thread groups of such a CTA walks (decode, head, 32-column slice) tiles with a grid
// stride and runs the decode step of the recurrent kernel on each (same thread layout:
// thread (rg, cg) holds rows rg, rg + 16, ... of columns 4cg .. 4cg + 3), with group-local
// named barriers; the next tile's state streams into shared memory (cp.async) and its
// inputs into registers while the current one is computed. They run on the SMs the chains leave free (the chain CTAs come
// first in the grid and need the whole SM), so the decode state stream overlaps the
// prefill in one launch.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void group_bar(int g) { asm volatile("bar.sync %0, 128;" :: "r"(g + 1) : "memory"); }

struct DecodeIn {
    int64_t slot, row;
    int h, j0;
    float q, k, gr, b;
    float4 v;
};

// Loads tile `tile`'s inputs into registers and starts its state slice on its way into this
// thread's staging slots (cp.async; each thread stages exactly what it will hold).
// The row and the state slot of a tile (two index loads; issued a tile ahead of the data
// loads that need them, so no thread waits on them).
struct DecodeIdx {
    int64_t slot, row;
};

__device__ __forceinline__ DecodeIdx decode_index(const Args &args, uint32_t tile)
{
    const uint32_t e = tile / (static_cast<uint32_t>(args.p.H) * (VD / 32));
    return DecodeIdx{load_slot(args.p, e), static_cast<int64_t>(args.cu[e])};
}

__device__ __forceinline__ void decode_load(const Args &args, uint32_t tile, DecodeIdx ix, int gt,
                                            uint32_t stage, DecodeIn &in)
{
    constexpr int VS = VD / 32;
    const Params &p = args.p;
    const uint32_t per_e = static_cast<uint32_t>(p.H) * VS;
    const uint32_t e = tile / per_e, rem = tile - e * per_e;
    in.h = static_cast<int>(rem / VS);
    in.j0 = static_cast<int>(rem % VS) * 32 + (gt & 7) * 4;
    in.row = ix.row;
    in.slot = ix.slot;
    const int rg = gt >> 3;
    if (in.slot >= 0 && in.slot < p.num_slots) {
        const float *src = p.pool + in.slot * p.slot_stride + static_cast<int64_t>(in.h) * KD * VD + in.j0;
#pragma unroll
        for (int i = 0; i < KD / 16; i++)
            cp_async16(stage + static_cast<uint32_t>(i * 128 * 16), src + static_cast<int64_t>(rg + 16 * i) * VD, true);
    }
    cp_async_commit();
    const int64_t HK = static_cast<int64_t>(p.H) * KD;
    const uint16_t *row = p.qkv + in.row * p.ld_qkv;
    in.q = bf16_to_f32(row[in.h * KD + gt]);
    in.k = bf16_to_f32(row[HK + in.h * KD + gt]);
    in.gr = bf16_to_f32(p.rg[in.row * p.ld_g + in.h * KD + gt]);
    in.b = bf16_to_f32(p.rb[in.row * p.ld_beta + in.h]);
    const uint16_t *vp = row + 2 * HK + static_cast<int64_t>(in.h) * VD + in.j0;
    in.v = make_float4(bf16_to_f32(vp[0]), bf16_to_f32(vp[1]), bf16_to_f32(vp[2]), bf16_to_f32(vp[3]));
}

__device__ __noinline__ void decode_worker(const Args &args, unsigned char *smem)
{
    constexpr int RPT = KD / 16;
    constexpr int NS = 3;   // tiles in flight per group: the current one and the next two
    const Params &p = args.p;
    const int tid = threadIdx.x, g = tid >> 7, gt = tid & 127, lane = tid & 31, gw = gt >> 5;
    const int cg = gt & 7, rg = gt >> 3;
    // per group: s_a [KD], s_k [2][KD] (by tile parity: it is read after the group's second
    // barrier), s_q [KD], s_part [4][3], s_red [4][2][32]; then NS staging buffers of
    // [RPT][128] float4 per group (208 KiB in all, inside the chain kernel's allocation)
    float *fs = reinterpret_cast<float *>(smem) + g * 1024;
    float *s_a = fs, *s_k = fs + KD, *s_q = fs + 3 * KD, *s_part = fs + 4 * KD, *s_red = fs + 4 * KD + 16;
    const float4 *stage0 = reinterpret_cast<const float4 *>(smem + 16384 + g * NS * RPT * 128 * 16) + gt;
    const uint32_t ntiles = static_cast<uint32_t>(args.num_decodes) * static_cast<uint32_t>(p.H) * (VD / 32);
    const uint32_t step = (gridDim.x - static_cast<uint32_t>(args.n_chunk)) * 4u;
    uint32_t tile = (blockIdx.x - static_cast<uint32_t>(args.n_chunk)) * 4u + static_cast<uint32_t>(g);
    if (tile >= ntiles) return;
    // tiles tile, tile + step, tile + 2 step live in c0, c1, c2 and in stages si, si+1, si+2
    DecodeIn c0, c1, c2;
    decode_load(args, tile, decode_index(args, tile), gt, tc::smem_addr(stage0), c0);
    c1 = c0;
    c2 = c0;
    if (tile + step < ntiles)
        decode_load(args, tile + step, decode_index(args, tile + step), gt, tc::smem_addr(stage0 + RPT * 128), c1);
    else
        cp_async_commit();
    // indices of the tile two steps ahead (its data loads are issued next iteration)
    DecodeIdx ix2 = tile + 2 * step < ntiles ? decode_index(args, tile + 2 * step) : DecodeIdx{0, 0};
    int kb = 0, si = 0;
    for (; tile < ntiles; tile += step) {
        // the stage being refilled is the previous tile's: every thread of the group read
        // its slots there before that tile's first group barrier
        const int s2 = si == 0 ? 2 : si - 1;
        const DecodeIdx ix3 = tile + 3 * step < ntiles ? decode_index(args, tile + 3 * step) : DecodeIdx{0, 0};
        if (tile + 2 * step < ntiles)
            decode_load(args, tile + 2 * step, ix2, gt, tc::smem_addr(stage0 + s2 * RPT * 128), c2);
        else
            cp_async_commit();
        ix2 = ix3;
        const DecodeIn &cur = c0;
        const float4 *stage_ptr = stage0 + si * RPT * 128;
        if (cur.slot >= p.num_slots) {                // out of range: flag, zero outputs
            if (gt == 0 && p.err) atomicOr(p.err, kErrSlotRange);
            if (rg == 0)
                *reinterpret_cast<uint2 *>(p.out + cur.row * p.ld_out + static_cast<int64_t>(cur.h) * VD + cur.j0) =
                    make_uint2(0u, 0u);
        } else {
            float4 S[RPT];
            cp_async_wait_group<NS - 1>();   // this tile's copies (the two newer may fly)
#pragma unroll
            for (int i = 0; i < RPT; i++) S[i] = cur.slot >= 0 ? stage_ptr[i * 128] : make_float4(0.f, 0.f, 0.f, 0.f);
            // ---- [A] gate + stash ----
            const float expA = expf(__ldg(p.A_log + cur.h));
            const float dtb = p.dt_bias ? __ldg(p.dt_bias + cur.h * KD + gt) : 0.f;
            s_a[gt] = expf(gate_log_decay(cur.gr + dtb, expA, p.has_lb, p.lb));
            s_k[kb * KD + gt] = cur.k;
            s_q[gt] = cur.q;
            {
                const float qq = warp_sum(cur.q * cur.q), kk = warp_sum(cur.k * cur.k), qk = warp_sum(cur.q * cur.k);
                if (lane == 0) { s_part[gw * 3] = qq; s_part[gw * 3 + 1] = kk; s_part[gw * 3 + 2] = qk; }
            }
            group_bar(g);
            // ---- [B] decay + partial reductions ----
            float qq = 0.f, kk = 0.f, qk = 0.f;
#pragma unroll
            for (int w = 0; w < 4; w++) { qq += s_part[w * 3]; kk += s_part[w * 3 + 1]; qk += s_part[w * 3 + 2]; }
            const float rq = p.scale * rsqrtf(qq + p.eps), rk = rsqrtf(kk + p.eps);
            float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < RPT; i++) {
                const int r = rg + 16 * i;
                const float a = s_a[r], kr = s_k[kb * KD + r], qr = s_q[r];
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
                    s_red[(gw * 2) * 32 + cg * 4 + jj] = pk[jj];
                    s_red[(gw * 2 + 1) * 32 + cg * 4 + jj] = pq[jj];
                }
            }
            group_bar(g);
            // ---- [C] u, o, rank-1 update ----
            const float beta = sigmoid_f(cur.b), qkh = qk * rq * rk;
            const float vv[4] = {cur.v.x, cur.v.y, cur.v.z, cur.v.w};
            float u[4], o[4];
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
                const int c = cg * 4 + jj;
                const float ks = (s_red[0 * 32 + c] + s_red[2 * 32 + c] + s_red[4 * 32 + c] + s_red[6 * 32 + c]) * rk;
                const float qs = (s_red[1 * 32 + c] + s_red[3 * 32 + c] + s_red[5 * 32 + c] + s_red[7 * 32 + c]) * rq;
                u[jj] = beta * (vv[jj] - ks);
                o[jj] = qs + qkh * u[jj];
            }
            const bool writable = cur.slot >= 0 && cur.slot != p.null_slot;
            float *tile_ptr = writable ? p.pool + cur.slot * p.slot_stride + static_cast<int64_t>(cur.h) * KD * VD : nullptr;
#pragma unroll
            for (int i = 0; i < RPT; i++) {
                const float kh = s_k[kb * KD + rg + 16 * i] * rk;
                S[i].x += kh * u[0]; S[i].y += kh * u[1]; S[i].z += kh * u[2]; S[i].w += kh * u[3];
                if (writable)
                    *reinterpret_cast<float4 *>(tile_ptr + static_cast<int64_t>(rg + 16 * i) * VD + cur.j0) = S[i];
            }
            if (rg == 0) {
                uint2 packed;
                packed.x = pack_bf16x2(o[0], o[1]);
                packed.y = pack_bf16x2(o[2], o[3]);
                *reinterpret_cast<uint2 *>(p.out + cur.row * p.ld_out + static_cast<int64_t>(cur.h) * VD + cur.j0) = packed;
            }
            kb ^= 1;
        }
        c0 = c1;
        c1 = c2;
        si = si == 2 ? 0 : si + 1;
    }
    cp_async_wait_all();
}

__global__ void __launch_bounds__(NT, 1) chunk_kernel(const __grid_constant__ Args args)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    if (static_cast<int>(blockIdx.x) >= args.n_chunk) {
        decode_worker(args, smem);
        return;
    }
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
    const uint32_t mbar = sbase + SM_MBAR, mbarc = sbase + SM_MBARC, mbarw = sbase + SM_MBARW;
    if (tid == 0) {
        tc::mbar_init(mbar, 3);    // number of issuing threads that commit to each
        tc::mbar_init(mbarw, 2);
        tc::mbar_init(mbarc, 1);
    }
    if (tid < KD) reinterpret_cast<float *>(smem + SM_DTB)[tid] = p.dt_bias ? p.dt_bias[h * KD + tid] : 0.f;
    if (warp == 0) tc::tmem_alloc<512>(sbase + SM_TMEMP);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TMEMP);
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);  // this warp's lanes
    uint32_t phase = 0, phasec = 0, phasew = 0;
    bool ok = true;
    bool os_pending = false;   // the last product (O and S) of the previous chunk is in flight

    // thread roles
    const int jv = 32 * (warp & 3) + lane;  // TMEM lane: value column j in phase D
    const int k4 = warp >> 2;               // column slice (0..3) of TMEM work
    const int ir = lane & 7, iq = lane >> 3;
    const int rga = warp & 7;               // phase A: rows 8*rga .. 8*rga+7
    const int ra = 8 * rga + ir;            // phase A: chunk row
    const int cb = 64 * (warp >> 3) + 16 * iq;  // phase A: first of 16 channels
    const int sA = rga >> 1, hfA = rga & 1; // phase A: row block, half of the block

    // O^T of a finished chunk (rows cs .. cs + nrows - 1) -> bf16 rows, straight from
    // registers: lane j of the warp holds column j of 16 rows, so each store instruction
    // writes 64 contiguous bytes of one row
    auto store_out = [&](int64_t cs, int nrows) {
        float v[16];
        const int r0 = 16 * k4;
        tc::tmem_ld16(tlane + TM_P + 64 + r0, v);
        tc::tmem_ld_wait();
        uint16_t *orow = p.out + (cs + r0) * p.ld_out + static_cast<int64_t>(h) * VD + jv;
#pragma unroll
        for (int u = 0; u < 16; u++)
            if (r0 + u < nrows) orow[u * p.ld_out] = f32_to_bf16(v[u]);
    };

    // ---- S0 -> TMEM (S^T: lane j, columns c in this thread's 32-column slice) ----
    {
#pragma unroll
        for (int cc = 0; cc < 32; cc += 16) {
            float v[16];
            const int c = 32 * k4 + cc;
#pragma unroll
            for (int u = 0; u < 16; u++)
                v[u] = has_state ? tile[static_cast<int64_t>(c + u) * VD + jv] : 0.f;
            tc::tmem_st16(tlane + TM_S + c, v);
        }
        tc::tmem_st_wait();
    }

    const float expA = __expf(p.A_log[h]);
    const float *dtb_s = reinterpret_cast<const float *>(smem + SM_DTB);
    // stage the first chunk's q, k, raw_g rows
    {
        const int n0 = static_cast<int>((row1 - row0) < C ? (row1 - row0) : C);
        stage_rows(sbase + SM_QST, p.qkv + row0 * p.ld_qkv + h * KD, p.ld_qkv, n0, tid);
        stage_rows(sbase + SM_KST, p.qkv + row0 * p.ld_qkv + HK + h * KD, p.ld_qkv, n0, tid);
        stage_rows(sbase + SM_GST, p.rg + row0 * p.ld_g + h * KD, p.ld_g, n0, tid);
        cp_async_commit();
    }
    uint16_t beta_raw = 0;   // raw_beta of row tid of the current chunk (threads < 64)
    if (tid < C && tid < row1 - row0) beta_raw = p.rb[(row0 + tid) * p.ld_beta + h];

    int64_t last_c0 = row0;
    int last_n = 0;
    for (int64_t c0 = row0; c0 < row1; c0 += C) {
        const int n = static_cast<int>((row1 - c0) < C ? (row1 - c0) : C);

        // ================= Phase A: gate, norms, cumulative decay, operands =================
        // staged inputs of this chunk (copied during the previous chain step); the same
        // barrier ends the previous chunk and carries its timeout result
        cp_async_wait_all();
        if (__syncthreads_or(ok ? 0 : 1)) {
            ok = false;
            break;
        }
        tc::fence_after_sync();
        RowIn in;
        const bool valid = ra < n;
        load_row_inputs(sbase, ra, cb, in);
        float qv[16], kv[16], bv[16];
        if (valid) {
            unpack_bf16x8(in.q[0], qv); unpack_bf16x8(in.q[1], qv + 8);
            unpack_bf16x8(in.k[0], kv); unpack_bf16x8(in.k[1], kv + 8);
            unpack_bf16x8(in.g[0], bv); unpack_bf16x8(in.g[1], bv + 8);
        } else {
#pragma unroll
            for (int u = 0; u < 16; u++) { qv[u] = 0.f; kv[u] = 0.f; bv[u] = 0.f; }
        }
        float qq = 0.f, kk = 0.f;
#pragma unroll
        for (int u = 0; u < 16; u++) {
            bv[u] = valid ? gate_log_decay_fast(bv[u] + dtb_s[cb + u], expA, p.has_lb, p.lb) : 0.f;
            qq += qv[u] * qv[u];
            kk += kv[u] * kv[u];
        }
        qq += __shfl_xor_sync(0xffffffffu, qq, 8);
        qq += __shfl_xor_sync(0xffffffffu, qq, 16);
        kk += __shfl_xor_sync(0xffffffffu, kk, 8);
        kk += __shfl_xor_sync(0xffffffffu, kk, 16);
        float *nrm = reinterpret_cast<float *>(smem + SM_NRM);   // [half][row][2]
        if (iq == 0) *reinterpret_cast<float2 *>(nrm + ((warp >> 3) * 64 + ra) * 2) = make_float2(qq, kk);
        // in-warp inclusive scan over the 8 rows (lanes ir = 0..7 of the same channel group)
#pragma unroll
        for (int u = 0; u < 16; u++) {
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
            for (int u = 0; u < 16; u += 4)
                *reinterpret_cast<float4 *>(tot + rga * KD + cb + u) = make_float4(bv[u], bv[u + 1], bv[u + 2], bv[u + 3]);
        }
        if (tid < C) reinterpret_cast<float *>(smem + SM_BETA)[tid] = (tid < n) ? sigmoid_f(bf16_to_f32(beta_raw)) : 0.f;
        if (os_pending) {
            // this barrier also ends the previous chunk's last product (issued ~4k cycles
            // ago, so the wait is short): its O rows are stored here, off the chain's
            // critical path, and its Kd^T operand rows are free for this chunk's
            ok &= wait_mma(mbarc, phasec, warp, smem);
            phasec ^= 1;
            os_pending = false;
            store_out(c0 - C, C);   // every chunk but the last is full
        } else {
            __syncthreads();
        }

        // per-(block, channel) constants: thread tid handles channel tid & 127, block tid >> 7
        int flag = 0;
        {
            const int c = tid & (KD - 1), s = tid >> 7;
            // block s covers warps 2s, 2s+1; scalars only, so everything stays in registers
            float G = 1.f, Hh = 1.f, D1 = 1.f, D12 = 1.f, T0 = 0.f, X = 1.f, Y = 1.f, gc = 1.f, P = 0.f;
#pragma unroll
            for (int w = 0; w < 8; w++) {
                const float t = tot[w * KD + c];
                const float ew = __expf(t);
                if (w < 2 * s) G *= ew;
                if (w >= 2 * s + 2) Hh *= ew;
                if (w == 2 * s) { T0 = t; X = ew; }
                if (w == 2 * s + 1) Y = ew;
                if (w == 2 * s + 2 || w == 2 * s + 3) D1 *= ew;
                if (w >= 2 * s + 2 && w <= 2 * s + 5) D12 *= ew;
                flag |= (t < -kHalfSpan) ? 1 : 0;
                gc *= ew;
                P += t;
            }
            if (s > 2) D1 = 0.f;
            if (s > 1) D12 = 0.f;
            float *tabp = reinterpret_cast<float *>(smem + SM_TAB);
            tabp[tab_off(s, 0, c) >> 2] = T0;
            tabp[tab_off(s, 1, c) >> 2] = X;
            tabp[tab_off(s, 2, c) >> 2] = Y;
            tabp[tab_off(s, 3, c) >> 2] = G;
            tabp[tab_off(s, 4, c) >> 2] = Hh;
            tabp[tab_off(s, 5, c) >> 2] = D1;
            tabp[tab_off(s, 6, c) >> 2] = D12;
            if (s == 0) {
                reinterpret_cast<float *>(smem + SM_GC)[c] = gc;
                reinterpret_cast<float *>(smem + SM_BLAST)[c] = P;
            }
        }
        // prefixes P_w replace the per-warp sums (read only on the flagged path)
        const bool flagged = __syncthreads_or(flag) != 0;
        if (flagged && tid < KD) {
            float P = 0.f;
#pragma unroll
            for (int w = 0; w < 8; w++) {
                const float t = tot[w * KD + tid];
                tot[w * KD + tid] = P;
                P += t;
            }
        }
        if (flagged) __syncthreads();


        {
            // full-row norms from the two channel halves
            const float2 n0 = *reinterpret_cast<const float2 *>(nrm + ra * 2);
            const float2 n1 = *reinterpret_cast<const float2 *>(nrm + (64 + ra) * 2);
            const float rq = p.scale * rsqrtf(n0.x + n1.x + p.eps), rk = rsqrtf(n0.y + n1.y + p.eps);
            const uint32_t offa = sbase + SM_OFFA, offb = sbase + SM_OFFB, diaga = sbase + SM_DIAGA,
                           diagb = sbase + SM_DIAGB, pb = sbase + SM_PB, sbkd = sbase + SM_SB_KD;
            const uint32_t tab = sbase + SM_TAB;
            // 8 channels of table constant k for this thread's block
            auto tab8 = [&](int k, int k0, float *dst) {
                const float4 a = ld_shared_f4(tab + tab_off(sA, k, k0));
                const float4 b = ld_shared_f4(tab + tab_off(sA, k, k0 + 4));
                dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
                dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
            };
#pragma unroll
            for (int g8 = 0; g8 < 2; g8++) {          // 8 channels at a time
                const int k0 = cb + 8 * g8;           // first channel of the 8
                float kh[8], qh[8], A8[8], B8[8], t8[8], v8[8];
#pragma unroll
                for (int o = 0; o < 8; o++) { kh[o] = kv[8 * g8 + o] * rk; qh[o] = qv[8 * g8 + o] * rq; }
                if (!flagged) {
                    // A8 = L = e^{b - b_mid}, B8 = R = 1/L  (middle-row reference of the block)
                    tab8(0, k0, t8);
#pragma unroll
                    for (int o = 0; o < 8; o++) {
                        A8[o] = __expf(bv[8 * g8 + o] - (hfA ? 0.f : t8[o]));
                        B8[o] = __fdividef(1.f, A8[o]);
                    }
#pragma unroll
                    for (int o = 0; o < 8; o++) v8[o] = kh[o] * A8[o];
                    st_shared_u4(diaga + tc::core_offset(ra, k0, KD, 4), pack4_tf32(v8));
                    st_shared_u4(diaga + tc::core_offset(ra, k0 + 4, KD, 4), pack4_tf32(v8 + 4));
#pragma unroll
                    for (int o = 0; o < 8; o++) v8[o] = qh[o] * A8[o];
                    st_shared_u4(diaga + tc::core_offset(64 + ra, k0, KD, 4), pack4_tf32(v8));
                    st_shared_u4(diaga + tc::core_offset(64 + ra, k0 + 4, KD, 4), pack4_tf32(v8 + 4));
#pragma unroll
                    for (int o = 0; o < 8; o++) v8[o] = kh[o] * B8[o];
                    st_shared_u4(diagb + tc::core_offset(ra, k0, KD, 4), pack4_tf32(v8));
                    st_shared_u4(diagb + tc::core_offset(ra, k0 + 4, KD, 4), pack4_tf32(v8 + 4));
                    // A8 <- e_loc = L * e^{T_first_half}, B8 <- F = R * e^{T_second_half}
                    tab8(1, k0, t8);
#pragma unroll
                    for (int o = 0; o < 8; o++) A8[o] *= t8[o];
                    tab8(2, k0, t8);
#pragma unroll
                    for (int o = 0; o < 8; o++) B8[o] *= t8[o];
                } else {
                    const float *Pw = reinterpret_cast<const float *>(smem + SM_TOT);
                    const float *blast = reinterpret_cast<const float *>(smem + SM_BLAST);
#pragma unroll
                    for (int o = 0; o < 8; o++) {
                        const int c = k0 + o;
                        const float babs = Pw[rga * KD + c] + bv[8 * g8 + o];
                        const float pstart = Pw[(2 * sA) * KD + c];
                        const float pend = (sA < 3) ? Pw[(2 * sA + 2) * KD + c] : blast[c];
                        A8[o] = __expf(babs - pstart);   // e_loc
                        B8[o] = __expf(pend - babs);     // F
                        // stash for the pairwise diagonal blocks
                        reinterpret_cast<float *>(smem + SM_STK)[ra * KD + c] = kh[o];
                        reinterpret_cast<float *>(smem + SM_STQ)[ra * KD + c] = qh[o];
                        reinterpret_cast<float *>(smem + SM_STB)[ra * KD + c] = babs;
                    }
                }
                // off-diagonal A operand (K^e, Q^e)
#pragma unroll
                for (int o = 0; o < 8; o++) v8[o] = kh[o] * A8[o];
                st_shared_u4(offa + tc::core_offset(ra, k0, KD, 2), pack8_f16(v8));
#pragma unroll
                for (int o = 0; o < 8; o++) v8[o] = qh[o] * A8[o];
                st_shared_u4(offa + tc::core_offset(64 + ra, k0, KD, 2), pack8_f16(v8));
                // A8 <- Gamma = e_loc * e^{b at the block start}
                tab8(3, k0, t8);
#pragma unroll
                for (int o = 0; o < 8; o++) A8[o] *= t8[o];
#pragma unroll
                for (int o = 0; o < 8; o++) v8[o] = kh[o] * A8[o];
                st_shared_u4(pb + tc::core_offset(ra, k0, KD, 2), pack8_f16(v8));
#pragma unroll
                for (int o = 0; o < 8; o++) v8[o] = qh[o] * A8[o];
                st_shared_u4(pb + tc::core_offset(64 + ra, k0, KD, 2), pack8_f16(v8));
                // rows of B_R for the later row blocks R = sA+1 .. 3: k^ F, k^ F D1, k^ F D12
#pragma unroll
                for (int o = 0; o < 8; o++) kh[o] *= B8[o];      // kh <- k^ F
                if (sA < 3) {
                    st_shared_u4(offb + tc::core_offset(off_b_base(sA + 1) + ra, k0, KD, 2), pack8_f16(kh));
                    if (sA < 2) {
                        tab8(5, k0, t8);
#pragma unroll
                        for (int o = 0; o < 8; o++) v8[o] = kh[o] * t8[o];
                        st_shared_u4(offb + tc::core_offset(off_b_base(sA + 2) + ra, k0, KD, 2), pack8_f16(v8));
                        if (sA < 1) {
                            tab8(6, k0, t8);
#pragma unroll
                            for (int o = 0; o < 8; o++) v8[o] = kh[o] * t8[o];
                            st_shared_u4(offb + tc::core_offset(off_b_base(3) + ra, k0, KD, 2), pack8_f16(v8));
                        }
                    }
                }
                // Kd^T = (k^ F e^{b_last - b_block_end})^T
                tab8(4, k0, t8);
#pragma unroll
                for (int o = 0; o < 8; o++)
                    st_shared_u16(sbkd + sb_offset(k0 + o, ra), f16_bits(kh[o] * t8[o]));
            }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();

        // ================= Phase B: decay-weighted Gram blocks =================
        // three issuing threads (in different warps), each committing its own products: one
        // thread's tcgen05.mma issue takes longer than these small products take to run.
        // The tf32 diagonal product is split by channels (0..63, 64..127) into two
        // accumulators that the row assembly adds.
        if (tid == 0) {
            tc::fence_after_sync();
            tc::gemm<0, 96, 128>(tmem + TM_XOFF, sbase + SM_OFFA, SBO128_F16, sbase + SM_OFFB, SBO128_F16, false);
            tc::commit(mbar);
        } else if (tid == 32 || tid == 64) {
            tc::fence_after_sync();
            // channel c's 16-byte K chunk sits at (c / 4) * 128 bytes: channels 64.. at 2048
            const uint32_t koff = tid == 32 ? 0u : 2048u;
            if (!flagged)
                tc::gemm<2, 64, 64>(tmem + (tid == 32 ? TM_XDIAG : TM_XDIAG2), sbase + SM_DIAGA + koff, SBO128_TF32,
                                    sbase + SM_DIAGB + koff, SBO128_TF32, false);
            tc::commit(mbar);
        }
        // D1 while the Gram MMAs run: S^T -> fp16 pairs in TMEM (A of P), and
        // TMEM S^T <- S^T Diag(e^{b_last}).
        {
            const float *gc = reinterpret_cast<const float *>(smem + SM_GC);
            float v[2][16];
            tc::tmem_ld16(tlane + TM_S + 32 * k4, v[0]);
            tc::tmem_ld16(tlane + TM_S + 32 * k4 + 16, v[1]);
            tc::tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const int c = 32 * k4 + 16 * hh;
                uint32_t pk8[8];
                pack_pairs<8>(v[hh], pk8);
                tc::tmem_st8u(tlane + TM_A + (c >> 1), pk8);
#pragma unroll
                for (int u = 0; u < 16; u += 4) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(gc + c + u);
                    v[hh][u] *= g4.x; v[hh][u + 1] *= g4.y; v[hh][u + 2] *= g4.z; v[hh][u + 3] *= g4.w;
                }
                tc::tmem_st16(tlane + TM_S + c, v[hh]);
            }
            tc::tmem_st_wait();
        }
        // the barrier ends the Gram wait and orders every thread's S^T operand before the
        // P issue (after the row assembly, which reads the second diagonal accumulator)
        tc::fence_before_sync();
        ok &= wait_mma(mbar, phase, warp, smem);
        phase ^= 1;

        // ================= Phase C: A, Aqk, T (the P product is issued after assembly) =================
        // The V tile (read in D3) overlays the diagonal B operand (consumed by now) or, on
        // the pairwise path, the stash (dead once flagged_diag has run).
        const uint16_t *vsrc = p.qkv + c0 * p.ld_qkv + 2 * HK + static_cast<int64_t>(h) * VD;
        if (flagged) {   // the pairwise diagonal blocks; after them the stash is dead
            flagged_diag(smem, warp, lane);
            __syncthreads();
        }
        stage_rows(sbase + SM_VST, vsrc, p.ld_qkv, n, tid);
        cp_async_commit();
        assemble_slice(smem, tlane, warp, lane, flagged);
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 64) {
            // P = S^T [K^G; Q^G]^T (overwrites the second diagonal accumulator, read above);
            // it runs during the solve
            tc::fence_after_sync();
            tc::gemm_ta<128, 128>(tmem + TM_P, tmem + TM_A, sbase + SM_PB, SBO128_F16, false);
            tc::commit(mbarc);
        }
        // T^T (fp16) is complete and fenced when the solve returns; the Aqk rows of SB were
        // written before the solve's barriers and fenced at its end as well
        solve_T(smem, tid, sbase + SM_TB);
        if (tid == 0 || tid == 32) {
            // [Aqk; Kd^T] T -> TMEM (lane = row of SB), one half per issuing thread; it runs
            // while the inputs are staged and P is awaited
            tc::fence_after_sync();
            if (tid == 0)
                tc::gemm<0, 64, 64>(tmem + TM_W, sbase + SM_SB, SBO_SB, sbase + SM_TB, SBO64_F16, false);
            else
                tc::gemm<0, 64, 64>(tmem + TM_W + 64, sbase + SM_SB_KD, SBO_SB, sbase + SM_TB, SBO64_F16, false);
            tc::commit(mbarw);
        }

        // ================= Phase D: the rest of the chain step =================
        // the next chunk's q, k, raw_g rows -> staging (the scratch of phase C is dead now)
        if (c0 + C < row1) {
            const int64_t nx = c0 + C;
            const int nn = static_cast<int>((row1 - nx) < C ? (row1 - nx) : C);
            stage_rows(sbase + SM_QST, p.qkv + nx * p.ld_qkv + h * KD, p.ld_qkv, nn, tid);
            stage_rows(sbase + SM_KST, p.qkv + nx * p.ld_qkv + HK + h * KD, p.ld_qkv, nn, tid);
            stage_rows(sbase + SM_GST, p.rg + nx * p.ld_g + h * KD, p.ld_g, nn, tid);
            if (tid < nn) beta_raw = p.rb[(nx + tid) * p.ld_beta + h];
        }
        cp_async_commit();
        // the V tile (the older group) has landed for this thread; the barrier inside the
        // wait makes every thread's part of it visible
        cp_async_wait_group<1>();
        ok &= wait_mma2(mbarc, phasec, mbarw, phasew, warp, smem);   // P and [Aqk; Kd^T] T
        phasec ^= 1;
        phasew ^= 1;
        // D3: (beta Y)^T = beta (V - K^G S)^T -> fp16 pairs in TMEM (rows r = 16 k4 .. +15)
        {
            const float *bet = reinterpret_cast<const float *>(smem + SM_BETA);
            const uint16_t *vt = reinterpret_cast<const uint16_t *>(smem + SM_VST);
            float v[16];
            const int r0 = 16 * k4;
            tc::tmem_ld16(tlane + TM_P + r0, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; u++) {
                const int r = r0 + u;
                const float vv = bf16_to_f32(vt[(st_off(r, jv >> 3) >> 1) + (jv & 7)]);
                v[u] = bet[r] * (vv - v[u]);
            }
            uint32_t pk8[8];
            pack_pairs<8>(v, pk8);
            tc::tmem_st8u(tlane + TM_A + (r0 >> 1), pk8);
            tc::tmem_st_wait();
        }
        // D5: [Aqk T; Kd^T T] -> fp16 rows of SB, in place (the B operand of the last
        // product); TMEM lane = row, 16 of the 64 K columns per warp
        {
            const uint32_t sb = sbase + SM_SB;
            const int row = 32 * (warp & 3) + lane;
            float v[16];
            tc::tmem_ld16(tlane + TM_W + 16 * k4, v);
            tc::tmem_ld_wait();
            st_shared_u4(sb + sb_offset(row, 16 * k4), pack8_f16(v));
            st_shared_u4(sb + sb_offset(row, 16 * k4 + 8), pack8_f16(v + 8));
            if ((warp & 3) >= 2) {   // lanes 64..127 of the second product: rows 128..191
                tc::tmem_ld16(tlane + TM_W + 64 + 16 * k4, v);
                tc::tmem_ld_wait();
                st_shared_u4(sb + sb_offset(row + 64, 16 * k4), pack8_f16(v));
                st_shared_u4(sb + sb_offset(row + 64, 16 * k4 + 8), pack8_f16(v + 8));
            }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            tc::gemm_ta<192, 64>(tmem + TM_P + 64, tmem + TM_A, sbase + SM_SB, SBO_SB, true);
            tc::commit(mbarc);
        }
        // D7 (the O rows) runs in the next chunk's phase A, or below for the last chunk
        os_pending = true;
        last_c0 = c0;
        last_n = n;
        tc::fence_before_sync();
    }
    // the last chunk's product; also waited for after a timeout elsewhere, so that no MMA
    // is in flight when the tensor memory is released
    if (os_pending) {
        ok &= wait_mma(mbarc, phasec, warp, smem);
        phasec ^= 1;
        if (ok) store_out(last_c0, last_n);
    }

    // ---- final state -> pool ----
    if (ok && writable) {
#pragma unroll
        for (int cc = 0; cc < 32; cc += 16) {
            float v[16];
            const int c = 32 * k4 + cc;
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

// One CTA of NT threads waits, as the chain CTAs do (one warp polls, the rest park on the
// barrier), on an mbarrier that nothing arrives at. The bounded wait gives up after ~2 s;
// the kernel then records the timeout in the error word and returns normally.
__global__ void __launch_bounds__(chunk::NT, 1) bounded_wait_selftest_kernel(uint32_t *err)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int waitok;
    const uint32_t mbar = tc::smem_addr(&bar);
    if (threadIdx.x == 0) tc::mbar_init(mbar, 1);
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        const bool ok = tc::mbar_wait(mbar, 0);
        if ((threadIdx.x & 31) == 0) waitok = ok ? 1 : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0 && !waitok && err) atomicOr(err, kErrTimeout);
}

size_t chunk_workspace_bytes(const int32_t *, int64_t, int, int, int, int) { return 0; }

cudaError_t launch_bounded_wait_selftest(uint32_t *err, cudaStream_t stream)
{
    bounded_wait_selftest_kernel<<<1, chunk::NT, 0, stream>>>(err);
    return cudaGetLastError();
}

// One launch: the prefill chains of entries [entry_base, entry_base + num_seqs), ordered
// longest first, then (num_decodes > 0) decode-worker CTAs for the length-1 entries
// [0, num_decodes) of a mixed batch.
static cudaError_t launch_chunk_grid(const Params &p, const int32_t *cu, const int32_t *cu_host,
                                     int64_t entry_base, int64_t num_seqs, int64_t num_decodes,
                                     cudaStream_t stream)
{
    cudaError_t err = cudaFuncSetAttribute(chunk::chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(chunk::SMEM_BYTES));
    if (err != cudaSuccess) return err;
    chunk::Args a;
    a.p = p;
    a.cu = cu;
    a.entry_base = entry_base;
    a.num_seqs = static_cast<int32_t>(num_seqs);
    a.n_chunk = static_cast<int32_t>(num_seqs * p.H);
    a.num_decodes = static_cast<int32_t>(num_decodes);
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
    int64_t workers = 0;
    if (num_decodes > 0) {
        // one worker CTA per SM the chains leave free, at least a quarter of the SMs (they
        // also take over SMs whose chains finish early), at most one tile per group
        int dev = 0, sms = 0;
        if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        const int64_t tiles = num_decodes * p.H * (chunk::VD / 32);
        workers = sms - static_cast<int64_t>(a.n_chunk);
        if (workers < sms / 4) workers = sms / 4;
        if (workers < 1) workers = 1;
        if (workers > (tiles + 3) / 4) workers = (tiles + 3) / 4;
    }
    const int64_t grid = static_cast<int64_t>(a.n_chunk) + workers;
    if (grid <= 0) return cudaSuccess;
    chunk::chunk_kernel<<<static_cast<unsigned>(grid), chunk::NT, chunk::SMEM_BYTES, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_chunk_prefill(const Params &p, int K, int V, const int32_t *cu,
                                 const int32_t *cu_host, int64_t entry_base, int64_t num_seqs,
                                 int, void *, size_t, cudaStream_t stream)
{
    if (num_seqs <= 0) return cudaSuccess;
    if (K != chunk::KD || V != chunk::VD)  // other head sizes take the token-recurrent kernel
        return launch_recurrent(p, K, V, 2, 1, cu, entry_base, num_seqs, stream);
    return launch_chunk_grid(p, cu, cu_host, entry_base, num_seqs, 0, stream);
}

cudaError_t launch_mixed(const Params &p, int K, int V, const int32_t *cu, const int32_t *cu_host,
                         int64_t num_decodes, int64_t num_prefills, cudaStream_t stream)
{
    if (K != chunk::KD || V != chunk::VD || num_decodes <= 0 || num_prefills <= 0) {
        if (num_decodes > 0) {
            cudaError_t e = launch_recurrent(p, K, V, 2, 1, cu, 0, num_decodes, stream);
            if (e != cudaSuccess) return e;
        }
        return launch_chunk_prefill(p, K, V, cu, cu_host, num_decodes, num_prefills, 64, nullptr, 0, stream);
    }
    return launch_chunk_grid(p, cu, cu_host, num_decodes, num_prefills, num_decodes, stream);
}

}  // namespace kda
