// Chunked varlen prefill on tcgen05 tensor cores (K and V in {64, 128} on 128 x 128 tiles,
// chunk C = 64).
//
// The chunked (WY) form of the gated delta rule (chunk_kda_with_fused_gate with its
// recompute_w_u step, vLLM PR #50649, section Purpose). For one (sequence, head) and a
// chunk of n <= 64 rows with in-chunk cumulative log-decay b_r = sum_{i<=r} g_i (per
// channel), Gamma_r = e^{b_r} and gamma = e^{b_last}:
//   A[r,i]   = beta_r sum_c k^_r k^_i e^{b_r - b_i}   (i < r)    T = (I + A)^-1
//   Aqk[r,i] = sum_c q^_r k^_i e^{b_r - b_i}          (i <= r)
//   Kd       = K^ * e^{b_last - b}
//   M1 = Aqk T diag(beta),   M2 = Kd^T T diag(beta)
//   Y   = V - (K^ * Gamma) S0
//   O   = (Q^ * Gamma) S0 + M1 Y
//   S_C = Diag(gamma) S0 + M2 Y
// (The recompute_w_u form U = T diag(beta) (V - (K^ * Gamma) S0) with O = ... + Aqk U and
// S_C = ... + Kd^T U, with T folded into the two products that consume U.)
//
// Everything but Y, O and S_C depends on the chunk's inputs alone, so the work splits in
// two kernels:
//   prep_kernel   one CTA per (chunk, head), all of them in parallel (two CTAs per SM):
//                 gate, norms, cumulative decay, the decay-weighted Gram matrices on the
//                 tensor cores, the triangular solve (its last level on the tensor cores)
//                 and [Aqk; Kd^T] T diag(beta) on the tensor cores. It writes one record
//                 per (chunk, head) to the workspace: [K^G; Q^G] (fp16), gamma (fp32) and
//                 [M1; M2] (fp16), each already in the shared-memory layout the chain's
//                 MMAs read, and a flag per unit; a second launch redoes the flagged units
//                 (a channel half decaying too fast within a block) with the pairwise path.
//   chain_kernel  one CTA per (sequence, head) chain (one per SM): the state stays in
//                 tensor memory, transposed (lane = value column j, column = key channel);
//                 per chunk two products
//                   P = S^T [K^G; Q^G]^T                 M=128 N=128 K=128  fp16
//                   [O^T | S^T] += Y^T [M1; M2]^T         M=128 N=192 K=64   fp16
//                 with S^T pre-scaled by gamma, the records streamed in by bulk copies two
//                 chunks ahead.
//
// The decay-weighted Gram matrices are split into 16-row blocks s = 0..3 with prefixes
// P_s = b at the last row before block s (P_0 = 0). Every row carries its own block's
// reference, so the A operand is one tile for both products:
//   A_op = [K^e; Q^e],  K^e_r = k^_r e^{b_r - P_s(r)} (<= 1)      (tf32, in tensor memory)
// Diagonal blocks:      X_diag = A_op (K^R)^T,  K^R_i = k^_i e^{P_s(i) - b_i}   (>= 1)
// Off-diagonal blocks:  X_off  = A_op [B_1; B_2; B_3]^T,  B_R = rows i < 16R at
//                       k^_i e^{P_R - b_i} (<= 1), for the rows of block R; both operands
//                       in fp16 (every factor is at most 1 in magnitude: half the tf32
//                       tensor time; parts below 2^-24 of the largest are lost).
// K^R reaches e^{(decay over the block)}, which tf32 (fp32 range) holds while a block's
// decay stays below 80 nats; a channel half in which some channel decays more within a
// block computes its share of the diagonal blocks pairwise in fp32 instead.
//
// fp16 (11-bit significand, round to nearest) carries the same precision as tf32 with
// round to nearest; bf16 operands would exceed the 2e-3 relative error bar.
#include <algorithm>
#include <mutex>
#include <numeric>
#include <vector>

#include <cuda.h>          // CUtensorMap and its enums (the encoder is fetched through the runtime)
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "kda_common.cuh"
#include "kda_f32x2.cuh"
#include "kda_launch.h"
#include "kda_pdl.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace chunk {

constexpr int C = 64;
constexpr int KD = 128;
constexpr int PT = 256;          // prep threads
constexpr int CT = 256;          // chain threads
constexpr int kMaxSeqs = 1024;   // sequences per launch (the host splits larger calls)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kBlockSpan2 = 80.f * kLog2e;   // largest in-block decay of the tf32 diagonal path (log2 units)

// ---- one (chunk, head) record in the workspace ----
constexpr uint32_t REC_KQG = 0;        // fp16 [128 rows][128] K-major, SBO 2048: K^G rows 0..63, Q^G 64..127
constexpr uint32_t REC_GAM = 32768;    // fp32 [128] gamma = e^{b_last}
constexpr uint32_t REC_MM = 33280;     // fp16 [192 rows][64] K-major, SBO 1024: M1 rows 0..63, M2 64..191
constexpr uint32_t REC_A_BYTES = REC_MM;   // first bulk copy: [K^G; Q^G] and gamma
constexpr uint32_t REC_B_BYTES = 24576;    // second: [M1; M2]
constexpr uint32_t REC_BYTES = REC_MM + REC_B_BYTES;
static_assert(REC_BYTES % 256 == 0 || REC_BYTES % 16 == 0, "records stay 16-byte aligned");

// stride byte offsets of the K-major operand tiles
constexpr uint32_t SBO128_F16 = 128 * 2 * 8;   // K = 128 fp16
constexpr uint32_t SBO64_F16 = 64 * 2 * 8;     // K = 64 fp16
constexpr uint32_t SBO64_TF32 = 64 * 4 * 8;    // K = 64 tf32
// SB's 8-row core-matrix blocks sit SBO_SB = 1040 bytes apart (16 bytes of padding per
// block): the transposed Kd^T stores of a warp's four 8-row groups then land in
// different banks
constexpr uint32_t SBO_SB = SBO64_F16 + 16;

// ---- prep shared memory (bytes) ----
constexpr uint32_t SM_G = 0;            // bf16 [2][64][64] raw_g as two TMA boxes (128B swizzle, see tma_off)
constexpr uint32_t SM_BH = 16384;       // fp32 [64][64]  b (log2 units) of the current channel half, swizzled
constexpr uint32_t SM_BOFF = 32768;     // fp16 [96][64]  [B_1; B_2; B_3] of the current half (SBO 1024)
constexpr uint32_t SM_BDIAG = 57344;    // tf32 [64][64]  K^R of the current half (SBO 2048); on the
                                        // pairwise path: fp16 [64][64] k^ then q^ (swizzled)
constexpr uint32_t SM_SB = 73728;       // fp16 [192][64] Aqk rows 0..63, Kd^T rows 64..191 (SBO 1040)
constexpr uint32_t SM_QSTG = SM_BOFF;   // bf16 [2][64][64] q, staged like raw_g (read before operand generation)
constexpr uint32_t SM_KSTG = SM_BDIAG;  // bf16 [2][64][64] k
static_assert(SM_QSTG + 16384 <= SM_BDIAG && SM_KSTG + 16384 <= SM_SB, "q/k staging regions");
static_assert(SM_G % 1024 == 0 && SM_QSTG % 1024 == 0 && SM_KSTG % 1024 == 0, "128B-swizzled boxes");
constexpr uint32_t SM_TAB = SM_SB + 24 * SBO_SB;   // fp32 [4 blocks][8][64] per-(block, channel) constants
constexpr uint32_t SM_TOT = SM_TAB + 8192;         // fp32 [8][64] sums of g over 8-row octets
constexpr uint32_t SM_NRM = SM_TOT + 2048;         // fp32 [2][128] half-row |k|^2, |q|^2
constexpr uint32_t SM_BETA = SM_NRM + 1024;        // fp32 [64]
constexpr uint32_t SM_MBAR = SM_BETA + 256;        // mbarrier of the MMAs (two committing threads)
constexpr uint32_t SM_LBAR = SM_MBAR + 8;          // mbarriers of the tensor copies: raw_g, then q and k
constexpr uint32_t SM_TMEMP = SM_LBAR + 16;
constexpr uint32_t SM_WAITOK = SM_TMEMP + 4;
constexpr uint32_t SM_GFLAG = SM_WAITOK + 4;       // int: some channel of the gate pass's half decays too fast
constexpr uint32_t PREP_SMEM = SM_GFLAG + 4;
static_assert(SM_MBAR % 8 == 0, "mbarrier alignment");
static_assert(2 * (PREP_SMEM + 1024) <= 233472, "two prep CTAs per SM");
// solve-phase aliases over SM_G .. SM_BDIAG (dead once the Gram products are done)
constexpr uint32_t SM_AMAT = 0;        // fp32 [64][68]
constexpr uint32_t SM_TMAT = 17408;    // fp32 [64][68]
constexpr uint32_t SM_XTMP = 34816;    // fp32 scratch (<= 4608 B)
constexpr uint32_t SM_TT = 40960;      // fp16 [64][64] (T diag(beta))^T, K-major SBO 1024
constexpr uint32_t SM_XD = 49152;      // fp32 [2][64][16] pairwise diagonal blocks (read before the solve)
constexpr int AP = 68;                 // fp32 row pitch of AMAT / TMAT
static_assert(SM_XD + 8192 <= SM_SB, "solve scratch overlaps SB");

// ---- prep tensor memory columns (256) ----
constexpr uint32_t TM_XOFF = 0;     // X_off   96 columns
constexpr uint32_t TM_XDIAG = 96;   // X_diag  64 columns
constexpr uint32_t TM_A = 160;      // tf32 A operand [K^e; Q^e] of the current channel half (64 columns)
constexpr uint32_t TM_A16 = 224;    // the same in fp16 pairs, the A operand of X_off (32 columns)
constexpr uint32_t TM_W1 = 0;       // [Aqk; Kd^T rows 0..63] T diag(beta)   (after assembly)
constexpr uint32_t TM_W2 = 64;      // Kd^T T diag(beta)
constexpr uint32_t TM_L3X = 160;    // the solve's last level: X^T (32 columns)
constexpr uint32_t TM_L3T = 192;    //                         X^T T_b^T (32 columns)

// per-(block, channel) constants, [block][constant][channel of the half]
enum Tab { kP1 = 1, kE = 2, kBD = 3, kD4 = 4, kD2 = 5, kD3 = 6 };   // kP1: the block's log2 decay

__device__ __forceinline__ uint32_t off_b_base(int R) { return R == 1 ? 0 : (R == 2 ? 16 : 48); }

struct Args {
    CUtensorMap tm_qkv;        // mixed_qkv [rows][2HK + HV] bf16, boxes of 64 rows x 64 columns, 128B swizzle
    CUtensorMap tm_g;          // raw_g [rows][HK], the same boxes
    Params p;
    const int32_t *cu;         // device cu_seqlens (entries)
    int64_t entry_base;        // first entry of this launch
    int32_t num_seqs;
    int32_t pf_stride;         // prep: the unit whose inputs a CTA prefetches into L2 (bid + pf_stride)
    unsigned char *rec;        // records of this launch: (chunk, head) at (cb + j) * H + h
    unsigned char *flags;      // unit flags of the call (16-byte aligned, after every record): 1 where
                               // the unit needs the pairwise path; this launch's unit u at flag0 + u
    int32_t flag0;
    int32_t cb[kMaxSeqs + 1];  // chunk prefix over the launch's sequences
    int32_t rs[kMaxSeqs + 1];  // row starts of the launch's sequences (the host copy of cu_seqlens)
    int32_t order[kMaxSeqs];   // chain order: longest sequence first
};

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

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
// 8 floats -> 8 fp16 in one 16-byte chunk
__device__ __forceinline__ uint4 pack8_f16(const float *v)
{
    return make_uint4(tc::pack_f16x2(v[0], v[1]), tc::pack_f16x2(v[2], v[3]),
                      tc::pack_f16x2(v[4], v[5]), tc::pack_f16x2(v[6], v[7]));
}
// fp32 -> tf32 operand, rounded to nearest with ties away from zero: the tensor core reads
// the top 19 bits, so adding half a unit of the kept significand (bit 12) to the pattern
// rounds the magnitude, carrying into the exponent where the significand overflows.
__device__ __forceinline__ uint32_t tf32_rna(float x) { return __float_as_uint(x) + 0x1000u; }
__device__ __forceinline__ uint4 pack4_tf32(const float *v)
{
    return make_uint4(tf32_rna(v[0]), tf32_rna(v[1]), tf32_rna(v[2]), tf32_rna(v[3]));
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

// byte offset of 16-byte chunk `ch` (0..15) of row r in a staged [64][128] bf16 tile
__device__ __forceinline__ uint32_t st_off(int r, int ch) { return static_cast<uint32_t>(r * 256 + ((ch ^ (r & 7)) << 4)); }
// byte offset of fp32 element (r, c) of the [64][64] b tile (16-byte chunks swizzled by row)
__device__ __forceinline__ uint32_t bh_off(int r, int c)
{
    return static_cast<uint32_t>(r * 256 + ((((c >> 2) ^ (r & 7))) << 4) + (c & 3) * 4);
}
// byte offset of fp16 element (row, k) of SB (K = 64, padded block stride SBO_SB)
__device__ __forceinline__ uint32_t sb_offset(int row, int k)
{
    return static_cast<uint32_t>((row >> 3) * SBO_SB + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}
__device__ __forceinline__ uint32_t tab_off(int s, int k, int c) { return static_cast<uint32_t>(((s * 8 + k) * 64 + c) * 4); }

// Byte offset of 16-byte chunk ch (0..15) of row r in a tile staged as two TMA boxes of
// 64 rows x 128 bytes (channels 0..63, then 64..127) with the 128-byte swizzle: the chunk
// index within a row's 128 bytes is XORed with r mod 8.
__device__ __forceinline__ uint32_t tma_off(int r, int ch)
{
    return static_cast<uint32_t>((ch >> 3) * 8192 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// Copies rows [0, 64) of one 128-wide bf16 column block (base + row*ld) into a staged tile
// with NTH threads; rows at or past `nrows` and 16-byte chunks at or past `nch16` (of 16)
// are zero-filled (their source is not read).
template <int NTH>
__device__ __forceinline__ void stage_rows(uint32_t tile, const uint16_t *base, int64_t ld, int nrows, int tid,
                                           int nch16 = 16)
{
#pragma unroll
    for (int x = 0; x < 1024 / NTH; x++) {
        const int id = tid + NTH * x, r = id >> 4, ch = id & 15;
        const bool ok = r < nrows && ch < nch16;
        const uint16_t *src = base + (ok ? static_cast<int64_t>(r) * ld : 0) + 8 * ch;
        cp_async16(tile + st_off(r, ch), src, ok);
    }
}

// Waits for an mbarrier phase: warp 0 polls, the other warps park on the CTA barrier.
// Returns false (on every thread) if the wait gave up or `ok_in` was false on thread 0.
__device__ __forceinline__ bool cta_wait(uint32_t mbar, uint32_t parity, unsigned char *flag_smem, bool ok_in = true)
{
    volatile int *flag = reinterpret_cast<volatile int *>(flag_smem);
    if (threadIdx.x < 32) {
        const bool ok = tc::mbar_wait(mbar, parity);
        if (threadIdx.x == 0) *flag = (ok && ok_in) ? 1 : 0;
    }
    __syncthreads();
    const bool ok = *flag != 0;
    tc::fence_after_sync();
    return ok;
}

// d = a * b, d = a - b and d = a * s over 8 values
__device__ __forceinline__ void mul8(float *d, const float *a, const float *b)
{
#pragma unroll
    for (int o = 0; o < 8; o += 2) {
        const float2 v = fmul2(make_float2(a[o], a[o + 1]), make_float2(b[o], b[o + 1]));
        d[o] = v.x; d[o + 1] = v.y;
    }
}
__device__ __forceinline__ void sub8(float *d, const float *a, const float *b)
{
#pragma unroll
    for (int o = 0; o < 8; o += 2) {
        const float2 v = fsub2(make_float2(a[o], a[o + 1]), make_float2(b[o], b[o + 1]));
        d[o] = v.x; d[o + 1] = v.y;
    }
}
__device__ __forceinline__ void scale8(float *d, const float *a, float sc)
{
#pragma unroll
    for (int o = 0; o < 8; o += 2) {
        const float2 v = fmul2(make_float2(a[o], a[o + 1]), make_float2(sc, sc));
        d[o] = v.x; d[o + 1] = v.y;
    }
}
// ---------------------------------------------------------------------------
// T = (I + A)^-1 for the strictly lower 64x64 A in AMAT (fp32, pitch AP), first two
// levels (256 threads): the 16x16 diagonal-block inverses, then the block doubling to the
// two 32x32 diagonal blocks T_a, T_b. Each level writes its final entries of T diag(beta),
// transposed and in fp16, to the operand tile at `tbt` (row m, K = k holds T[k][m]
// beta_m); the six zero blocks of the transpose are written during the first level. The
// fp32 T keeps only what later levels read. The last level (the block T_ba) runs on the
// tensor cores in the prep kernel.
// ---------------------------------------------------------------------------
__device__ void solve_T(unsigned char *smem, int tid, uint32_t tbt, const float *beta)
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
        // column j of the block is row o + j of (T diag(beta))^T, K = o .. o + 15
        const float bj = beta[o + j];
        float u[16];
#pragma unroll
        for (int r = 0; r < 16; r++) u[r] = t[r] * bj;
        st_shared_u4(tbt + tc::core_offset(o + j, o, 64, 2), pack8_f16(u));
        st_shared_u4(tbt + tc::core_offset(o + j, o + 8, 64, 2), pack8_f16(u + 8));
    } else {
        // the transpose is zero where the K block precedes the row block: blocks (bm, bk) =
        // (1, 0), (2, 0), (2, 1), (3, 0), (3, 1), (3, 2); 16 rows x two 16-byte chunks each
        const int z = tid - 64, blk = z >> 5, rr = (z >> 1) & 15, hf = z & 1;
        const int bm = blk < 1 ? 1 : (blk < 3 ? 2 : 3), bk = blk - bm * (bm - 1) / 2;
        st_shared_u4(tbt + tc::core_offset(16 * bm + rr, 16 * bk + 8 * hf, 64, 2), make_uint4(0u, 0u, 0u, 0u));
    }
    __syncthreads();
    // level 2: within each 32-block p, X = A_10 T_00 then T_10 = -T_11 X (16x16); each
    // thread owns two adjacent columns (packed fp32x2 arithmetic)
    {
        const int p = tid >> 7, r = (tid >> 3) & 15, j = (tid & 7) * 2, o = 32 * p;
        float2 x = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 16; m++) {
            const float a = A[(o + 16 + r) * AP + o + m];
            x = ffma2(make_float2(a, a), *reinterpret_cast<const float2 *>(T + (o + m) * AP + o + j), x);
        }
        *reinterpret_cast<float2 *>(X + (p * 16 + r) * 18 + j) = x;
    }
    __syncthreads();
    {
        const int p = tid >> 7, r = (tid >> 3) & 15, j = (tid & 7) * 2, o = 32 * p;
        float2 y = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 16; m++) {
            if (m <= r) {
                const float t = T[(o + 16 + r) * AP + o + 16 + m];
                y = ffma2(make_float2(t, t), *reinterpret_cast<const float2 *>(X + (p * 16 + m) * 18 + j), y);
            }
        }
        *reinterpret_cast<float2 *>(T + (o + 16 + r) * AP + o + j) = make_float2(-y.x, -y.y);
        st_shared_u16(tbt + tc::core_offset(o + j, o + 16 + r, 64, 2), f16_bits(-y.x * beta[o + j]));
        st_shared_u16(tbt + tc::core_offset(o + j + 1, o + 16 + r, 64, 2), f16_bits(-y.y * beta[o + j + 1]));
    }
    __syncthreads();
}


__device__ __forceinline__ void ex2_8(float *d)
{
#pragma unroll
    for (int o = 0; o < 8; o++) d[o] = ex2(d[o]);
}
__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void unpack_f16x8(uint4 u, float *f)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __half2 h2 = *reinterpret_cast<const __half2 *>(&w[i]);
        const float2 v = __half22float2(h2);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}
__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
// fp16 [64][64] stash of the pairwise path: 16-byte chunks XOR-swizzled by row
__device__ __forceinline__ uint32_t stash_off(int r, int c) { return static_cast<uint32_t>(r * 128 + (((c >> 3) ^ (r & 7)) << 4)); }

// The per-channel log-decay in log2 units, g * log2(e): -e^{A_log} softplus(x) log2(e)
// = -e^{A_log} (max(x, 0) log2(e) + log2(1 + 2^{-|x| log2(e)})), or lower_bound log2(e)
// sigmoid(e^{A_log} x) with a lower bound.
__device__ __forceinline__ float gate_log2(float x, float expA, float expA_l2e, int has_lb, float lb_l2e)
{
    if (has_lb) return lb_l2e * __fdividef(1.f, 1.f + ex2(-expA_l2e * x));
    return -expA_l2e * fmaxf(x, 0.f) - expA * lg2(1.f + ex2(-kLog2e * fabsf(x)));
}

// ---------------------------------------------------------------------------
// prep_kernel: one CTA of 256 threads per (chunk, head); two CTAs per SM.
//
// Thread roles: TMEM lane l = 32 (warp & 3) + lane and channel quarter sub = warp >> 2.
// Lanes 0..63 are the K side (key row r = l), lanes 64..127 the Q side (query row
// r = l - 64); in a channel half a thread covers channels 32 sub .. 32 sub + 31. The
// key-side work beyond the A operand (F = e^{P_{s+1} - b}, K^R, the B_R rows, Kd^T) is
// split between the two threads of a row: the K thread takes the first 16 of the 32
// channels, the Q thread the last 16. The gate pass uses channel c = tid & 63 of the
// half and row block tid >> 6.
//
// Two instances per K. PW = false: one CTA per unit, without the pairwise path. A unit in
// which some channel half needs that path is only marked in the unit flags, and its
// [M1; M2] are not written. PW = true: the pass over the marked units, with the pairwise
// path. A grid of a few CTAs per SM runs it; each CTA takes the marked units whose rank
// among them is congruent to its index. Keeping the pairwise code out of the first
// instance keeps that instance's code small and its registers for the common path.
// LB: the gate form with a lower bound (the first pass only; the second reads it from the
// parameters).
// ---------------------------------------------------------------------------
template <int NH, bool PW, bool LB>   // NH: channel halves that hold data (K = 64 NH)
__global__ void __launch_bounds__(PT, 2) prep_kernel(const __grid_constant__ Args a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    const Params &p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    constexpr int kr = 64 * NH, nhalf = NH;
    const int64_t HK = static_cast<int64_t>(H) * kr;
    const int total = a.cb[a.num_seqs] * H;   // (chunk, head) units of this launch
    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t mbar = sbase + SM_MBAR;
    float *tab = reinterpret_cast<float *>(smem + SM_TAB);
    float *tot = reinterpret_cast<float *>(smem + SM_TOT);
    float *nrm = reinterpret_cast<float *>(smem + SM_NRM);
    float *betas = reinterpret_cast<float *>(smem + SM_BETA);
    const int l = 32 * (warp & 3) + lane, sub = warp >> 2;
    const bool kside = l < 64;
    const int r = l & 63, s = r >> 4;
    const int side = kside ? 0 : 1;
    const uint32_t lbar = sbase + SM_LBAR;
    if (tid == 0) {
        tc::prefetch_tensormap(&a.tm_g);
        tc::prefetch_tensormap(&a.tm_qkv);
        tc::mbar_init(mbar, 2);   // two issuing threads commit to every MMA stage
        tc::mbar_init(lbar, 1);
        tc::mbar_init(lbar + 8, 1);
    }
    // the unit's head, first row and row count (the sequence: the last s with cb[s] <=
    // chunk; a later unit's search starts from the known sequence of an earlier one,
    // usually ending at once)
    auto locate = [&](int bid, int &hh, int64_t &r0, int &nn, int &sq) {
        const int cgi = bid / H;
        hh = bid - cgi * H;
        if (sq < 0) {
            int lo = 0, hi = a.num_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (a.cb[mid] <= cgi) lo = mid; else hi = mid - 1;
            }
            sq = lo;
        } else {
            while (sq + 1 < a.num_seqs && a.cb[sq + 1] <= cgi) sq++;
        }
        r0 = static_cast<int64_t>(a.rs[sq]) + static_cast<int64_t>(cgi - a.cb[sq]) * C;
        const int64_t rem = static_cast<int64_t>(a.rs[sq + 1]) - r0;
        nn = static_cast<int>(rem < C ? rem : C);
    };
    // ---- raw_g, then q and k (into the B-operand regions, free until operand generation)
    // by tensor copies from thread 0, issued before the tensor-memory allocation; thread 32
    // prefetches a later unit's boxes into L2 (the unit pf_stride later starts on a CTA
    // slot about when this one ends). The first gate pass runs while q and k are still in
    // flight. Rows past the chunk hold the next sequence's rows (or zeros past the tensor)
    // and are masked where read. ----
    auto issue_loads = [&](const int bid, const int h, const int64_t row0, const int sq) {
    if (tid == 0) {
        const int y = static_cast<int>(row0), xg = h * kr;
        tc::mbar_expect_tx(lbar, 8192u * nhalf);
        for (int hf = 0; hf < nhalf; hf++) tc::tma_load_2d(sbase + SM_G + 8192 * hf, &a.tm_g, xg + 64 * hf, y, lbar);
        tc::mbar_expect_tx(lbar + 8, 16384u * nhalf);
        for (int hf = 0; hf < nhalf; hf++) {
            tc::tma_load_2d(sbase + SM_QSTG + 8192 * hf, &a.tm_qkv, xg + 64 * hf, y, lbar + 8);
            tc::tma_load_2d(sbase + SM_KSTG + 8192 * hf, &a.tm_qkv, static_cast<int>(HK) + xg + 64 * hf, y, lbar + 8);
        }
    } else if (!PW && tid == 32 && bid + a.pf_stride < total) {
        int h2, n2, sq2 = sq;
        int64_t r2;
        locate(bid + a.pf_stride, h2, r2, n2, sq2);
        const int y2 = static_cast<int>(r2), x2 = h2 * kr;
        for (int hf = 0; hf < nhalf; hf++) {
            tc::tma_prefetch_2d(&a.tm_g, x2 + 64 * hf, y2);
            tc::tma_prefetch_2d(&a.tm_qkv, x2 + 64 * hf, y2);
            tc::tma_prefetch_2d(&a.tm_qkv, static_cast<int>(HK) + x2 + 64 * hf, y2);
        }
    }
    };
    uint32_t tmem = 0, tlane = 0;
    auto alloc_tmem = [&]() {
        if (warp == 0) tc::tmem_alloc<256>(sbase + SM_TMEMP);
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TMEMP);
        tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    };
    uint32_t phase = 0;   // parity of the MMA barrier (kept across the units of a CTA)
    bool ok = true;
    // ---- one unit, from its tensor copies (issued) to its record; lpar: the parity of the
    // copies' barriers for this unit ----
    auto compute = [&](const int bid, const int h, const int64_t row0, const int n, const uint32_t lpar) {
    // this unit's beta (consumed after the first gate pass, so its latency is hidden)
    const uint16_t braw = (tid < C && tid < n) ? p.rb[(row0 + tid) * p.ld_beta + h] : static_cast<uint16_t>(0);
    unsigned char *rec = a.rec + static_cast<size_t>(bid) * REC_BYTES;

    const float expA = __expf(__ldg(p.A_log + h));
    const float expA_l2e = expA * kLog2e, lb_l2e = p.lb * kLog2e;
    // dt_bias of this thread's channel pair in the gate passes (channels 64 hf + 2 (tid & 31) ..),
    // loaded before the passes so that its latency is hidden
    float2 dtb_h[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    if (p.dt_bias) {
#pragma unroll
        for (int hf = 0; hf < nhalf; hf++)
        {   // two scalar loads: dt_bias is only 4-byte aligned
            const float *d = p.dt_bias + h * kr + 64 * hf + 2 * (tid & 31);
            dtb_h[hf] = make_float2(__ldg(d), __ldg(d + 1));
        }
    }
    uint4 xr[2][4];   // own row of q or k: [half][4 x 8 bf16] = channels 64 hf + 32 sub .. + 31
    float rn = 0.f, rk = 0.f;   // norm factors of the own row and of the key row r
    ok &= cta_wait(lbar, lpar, smem + SM_WAITOK);   // raw_g has landed

    // ---- gate pass over one channel half: per (row, channel) e1 = e^{b - P_s} (the decay
    // since the block's reference) into SM_BH, or on the pairwise path the in-block log2
    // prefix itself; the per-(block, channel) constants; gamma into the record. Returns
    // whether some channel of the half decays by more than the tf32 diagonal path holds
    // within a block. Thread (cp, o8): channels 2 cp, 2 cp + 1 of the half (packed pairs),
    // rows 8 o8 .. 8 o8 + 7. ----
    auto gate_half = [&](int hf) -> bool {
        const int cp = tid & 31, o8 = tid >> 5, sg = o8 >> 1;
        const int cg = 64 * hf + 2 * cp;                 // first channel of the pair (in the head)
        const float2 dtb = hf ? dtb_h[1] : dtb_h[0];
        const int ch = cg >> 3;
        const unsigned char *gt = smem + SM_G + (ch >> 3) * 8192 + 8 * o8 * 128 + (cg & 7) * 2;
        const int nv = n - 8 * o8;               // rows of this octet inside the chunk
        float2 v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(gt + j * 128 + (((ch & 7) ^ j) << 4));
            v[j] = fadd2(make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)), dtb);
        }
        if (PW ? p.has_lb != 0 : LB) {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const float2 t = fmul2(v[j], make_float2(-expA_l2e, -expA_l2e));
                v[j] = make_float2(lb_l2e * rcp_approx(1.f + ex2(t.x)), lb_l2e * rcp_approx(1.f + ex2(t.y)));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const float lx = lg2(1.f + ex2(-kLog2e * fabsf(v[j].x)));
                const float ly = lg2(1.f + ex2(-kLog2e * fabsf(v[j].y)));
                const float2 m = make_float2(fmaxf(v[j].x, 0.f), fmaxf(v[j].y, 0.f));
                v[j] = ffma2(m, make_float2(-expA_l2e, -expA_l2e), fmul2(make_float2(lx, ly), make_float2(-expA, -expA)));
            }
        }
#pragma unroll
        for (int j = 0; j < 8; j++)
            if (j >= nv) v[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 1; j < 8; j++) v[j] = fadd2(v[j], v[j - 1]);
        *reinterpret_cast<float2 *>(tot + o8 * 64 + 2 * cp) = v[7];
        if (!PW && tid == 0) *reinterpret_cast<int *>(smem + SM_GFLAG) = 0;   // read only after the pass's
                                                                             // last barrier, set after its first
        // the second octet of a block starts from the first octet's sum; the block sum
        // decides the path (a block decaying beyond kBlockSpan2 nats)
        __syncthreads();
        float2 oct[8];
#pragma unroll
        for (int q = 0; q < 8; q++) oct[q] = *reinterpret_cast<const float2 *>(tot + q * 64 + 2 * cp);
        const float2 blk0 = fadd2(oct[0], oct[1]), blk1 = fadd2(oct[2], oct[3]);
        const float2 blk2 = fadd2(oct[4], oct[5]), blk3 = fadd2(oct[6], oct[7]);
        const float2 acc = sg == 0 ? blk0 : (sg == 1 ? blk1 : (sg == 2 ? blk2 : blk3));
        const int fl = (-acc.x > kBlockSpan2 || -acc.y > kBlockSpan2) ? 1 : 0;
        // with the pairwise path compiled in, the values stored below depend on the decision;
        // otherwise it is only reported, read after the pass's last barrier
        bool flagged = false;
        if (PW) flagged = __syncthreads_or(fl) != 0;
        else if (fl) atomicOr(reinterpret_cast<int *>(smem + SM_GFLAG), 1);
        if (o8 & 1) {
            const float2 first = sg == 0 ? oct[0] : (sg == 1 ? oct[2] : (sg == 2 ? oct[4] : oct[6]));
#pragma unroll
            for (int j = 0; j < 8; j++) v[j] = fadd2(v[j], first);
        }
        {
            float *bh = reinterpret_cast<float *>(smem + SM_BH + 8 * o8 * 256);
            const int q4 = cp >> 1, e4 = (cp & 1) * 2;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int rr = 8 * o8 + j;
                const float2 val = (PW && flagged) ? v[j] : make_float2(ex2(v[j].x), ex2(v[j].y));
                *reinterpret_cast<float2 *>(bh + (j * 256 + ((q4 ^ (rr & 7)) << 4)) / 4 + e4) = val;
            }
        }
        if ((o8 & 1) == 0) {   // the first octet of each block writes the block's constants
            const float2 P0 = sg == 0 ? make_float2(0.f, 0.f)
                            : (sg == 1 ? blk0 : (sg == 2 ? fadd2(blk0, blk1) : fadd2(fadd2(blk0, blk1), blk2)));
            const float2 P4 = fadd2(fadd2(blk0, blk1), fadd2(blk2, blk3));
            const float2 n1 = sg == 0 ? blk1 : (sg == 1 ? blk2 : (sg == 2 ? blk3 : make_float2(0.f, 0.f)));
            const float2 n2 = sg == 0 ? blk2 : (sg == 1 ? blk3 : make_float2(0.f, 0.f));
            float *tb = tab + sg * 8 * 64 + 2 * cp;
            auto put2 = [&](int k, float2 x) { *reinterpret_cast<float2 *>(tb + k * 64) = x; };
            put2(kE, make_float2(ex2(P0.x), ex2(P0.y)));
            put2(kBD, make_float2(ex2(acc.x), ex2(acc.y)));                                   // e^{P_{s+1} - P_s}
            const float2 d4 = fsub2(fsub2(P4, P0), acc);
            put2(kD4, make_float2(ex2(d4.x), ex2(d4.y)));                                     // e^{P_4 - P_{s+1}}
            put2(kD2, make_float2(ex2(n1.x), ex2(n1.y)));                                     // e^{P_{s+2} - P_{s+1}}
            const float2 n12 = fadd2(n1, n2);
            put2(kD3, make_float2(ex2(n12.x), ex2(n12.y)));                                   // e^{P_{s+3} - P_{s+1}}
            put2(kP1, acc);                                                                   // the block's log2 decay
            if (sg == 3) *reinterpret_cast<float2 *>(rec + REC_GAM + 4 * cg) = make_float2(ex2(P4.x), ex2(P4.y));
        }
        __syncthreads();
        if (!PW) flagged = *reinterpret_cast<volatile int *>(smem + SM_GFLAG) != 0;
        return flagged;
    };
    // fl: the half needs the pairwise path; pw: it takes it here
    const bool fl0 = gate_half(0), pw0 = PW && fl0;
    if (tid < C) betas[tid] = tid < n ? sigmoid_f(bf16_to_f32(braw)) : 0.f;   // read in the assembly
    ok &= cta_wait(lbar + 8, lpar, smem + SM_WAITOK);   // q and k have landed
    {   // own row from the staged tile (zero past the chunk) and its half-row sums of squares
        const uint32_t stg = sbase + (kside ? SM_KSTG : SM_QSTG);
        float2 ss = make_float2(0.f, 0.f);
#pragma unroll
        for (int hf = 0; hf < 2; hf++)
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++) {
                const uint4 v = (r < n && hf < nhalf) ? ld_shared_u4(stg + tma_off(r, 8 * hf + 4 * sub + q4))
                                                      : make_uint4(0u, 0u, 0u, 0u);
                xr[hf][q4] = v;
                float f[8];
                unpack_bf16x8(v, f);
#pragma unroll
                for (int o = 0; o < 8; o += 2) ss = ffma2(make_float2(f[o], f[o + 1]), make_float2(f[o], f[o + 1]), ss);
            }
        nrm[sub * 128 + l] = ss.x + ss.y;
    }
    // the Q thread's key share of channel half 0 (key row r, channels 32 sub + 16 .. + 31), from
    // the staged k before operand generation overwrites it
    uint4 kq0[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    if (!kside && r < n) {
        kq0[0] = ld_shared_u4(sbase + SM_KSTG + tma_off(r, 4 * sub + 2));
        kq0[1] = ld_shared_u4(sbase + SM_KSTG + tma_off(r, 4 * sub + 3));
    }
    // ... and of half 1: the key thread of row r leaves those channels of its own row in SB's
    // Aqk rows (free until the row assembly) for the query thread
    if (nhalf == 2 && kside) {
        st_shared_u4(sbase + SM_SB + (r * 2 + sub) * 32, xr[1][2]);
        st_shared_u4(sbase + SM_SB + (r * 2 + sub) * 32 + 16, xr[1][3]);
    }
    __syncthreads();   // the half-row norms; the staged q and k are consumed
    {   // rows past the chunk hold zeros; their norm factor is 0 so that eps = 0 gives no NaN
        auto norm_of = [&](int lane_idx, int row) -> float {
            const float f = (lane_idx < 64 ? 1.f : p.scale) * rsqrtf(nrm[lane_idx] + nrm[128 + lane_idx] + p.eps);
            return row < n ? f : 0.f;
        };
        rn = norm_of(l, r);
        rk = kside ? rn : norm_of(r, r);
    }

    // ---- operand generation over one channel half; pw: this half's diagonal blocks take
    // the pairwise path (SM_BH then holds the in-block log2 prefix, k^ and q^ go to the
    // stash instead of K^R) ----
    const uint32_t bh_row = sbase + SM_BH + r * 256;
    const int swz = r & 7;
    const uint32_t tb_blk = sbase + SM_TAB + s * 8 * 256;
    const int row_g = kside ? r : 64 + r;     // record row of K^G / Q^G
    unsigned char *kqg_row = rec + REC_KQG + tc::core_offset(row_g, 0, 128, 2);
    const uint32_t bdiag_row = sbase + SM_BDIAG + tc::core_offset(r, 0, 64, 4);
    const uint32_t boff = sbase + SM_BOFF;
    const uint32_t kd_base = sbase + SM_SB + 8 * SBO_SB + static_cast<uint32_t>((r >> 3) * 128 + (r & 7) * 2);
    auto gen_half = [&](int hf, bool pw) {
        auto ld8 = [&](uint32_t addr, float *dst) {   // 8 floats at addr, addr + 16
            const float4 lo4 = ld_shared_f4(addr), hi4 = ld_shared_f4(addr + 16);
            dst[0] = lo4.x; dst[1] = lo4.y; dst[2] = lo4.z; dst[3] = lo4.w;
            dst[4] = hi4.x; dst[5] = hi4.y; dst[6] = hi4.z; dst[7] = hi4.w;
        };
        // the Q thread's key share: key row r, channels 32 sub + 16 .. + 31 of the half (half 0
        // from the staged tile, half 1 as the key thread left it)
        uint4 kq[2] = {kq0[0], kq0[1]};
        if (hf > 0 && !kside) {
            kq[0] = ld_shared_u4(sbase + SM_SB + (r * 2 + sub) * 32);
            kq[1] = ld_shared_u4(sbase + SM_SB + (r * 2 + sub) * 32 + 16);
        }
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int cl = 32 * sub + 8 * u;       // channel within the half
            const int c = 64 * hf + cl;            // channel within the head
            const uint32_t tbu = tb_blk + cl * 4;  // this block's constants of channels cl ..
            float x[8], e1[8], t[8], xe[8], v8[8];
            unpack_bf16x8(xr[hf][u], x);
            scale8(x, x, rn);
            {
                const int q = cl >> 2;
                const float4 lo4 = ld_shared_f4(bh_row + ((q ^ swz) << 4));
                const float4 hi4 = ld_shared_f4(bh_row + (((q + 1) ^ swz) << 4));
                e1[0] = lo4.x; e1[1] = lo4.y; e1[2] = lo4.z; e1[3] = lo4.w;
                e1[4] = hi4.x; e1[5] = hi4.y; e1[6] = hi4.z; e1[7] = hi4.w;
            }
            float lp[8];   // pairwise path: the in-block log2 prefix
            if (pw) {
#pragma unroll
                for (int o = 0; o < 8; o++) { lp[o] = e1[o]; e1[o] = ex2(lp[o]); }
            }
            mul8(xe, x, e1);
            {   // the A operand (tf32) -> tensor memory, lane l, column of the channel in the half
                uint32_t d8[8];
#pragma unroll
                for (int o = 0; o < 8; o++) d8[o] = tf32_rna(xe[o]);
                tc::tmem_st8u(tlane + TM_A + cl, d8);
                const uint4 h4 = pack8_f16(xe);
                const uint32_t d4[4] = {h4.x, h4.y, h4.z, h4.w};
                tc::tmem_st4u(tlane + TM_A16 + cl / 2, d4);
            }
            if (pw)      // the stash of the pairwise path: k^ / q^ in fp16
                st_shared_u4(sbase + SM_BDIAG + side * 8192 + stash_off(r, cl), pack8_f16(x));
            // K^G / Q^G = x e^{b} -> the record
            ld8(tbu + kE * 256, t);
            mul8(v8, xe, t);
            *reinterpret_cast<uint4 *>(kqg_row + (c >> 3) * 128) = pack8_f16(v8);
            // key-side share
            if (kside ? (u < 2) : (u >= 2)) {
                float kk[8], kf[8];
                if (kside) {
#pragma unroll
                    for (int o = 0; o < 8; o++) kk[o] = x[o];
                } else {
                    unpack_bf16x8(kq[u - 2], kk);
                    scale8(kk, kk, rk);
                }
                if (!pw) {
                    // K^R = k e^{P_s - b} = k / e1 (tf32) -> SM_BDIAG row r; k F = K^R e^{P_{s+1} - P_s}
#pragma unroll
                    for (int o = 0; o < 8; o++) v8[o] = kk[o] * rcp_approx(e1[o]);
                    st_shared_u4(bdiag_row + (cl >> 2) * 128, pack4_tf32(v8));
                    st_shared_u4(bdiag_row + ((cl >> 2) + 1) * 128, pack4_tf32(v8 + 4));
                    ld8(tbu + kBD * 256, t);
                    mul8(kf, v8, t);
                } else {   // k F = k e^{P_{s+1} - b} = k 2^{(block decay) - prefix}
                    ld8(tbu + kP1 * 256, t);
#pragma unroll
                    for (int o = 0; o < 8; o++) kf[o] = kk[o] * ex2(t[o] - lp[o]);
                }
                // B_R rows (R = s + 1 .. 3): k e^{P_R - b} -> SM_BOFF row off_b_base(R) + r
                if (s < 3) st_shared_u4(boff + tc::core_offset(off_b_base(s + 1) + r, cl, 64, 2), pack8_f16(kf));
                if (s < 2) {
                    ld8(tbu + kD2 * 256, t);
                    mul8(v8, kf, t);
                    st_shared_u4(boff + tc::core_offset(off_b_base(s + 2) + r, cl, 64, 2), pack8_f16(v8));
                }
                if (s < 1) {
                    ld8(tbu + kD3 * 256, t);
                    mul8(v8, kf, t);
                    st_shared_u4(boff + tc::core_offset(48 + r, cl, 64, 2), pack8_f16(v8));
                }
                // Kd^T = (k F e^{b_last - P_{s+1}})^T -> SB rows 64 + c
                ld8(tbu + kD4 * 256, t);
                mul8(v8, kf, t);
                const uint32_t kd = kd_base + static_cast<uint32_t>(c >> 3) * SBO_SB;
#pragma unroll
                for (int o = 0; o < 8; o++) st_shared_u16(kd + o * 16, f16_bits(v8[o]));
            }
        }
    };

    // ---- the pairwise diagonal blocks of one channel half (flagged halves): pair
    // pi = tid + 256 k of the 4 x 136 (row, column <= row) pairs of the diagonal blocks,
    // summed into registers (key rows: A before beta; query rows: Aqk) ----
    float pa[3] = {0.f, 0.f, 0.f}, pq[3] = {0.f, 0.f, 0.f};
    auto pair_of = [](int pi, int &rr, int &il) {
        const int sb = pi / 136, q = pi - sb * 136;
        int rl = static_cast<int>((sqrtf(8.f * q + 1.f) - 1.f) * 0.5f);
        if ((rl + 1) * (rl + 2) / 2 <= q) rl++;
        if (rl * (rl + 1) / 2 > q) rl--;
        il = q - rl * (rl + 1) / 2;
        rr = 16 * sb + rl;
    };
    auto pairwise_half = [&]() {
        const uint32_t ks = sbase + SM_BDIAG, qs = ks + 8192, bh = sbase + SM_BH;
#pragma unroll
        for (int k = 0; k < 3; k++) {
            const int pi = tid + 256 * k;
            if (pi < 4 * 136) {
                int rr, il;
                pair_of(pi, rr, il);
                const int ii = (rr & ~15) + il;
                float sa = 0.f, sq = 0.f;
                for (int cc = 0; cc < 64; cc += 8) {
                    float kr[8], ki[8], qr[8], br[8], bi[8];
                    unpack_f16x8(ld_shared_u4(ks + stash_off(rr, cc)), kr);
                    unpack_f16x8(ld_shared_u4(ks + stash_off(ii, cc)), ki);
                    unpack_f16x8(ld_shared_u4(qs + stash_off(rr, cc)), qr);
                    const float4 a0 = ld_shared_f4(bh + bh_off(rr, cc)), a1 = ld_shared_f4(bh + bh_off(rr, cc + 4));
                    const float4 c0 = ld_shared_f4(bh + bh_off(ii, cc)), c1 = ld_shared_f4(bh + bh_off(ii, cc + 4));
                    br[0] = a0.x; br[1] = a0.y; br[2] = a0.z; br[3] = a0.w; br[4] = a1.x; br[5] = a1.y; br[6] = a1.z; br[7] = a1.w;
                    bi[0] = c0.x; bi[1] = c0.y; bi[2] = c0.z; bi[3] = c0.w; bi[4] = c1.x; bi[5] = c1.y; bi[6] = c1.z; bi[7] = c1.w;
#pragma unroll
                    for (int o = 0; o < 8; o++) {
                        const float w = ex2(br[o] - bi[o]) * ki[o];
                        sa += kr[o] * w;
                        sq += qr[o] * w;
                    }
                }
                pa[k] += sa;
                pq[k] += sq;
            }
        }
    };
    auto issue_gram = [&](bool pw, bool acc_diag, bool acc_off) {
        if (tid == 0 || tid == 32) {
            tc::fence_after_sync();
            if (tid == 0)
                tc::gemm_ta<96, 64>(tmem + TM_XOFF, tmem + TM_A16, sbase + SM_BOFF, SBO64_F16, acc_off);
            else if (!pw)
                tc::gemm_ta_tf32<64, 64>(tmem + TM_XDIAG, tmem + TM_A, sbase + SM_BDIAG, SBO64_TF32, acc_diag);
            tc::commit(mbar);
        }
    };

    // ================= channel half 0 (its gate pass ran while q and k loaded) =================
    gen_half(0, pw0);
    tc::tmem_st_wait();
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    issue_gram(pw0, false, false);
    if (pw0) pairwise_half();
    // ================= channel half 1 =================
    bool fl1 = false, pw1 = false;
    if (nhalf == 2) {
        fl1 = gate_half(1);
        pw1 = PW && fl1;
        // the half-0 products read the A operand and SM_BOFF / SM_BDIAG, which half 1 rewrites
        ok &= cta_wait(mbar, phase, smem + SM_WAITOK);
        phase ^= 1;
        gen_half(1, pw1);
        tc::tmem_st_wait();
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        issue_gram(pw1, !pw0, true);
        if (pw1) pairwise_half();
    } else {
        // K = 64: channels 64 .. 127 hold no data. Their Kd^T rows are zero and their gamma is
        // 1, so the chain's state columns past K stay zero; their [K^G; Q^G] columns are not
        // written (the chain's products stop at K = 64).
        for (int i = tid; i < 8 * SBO_SB / 16; i += PT)
            st_shared_u4(sbase + SM_SB + 16 * SBO_SB + 16 * i, make_uint4(0u, 0u, 0u, 0u));
        if (tid < 64) reinterpret_cast<float *>(rec + REC_GAM)[64 + tid] = 1.f;
    }
    ok &= cta_wait(mbar, phase, smem + SM_WAITOK);
    phase ^= 1;
    // X_diag holds a product unless every half present took the pairwise path
    const bool mma_diag = nhalf == 2 ? !(pw0 && pw1) : !pw0, pw_diag = pw0 || pw1;
    if (pw_diag) {   // the pairwise sums -> SM_XD [side][row][column in the block]
        float *xd = reinterpret_cast<float *>(smem + SM_XD);
#pragma unroll
        for (int k = 0; k < 3; k++) {
            const int pi = tid + 256 * k;
            if (pi < 4 * 136) {
                int rr, il;
                pair_of(pi, rr, il);
                xd[rr * 16 + il] = pa[k];
                xd[1024 + rr * 16 + il] = pq[k];
            }
        }
        __syncthreads();
    }

    // ================= row assembly: A (fp32, with beta) and Aqk (fp16 into SB) =================
    // Thread (l, sub) writes column blocks k4 = 2 sub, 2 sub + 1 of row r: zero above the
    // diagonal block, the diagonal block from X_diag (+ the pairwise sums), the blocks
    // left of it from X_off at column off_b_base(s) + i. A warp covers row blocks s0 and
    // s0 + 1; its TMEM loads are collective, so it loads every source some lane needs.
    if (ok) {
        const int qd = warp & 3;          // lane quadrant: 0/1 K rows 0..31/32..63, 2/3 Q rows
        const int s0 = 2 * (qd & 1);
        const int rl = r & 15;
        const int lim = kside ? rl : rl + 1;   // diagonal-block columns < lim are kept
        const float br = kside ? betas[r] : 1.f;
        float *arow = reinterpret_cast<float *>(smem + SM_AMAT) + r * AP;
        const float *xdr = reinterpret_cast<const float *>(smem + SM_XD) + side * 1024 + r * 16;
#pragma unroll
        for (int kk = 0; kk < 2; kk++) {
            const int k4 = 2 * sub + kk;
            float off0[16], off1[16], dg[16], v[16];
            if (k4 < s0) tc::tmem_ld16(tlane + TM_XOFF + off_b_base(s0) + 16 * k4, off0);
            if (k4 <= s0) tc::tmem_ld16(tlane + TM_XOFF + off_b_base(s0 + 1) + 16 * k4, off1);
            if (mma_diag && (k4 == s0 || k4 == s0 + 1)) tc::tmem_ld16(tlane + TM_XDIAG + 16 * k4, dg);
            tc::tmem_ld_wait();
            if (k4 < s) {
                if (s == s0) {
#pragma unroll
                    for (int u = 0; u < 16; u++) v[u] = off0[u];
                } else {
#pragma unroll
                    for (int u = 0; u < 16; u++) v[u] = off1[u];
                }
            } else if (k4 == s) {
                if (!mma_diag) {
#pragma unroll
                    for (int u = 0; u < 16; u++) dg[u] = 0.f;
                }
                if (pw_diag) {
#pragma unroll
                    for (int u = 0; u < 16; u++) dg[u] += (u <= rl) ? xdr[u] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 16; u++) v[u] = u < lim ? dg[u] : 0.f;
            } else {
#pragma unroll
                for (int u = 0; u < 16; u++) v[u] = 0.f;
            }
            if (kside) {
#pragma unroll
                for (int u = 0; u < 16; u += 4) {
                    const float2 a = fmul2(make_float2(v[u], v[u + 1]), make_float2(br, br));
                    const float2 b = fmul2(make_float2(v[u + 2], v[u + 3]), make_float2(br, br));
                    *reinterpret_cast<float4 *>(arow + 16 * k4 + u) = make_float4(a.x, a.y, b.x, b.y);
                }
            } else {
                st_shared_u4(sbase + SM_SB + sb_offset(r, 16 * k4), pack8_f16(v));
                st_shared_u4(sbase + SM_SB + sb_offset(r, 16 * k4 + 8), pack8_f16(v + 8));
            }
        }
    }
    tc::fence_proxy_async();   // the Aqk rows of SB are read by the last products
    __syncthreads();

    // ================= T = (I + A)^-1, then [Aqk; Kd^T] T diag(beta) =================
    if (ok) {
        solve_T(smem, tid, sbase + SM_TT, betas);
        // last level on the tensor cores (tf32): X^T = T_a^T A_ba^T (32 x 32), then
        // T_ba^T = -(X^T T_b^T) with X^T read from tensor memory. Operand tiles (K-major,
        // 32 K, SBO 1024): T_a^T at SM_BDIAG (the product is M = 128: its rows 32..127 read
        // the rest of that region and land in lanes nothing reads), A_ba at SM_XTMP, T_b
        // at SM_XD. The upper triangles of T_a and T_b are not stored in SM_TMAT: zeros.
        const float *Tm = reinterpret_cast<const float *>(smem + SM_TMAT);
        const int row = tid & 31, k4 = (tid >> 5) * 4;  // one 16-byte chunk of each tile per thread
                                                         // (a warp: 32 rows of one K chunk)
        const uint32_t off = tc::core_offset(row, k4, 32, 4);
        {
            const float *Am = reinterpret_cast<const float *>(smem + SM_AMAT);
            float ta[4], ab[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int m = k4 + u;
                ta[u] = m >= row ? Tm[m * AP + row] : 0.f;                  // T_a^T[row][m] = T_a[m][row]
            }
            const float4 a4 = *reinterpret_cast<const float4 *>(Am + (32 + row) * AP + k4);   // A_ba[row][k4..]
            ab[0] = a4.x; ab[1] = a4.y; ab[2] = a4.z; ab[3] = a4.w;
            st_shared_u4(sbase + SM_BDIAG + off, pack4_tf32(ta));
            st_shared_u4(sbase + SM_XTMP + off, pack4_tf32(ab));
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0 || tid == 32) {
            tc::fence_after_sync();
            if (tid == 0) tc::gemm<2, 32, 32>(tmem + TM_L3X, sbase + SM_BDIAG, 1024, sbase + SM_XTMP, 1024, false);
            tc::commit(mbar);
        }
        {   // T_b, the second product's B operand, while the first runs
            const float4 b4 = *reinterpret_cast<const float4 *>(Tm + (32 + row) * AP + 32 + k4);   // T_b[row][k4..]
            float tb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int u = 0; u < 4; u++)
                if (k4 + u > row) tb[u] = 0.f;   // above T_b's diagonal: not stored
            st_shared_u4(sbase + SM_XD + off, pack4_tf32(tb));
            tc::fence_proxy_async();
        }
        ok &= cta_wait(mbar, phase, smem + SM_WAITOK);
        phase ^= 1;
    }
    if (ok) {
        if ((warp & 3) == 0) {   // X^T (lanes 0..31) rounded to tf32 in place: the next product's A
            // operand; warps 0 and 4 (both reach lanes 0..31) take 16 columns each
            const uint32_t col = TM_L3X + 16 * (warp >> 2);
            float x0[16];
            tc::tmem_ld16(tlane + col, x0);
            tc::tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; u++) x0[u] = __uint_as_float(tf32_rna(x0[u]));
            tc::tmem_st16(tlane + col, x0);
            tc::tmem_st_wait();
        }
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0 || tid == 32) {
            tc::fence_after_sync();
            if (tid == 0) tc::gemm_ta_tf32<32, 32>(tmem + TM_L3T, tmem + TM_L3X, sbase + SM_XD, 1024, false);
            tc::commit(mbar);
        }
        ok &= cta_wait(mbar, phase, smem + SM_WAITOK);
        phase ^= 1;
    }
    if (ok) {
        if ((warp & 3) == 0) {   // T_ba = -(X^T T_b^T)^T -> rows j of the (T diag(beta))^T tile,
            // K = 32..63; warps 0 and 4 take 16 columns each
            const int hv = warp >> 2;
            float y0[16];
            tc::tmem_ld16(tlane + TM_L3T + 16 * hv, y0);
            tc::tmem_ld_wait();
            const float nb = -betas[lane];
#pragma unroll
            for (int u = 0; u < 16; u++) y0[u] *= nb;
            const uint32_t tt = sbase + SM_TT;
            st_shared_u4(tt + tc::core_offset(lane, 32 + 16 * hv, 64, 2), pack8_f16(y0));
            st_shared_u4(tt + tc::core_offset(lane, 40 + 16 * hv, 64, 2), pack8_f16(y0 + 8));
        }
        tc::fence_proxy_async();   // the transpose is read by the products issued after the barrier
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0 || tid == 32) {
            tc::fence_after_sync();
            if (tid == 0)
                tc::gemm<0, 64, 64>(tmem + TM_W1, sbase + SM_SB, SBO_SB, sbase + SM_TT, SBO64_F16, false);
            else
                tc::gemm<0, 64, 64>(tmem + TM_W2, sbase + SM_SB + 8 * SBO_SB, SBO_SB, sbase + SM_TT, SBO64_F16, false);
            tc::commit(mbar);
        }
        ok &= cta_wait(mbar, phase, smem + SM_WAITOK);
        phase ^= 1;
    }
    // ================= [M1; M2] -> the record (left to the pass over marked units if the
    // pairwise path was needed and not taken) =================
    const bool marked = !PW && (fl0 || fl1);
    if (!PW && tid == 0) a.flags[a.flag0 + bid] = marked ? 1 : 0;
    if (ok && !marked) {
        float v[2][16], w1[2][16];
        tc::tmem_ld16(tlane + TM_W2 + 32 * sub, v[0]);
        tc::tmem_ld16(tlane + TM_W2 + 32 * sub + 16, v[1]);
        if (kside) {   // lanes 0..63 of the first product: M1 rows (loaded with the M2 rows)
            tc::tmem_ld16(tlane + TM_W1 + 32 * sub, w1[0]);
            tc::tmem_ld16(tlane + TM_W1 + 32 * sub + 16, w1[1]);
        }
        tc::tmem_ld_wait();
        unsigned char *mm = rec + REC_MM;
        bool bad = false;   // [M1; M2] travel in fp16
#pragma unroll
        for (int u = 0; u < 16; u++) bad |= !(fabsf(v[0][u]) < 65504.f) || !(fabsf(v[1][u]) < 65504.f);
        if (__any_sync(0xffffffffu, bad) && lane == 0 && p.err) atomicOr(p.err, kErrRange);
#pragma unroll
        for (int q = 0; q < 4; q++)
            *reinterpret_cast<uint4 *>(mm + tc::core_offset(64 + l, 32 * sub + 8 * q, 64, 2)) = pack8_f16(&v[q >> 1][8 * (q & 1)]);
        if (kside) {
#pragma unroll
            for (int q = 0; q < 4; q++)
                *reinterpret_cast<uint4 *>(mm + tc::core_offset(l, 32 * sub + 8 * q, 64, 2)) = pack8_f16(&w1[q >> 1][8 * (q & 1)]);
        }
    } else if (!ok && tid == 0 && p.err) {
        atomicOr(p.err, kErrTimeout);
    }
    if (PW) tc::fence_proxy_async();   // the next unit's tensor copies overwrite these regions
    tc::fence_before_sync();
    __syncthreads();
    };

    // ---- (PW) the next marked unit at or after unit pos whose rank among the marked units
    // (rk: the rank of the first marked unit at or after pos) is congruent to this CTA's
    // index modulo the grid, or -1; pos and rk move past it. Every CTA counts ranks over
    // the same flags, so each marked unit goes to exactly one CTA. A window is 16 flags
    // (one 16-byte load) per thread. ----
    auto next_marked = [&](int &pos, int &rk) -> int {
        int *sc = reinterpret_cast<int *>(smem + SM_TOT);   // [8] per-warp counts, [8] the unit found
        const int G = static_cast<int>(gridDim.x), me = static_cast<int>(blockIdx.x);
        while (pos < total) {
            const int g0 = (a.flag0 + pos) & ~15;    // flag index of the window's start
            const int gi = g0 + 16 * tid;            // this thread's 16 flags
            uint32_t bits = 0;                       // bit j: flag gi + j is set, within [pos, total)
            if (gi - a.flag0 < total) {
                const uint4 f = __ldcg(reinterpret_cast<const uint4 *>(a.flags + gi));   // from L2
                const uint32_t w4[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int u = gi + j - a.flag0;
                    if (((w4[j >> 2] >> (8 * (j & 3))) & 0xffu) != 0u && u >= pos && u < total) bits |= 1u << j;
                }
            }
            const int cnt = __popc(bits);
            int incl = cnt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += y;
            }
            if (lane == 31) sc[warp] = incl;
            __syncthreads();
            int before = 0, all = 0;
#pragma unroll
            for (int w = 0; w < PT / 32; w++) {
                const int c = sc[w];
                before += w < warp ? c : 0;
                all += c;
            }
            const int want = rk + ((me - rk) % G + G) % G;   // the first rank >= rk that is this CTA's
            const bool found = want < rk + all;
            if (found) {
                const int k = want - rk - (before + incl - cnt);   // among this thread's marked flags
                if (k >= 0 && k < cnt) {
                    uint32_t b = bits;
                    for (int i = 0; i < k; i++) b &= b - 1u;
                    sc[8] = gi + __ffs(static_cast<int>(b)) - 1 - a.flag0;
                }
            }
            __syncthreads();
            if (found) {
                const int u = sc[8];
                pos = u + 1;
                rk = want + 1;
                return u;
            }
            pos = g0 + 16 * PT - a.flag0;
            rk += all;
            __syncthreads();   // the counts are rewritten by the next window
        }
        return -1;
    };

    uint32_t lpar = 0;   // parity of the copy barriers for the current unit
    if (!PW) {
        const int bid = static_cast<int>(blockIdx.x);
        int h, n, sq = -1;
        int64_t row0;
        locate(bid, h, row0, n, sq);
        // launched by launch_pdl: the barriers, the unit's location and the tensor-map
        // prefetches above read kernel parameters only; every global read comes after this
        pdl_wait_then_release();
        issue_loads(bid, h, row0, sq);
        alloc_tmem();
        compute(bid, h, row0, n, 0u);
    } else {
        pdl_wait_then_release();   // the first pass's flags are complete
        alloc_tmem();
        int pos = 0, rk = 0;
        for (;;) {
            const int u = next_marked(pos, rk);
            if (u < 0) break;
            int h, n, sq = -1;
            int64_t row0;
            locate(u, h, row0, n, sq);
            issue_loads(u, h, row0, sq);
            compute(u, h, row0, n, lpar);
            if (!ok) break;
            lpar ^= 1u;
        }
    }
    if (!ok && tid == 0) {   // a wait gave up: give the copies and the product it waited for (bounded) time to end
        (void)tc::mbar_wait(lbar, lpar);
        (void)tc::mbar_wait(lbar + 8, lpar);
        (void)tc::mbar_wait(mbar, phase ^ 1u);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc<256>(tmem);
}

// ---------------------------------------------------------------------------
// chain_kernel: one CTA of 256 threads per (sequence, head) chain, one CTA per SM.
// Thread (j, sub): TMEM lane j = 32 (warp & 3) + lane (value column), sub = warp >> 2.
// ---------------------------------------------------------------------------
constexpr uint32_t CH_KQ = 0;             // [2] record part A (33280 B each, 1024-aligned slots)
constexpr uint32_t CH_KQ_STRIDE = 33792;
constexpr uint32_t CH_MM = 2 * CH_KQ_STRIDE;   // [2] record part B (24576 B each)
constexpr uint32_t CH_VT = CH_MM + 2 * REC_B_BYTES;   // [2] bf16 [64][128] V tiles, swizzled
constexpr uint32_t CH_BAR = CH_VT + 2 * 16384;        // mbarriers: kq[2], mm[2], mma
constexpr uint32_t CH_TMEMP = CH_BAR + 40;
constexpr uint32_t CH_WAITOK = CH_TMEMP + 4;
constexpr uint32_t CHAIN_SMEM = CH_WAITOK + 4;
static_assert(CH_BAR % 8 == 0, "mbarrier alignment");

// chain tensor memory columns (512)
constexpr uint32_t TC_PK = 0;      // (K^G S)^T      64 columns
constexpr uint32_t TC_PQ = 64;     // (Q^G S)^T -> O^T   64 columns
constexpr uint32_t TC_S = 128;     // S^T           128 columns
constexpr uint32_t TC_AS = 256;    // S^T as fp16 pairs (A of P)   64 columns
constexpr uint32_t TC_AY = 320;    // Y^T as fp16 pairs (A of the O/S product)   32 columns
constexpr uint32_t TC_PK2 = 384;   // the second K half of (K^G S)^T   64 columns
constexpr uint32_t TC_PQ2 = 448;   // the second K half of (Q^G S)^T   64 columns

template <int NH, int NV>   // key channel and value column halves that hold data: K = 64 NH, V = 64 NV
__global__ void __launch_bounds__(CT, 1) chain_kernel(const __grid_constant__ Args a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    const Params &p = a.p;
    pdl_wait_then_release();   // launched by launch_pdl: no global read before this
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int rank = static_cast<int>(blockIdx.x / H), h = static_cast<int>(blockIdx.x % H);
    const int sq = a.order[rank];
    const int64_t e = a.entry_base + sq;
    const int64_t row0 = a.rs[sq], row1 = a.rs[sq + 1];
    const int64_t slot = load_slot(p, e);
    const int j = 32 * (warp & 3) + lane, sub = warp >> 2;
    constexpr int kr = 64 * NH, vr = 64 * NV;   // state rows (channels) and columns that hold data
    if (slot >= p.num_slots) {      // flagged before the length check: empty sequences too
        if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
        for (int64_t t = row0 + (tid >> 6); t < row1; t += CT / 64) {
            uint32_t *o = reinterpret_cast<uint32_t *>(p.out + t * p.ld_out + static_cast<int64_t>(h) * vr);
            if ((tid & 63) < vr / 2) o[tid & 63] = 0u;
        }
        return;
    }
    if (row1 <= row0) return;
    const bool has_state = slot >= 0;
    const bool writable = has_state && slot != p.null_slot;
    float *tile = has_state ? p.pool + slot * p.slot_stride + static_cast<int64_t>(h) * kr * vr : nullptr;
    const int nch = static_cast<int>((row1 - row0 + C - 1) / C);
    const unsigned char *rec0 = a.rec + (static_cast<size_t>(a.cb[sq]) * H + h) * REC_BYTES;
    const size_t rec_step = static_cast<size_t>(H) * REC_BYTES;
    const int64_t HK = static_cast<int64_t>(H) * kr;

    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t bar = sbase + CH_BAR;   // kq[0], kq[1], mm[0], mm[1], mma
    if (tid == 0) {
        for (int i = 0; i < 4; i++) tc::mbar_init(bar + 8 * i, 1);
        tc::mbar_init(bar + 32, 2);   // the chain products: two issuing threads commit
    }
    if (warp == 0) tc::tmem_alloc<512>(sbase + CH_TMEMP);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + CH_TMEMP);
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);

    // prefetch the first two chunks' records and V tiles
    auto issue_kq = [&](int c) {
        const uint32_t b = c & 1;
        tc::mbar_expect_tx(bar + 8 * b, REC_A_BYTES);
        tc::bulk_g2s(sbase + CH_KQ + b * CH_KQ_STRIDE, rec0 + c * rec_step, REC_A_BYTES, bar + 8 * b);
    };
    auto issue_mm = [&](int c) {
        const uint32_t b = c & 1;
        tc::mbar_expect_tx(bar + 16 + 8 * b, REC_B_BYTES);
        tc::bulk_g2s(sbase + CH_MM + b * REC_B_BYTES, rec0 + c * rec_step + REC_MM, REC_B_BYTES, bar + 16 + 8 * b);
    };
    auto stage_v = [&](int c) {
        const int64_t r0 = row0 + static_cast<int64_t>(c) * C;
        const int nn = static_cast<int>((row1 - r0) < C ? (row1 - r0) : C);
        stage_rows<CT>(sbase + CH_VT + (c & 1) * 16384, p.qkv + r0 * p.ld_qkv + 2 * HK + static_cast<int64_t>(h) * vr,
                       p.ld_qkv, nn, tid, vr / 8);
    };
    // chunk whose copy into buffer b is in flight and not yet waited for (-1: none)
    int kq_pending[2] = {-1, -1}, mm_pending[2] = {-1, -1};
    if (tid == 0) {
        for (int c = 0; c < 2 && c < nch; c++) { issue_kq(c); issue_mm(c); }
    }
    for (int c = 0; c < 2 && c < nch; c++) { kq_pending[c] = c; mm_pending[c] = c; }
    stage_v(0);
    cp_async_commit();
    if (nch > 1) stage_v(1);
    cp_async_commit();

    // ---- S0 -> TMEM (S^T: lane j, columns c in this thread's half) ----
#pragma unroll
    for (int cc = 0; cc < 64; cc += 16) {
        float v[16];
        const int c = 64 * sub + cc;
        const bool in = has_state && c < kr && j < vr;   // the group of 16 channels is in or out whole
#pragma unroll
        for (int u = 0; u < 16; u++) v[u] = in ? tile[static_cast<int64_t>(c + u) * vr + j] : 0.f;
        tc::tmem_st16(tlane + TC_S + c, v);
    }
    if (kr < KD) {   // the second K half of P is not computed: its accumulators stay zero
        float z[16];
#pragma unroll
        for (int u = 0; u < 16; u++) z[u] = 0.f;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 16) tc::tmem_st16(tlane + (sub ? TC_PQ2 : TC_PK2) + cc, z);
    }
    tc::tmem_st_wait();

    bool ok = true;
    uint32_t phc = 0;
    int nprev = 0;
    int64_t prev0 = row0;
    // a value that left the fp16 range on the way (the state, Y or an operand) reaches the
    // outputs and the state as Inf or NaN: flag it (once per warp)
    auto flag_nonfinite = [&](bool bad) {
        if (__any_sync(0xffffffffu, bad) && lane == 0 && p.err) atomicOr(p.err, kErrRange);
    };
    auto store_o = [&](const float (&ov)[2][16], int64_t cs, int nrows) {
        uint16_t *orow = p.out + cs * p.ld_out + static_cast<int64_t>(h) * vr + j;
        if (j >= vr) nrows = 0;   // columns past V hold no data
        bool bad = false;
#pragma unroll
        for (int q = 0; q < 2; q++)
#pragma unroll
            for (int u = 0; u < 16; u++) {
                const int rr = 32 * sub + 16 * q + u;
                bad |= !(fabsf(ov[q][u]) < INFINITY) && rr < nrows;
                if (rr < nrows) orow[static_cast<int64_t>(rr) * p.ld_out] = f32_to_bf16(ov[q][u]);
            }
        flag_nonfinite(bad);
    };
    for (int c = 0; c < nch; c++) {
        const int b = c & 1;
        const uint32_t par = static_cast<uint32_t>(c >> 1) & 1u;
        const int64_t c0 = row0 + static_cast<int64_t>(c) * C;
        const int n = static_cast<int>((row1 - c0) < C ? (row1 - c0) : C);
        // ---- D1: the record's [K^G; Q^G] and gamma have landed ----
        ok &= cta_wait(bar + 8 * b, par, smem + CH_WAITOK);
        kq_pending[b] = -1;
        if (!ok) break;
        // D1: S^T -> fp16 pairs (the A operand of P); O^T of the previous chunk, read
        // before P overwrites it. All TMEM loads are issued before one wait.
        float ov[2][16], ow[2][16], sv[4][16];
        if (c > 0) {
            tc::tmem_ld16(tlane + TC_PQ + 32 * sub, ov[0]);
            tc::tmem_ld16(tlane + TC_PQ + 32 * sub + 16, ov[1]);
            tc::tmem_ld16(tlane + TC_PQ2 + 32 * sub, ow[0]);
            tc::tmem_ld16(tlane + TC_PQ2 + 32 * sub + 16, ow[1]);
        }
#pragma unroll
        for (int q = 0; q < 4; q++) tc::tmem_ld16(tlane + TC_S + 64 * sub + 16 * q, sv[q]);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t pk8[8];
#pragma unroll
            for (int i = 0; i < 8; i++) pk8[i] = tc::pack_f16x2(sv[q][2 * i], sv[q][2 * i + 1]);
            tc::tmem_st8u(tlane + TC_AS + 32 * sub + 8 * q, pk8);
        }
        {   // S^T <- S^T Diag(gamma), stored before P is issued (TMEM stores beside a running
            // product slow it down; P reads the fp16 copy only)
            const float *gam = reinterpret_cast<const float *>(smem + CH_KQ + b * CH_KQ_STRIDE + REC_GAM);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int cidx = 64 * sub + 16 * q;
#pragma unroll
                for (int u = 0; u < 16; u += 4) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(gam + cidx + u);
                    sv[q][u] *= g4.x; sv[q][u + 1] *= g4.y; sv[q][u + 2] *= g4.z; sv[q][u + 3] *= g4.w;
                }
                tc::tmem_st16(tlane + TC_S + cidx, sv[q]);
            }
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0 || tid == 32) {   // P = [(K^G S)^T | (Q^G S)^T], one half per issuing thread, each
            tc::fence_after_sync();      // as two accumulators over the two channel halves
            const uint32_t half = tid == 0 ? 0u : 64u;
            tc::gemm_ta_split<64, 128, NH>(tmem + TC_PK + half, tmem + TC_PK2 + half, tmem + TC_AS,
                                           sbase + CH_KQ + b * CH_KQ_STRIDE + half * 2 * 128, SBO128_F16);
            tc::commit(bar + 32);
        }
        // while P runs: the previous chunk's O rows, and this chunk's V values
        if (c > 0) {
#pragma unroll
            for (int q = 0; q < 2; q++)
#pragma unroll
                for (int u = 0; u < 16; u++) ov[q][u] += ow[q][u];
            store_o(ov, prev0, nprev);
        }
        cp_async_wait_group<1>();   // this chunk's V tile (the newer group may fly)
        ok &= cta_wait(bar + 32, phc, smem + CH_WAITOK);   // P done; the barrier publishes V
        phc ^= 1;
        if (!ok) break;
        if (c + 2 < nch) {
            if (tid == 0) issue_kq(c + 2);
            kq_pending[b] = c + 2;
        }
        // ---- Y^T = (V - K^G S)^T -> fp16 pairs in TMEM ----
        {
            const uint16_t *vt = reinterpret_cast<const uint16_t *>(smem + CH_VT + b * 16384);
            float pv[2][16], pw[2][16];
            tc::tmem_ld16(tlane + TC_PK + 32 * sub, pv[0]);
            tc::tmem_ld16(tlane + TC_PK + 32 * sub + 16, pv[1]);
            tc::tmem_ld16(tlane + TC_PK2 + 32 * sub, pw[0]);
            tc::tmem_ld16(tlane + TC_PK2 + 32 * sub + 16, pw[1]);
            float vv[2][16];
#pragma unroll
            for (int q = 0; q < 2; q++)
#pragma unroll
                for (int u = 0; u < 16; u++) {
                    const int rr = 32 * sub + 16 * q + u;
                    vv[q][u] = bf16_to_f32(vt[(st_off(rr, j >> 3) >> 1) + (j & 7)]);
                }
            tc::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 2; q++) {
                uint32_t pk8[8];
#pragma unroll
                for (int i = 0; i < 8; i++)
                    pk8[i] = tc::pack_f16x2(vv[q][2 * i] - (pv[q][2 * i] + pw[q][2 * i]),
                                            vv[q][2 * i + 1] - (pv[q][2 * i + 1] + pw[q][2 * i + 1]));
                tc::tmem_st8u(tlane + TC_AY + 16 * sub + 8 * q, pk8);
            }
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncthreads();
        // the V tile of this chunk is consumed: stage chunk c + 2's
        if (c + 2 < nch) stage_v(c + 2);
        cp_async_commit();
        bool mm_ok = true;
        if (tid == 0 || tid == 32) {   // [O^T | S^T] += Y^T [M1; M2]^T: O^T on one thread, S^T on the other
            mm_ok = tc::mbar_wait(bar + 16 + 8 * b, par);
            if (mm_ok) {
                tc::fence_after_sync();
                if (tid == 0)
                    tc::gemm_ta<64, 64>(tmem + TC_PQ, tmem + TC_AY, sbase + CH_MM + b * REC_B_BYTES, SBO64_F16, true);
                else
                    tc::gemm_ta<64 * NH, 64>(tmem + TC_S, tmem + TC_AY, sbase + CH_MM + b * REC_B_BYTES + 8 * 1024,
                                             SBO64_F16, true);   // K = 64: the state columns past K stay zero
            }
            tc::commit(bar + 32);
        }
        mm_pending[b] = -1;
        ok &= cta_wait(bar + 32, phc, smem + CH_WAITOK, mm_ok);
        phc ^= 1;
        if (!ok) break;
        if (c + 2 < nch) {
            if (tid == 0) issue_mm(c + 2);
            mm_pending[b] = c + 2;
        }
        prev0 = c0;
        nprev = n;
    }
    if (ok) {
        float ov[2][16], ow[2][16];
        tc::tmem_ld16(tlane + TC_PQ + 32 * sub, ov[0]);
        tc::tmem_ld16(tlane + TC_PQ + 32 * sub + 16, ov[1]);
        tc::tmem_ld16(tlane + TC_PQ2 + 32 * sub, ow[0]);
        tc::tmem_ld16(tlane + TC_PQ2 + 32 * sub + 16, ow[1]);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 2; q++)
#pragma unroll
            for (int u = 0; u < 16; u++) ov[q][u] += ow[q][u];
        store_o(ov, prev0, nprev);
        if (writable) {
            bool bad = false;
#pragma unroll
            for (int cc = 0; cc < 64; cc += 16) {
                float v[16];
                const int cidx = 64 * sub + cc;
                tc::tmem_ld16(tlane + TC_S + cidx, v);
                tc::tmem_ld_wait();
                if (cidx < kr && j < vr) {   // K is a multiple of 16: the group is in or out whole
#pragma unroll
                    for (int u = 0; u < 16; u++) {
                        bad |= !(fabsf(v[u]) < INFINITY);
                        tile[static_cast<int64_t>(cidx + u) * vr + j] = v[u];
                    }
                }
            }
            flag_nonfinite(bad);
        }
    } else {
        // a wait gave up: record it, then let the copies this CTA started finish (bounded)
        // before its shared and tensor memory are released
        if (tid == 0) {
            if (p.err) atomicOr(p.err, kErrTimeout);
            for (int b = 0; b < 2; b++) {
                if (kq_pending[b] >= 0) (void)tc::mbar_wait(bar + 8 * b, static_cast<uint32_t>(kq_pending[b] >> 1) & 1u);
                if (mm_pending[b] >= 0) (void)tc::mbar_wait(bar + 16 + 8 * b, static_cast<uint32_t>(mm_pending[b] >> 1) & 1u);
            }
            (void)tc::mbar_wait(bar + 32, phc);   // a product that was issued but not seen complete
        }
        cp_async_wait_all();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc<512>(tmem);
}

}  // namespace chunk

// One CTA of 512 threads waits, as the tensor-core kernels do (one warp polls, the rest
// park on the barrier), on an mbarrier that nothing arrives at. The bounded wait gives up
// after ~2 s; the kernel then records the timeout in the error word and returns normally.
__global__ void __launch_bounds__(512, 1) bounded_wait_selftest_kernel(uint32_t *err)
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

cudaError_t launch_bounded_wait_selftest(uint32_t *err, cudaStream_t stream)
{
    bounded_wait_selftest_kernel<<<1, 512, 0, stream>>>(err);
    return cudaGetLastError();
}

// Workspace of a K = V = 128 prefill: one record per (chunk, head).
static int64_t total_chunks(const int32_t *cu_host, int64_t num_seqs)
{
    int64_t t = 0;
    for (int64_t s = 0; s < num_seqs; s++) t += (static_cast<int64_t>(cu_host[s + 1]) - cu_host[s] + chunk::C - 1) / chunk::C;
    return t;
}

// Head sizes the tensor-core path takes: K and V each 64 or 128 (both run on 128 x 128
// tiles; at 64 the channels or columns past the data are held at zero).
static bool chunk_dims(int K, int V) { return (K == 64 || K == 128) && (V == 64 || V == 128); }

// The records, then one flag byte per record (rounded up to 16 bytes).
size_t chunk_workspace_bytes(const int32_t *cu_host, int64_t num_seqs, int H, int K, int V, int)
{
    if (!chunk_dims(K, V) || num_seqs <= 0) return 0;
    const size_t units = static_cast<size_t>(total_chunks(cu_host, num_seqs)) * H;
    if (units == 0) return 0;
    return units * chunk::REC_BYTES + (units + 15) / 16 * 16;
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link against the driver library)
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// A tensor map over a bf16 matrix of `rows` rows x `cols` columns with a row pitch of `ld`
// elements, read in boxes of 64 rows x 64 columns (128 bytes) with the 128-byte swizzle.
// Rows past the matrix read as zeros.
static cudaError_t encode_rows_map(CUtensorMap *m, const void *base, int64_t cols, int64_t rows, int64_t ld)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorSymbolNotFound;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The prefill chains of entries [entry_base, entry_base + num_seqs): per launch of at most
// kMaxSeqs sequences, the prep pass over every (chunk, head), then the chains (longest
// sequence first).
// after_prep: if not null, recorded on `stream` once the first launch's prep kernel is
// enqueued (before its chain kernel).
static cudaError_t launch_chunk_path(const Params &p, int K, int V, const int32_t *cu, const int32_t *cu_host,
                                     int64_t entry_base, int64_t num_seqs, void *workspace,
                                     cudaStream_t stream, cudaEvent_t after_prep = nullptr)
{
    using namespace chunk;
    static_assert(sizeof(Args) < 32000, "kernel parameter space");
    cudaError_t err;
    // the instances for this K and V (64: one half of the 128-wide tile holds data, 128: two)
    void (*prep)(Args) = K == 64 ? (p.has_lb ? prep_kernel<1, false, true> : prep_kernel<1, false, false>)
                                 : (p.has_lb ? prep_kernel<2, false, true> : prep_kernel<2, false, false>);
    void (*prep_pw)(Args) = K == 64 ? prep_kernel<1, true, false> : prep_kernel<2, true, false>;
    void (*chain)(Args) = K == 64 ? (V == 64 ? chain_kernel<1, 1> : chain_kernel<1, 2>)
                                  : (V == 64 ? chain_kernel<2, 1> : chain_kernel<2, 2>);
    if ((err = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(PREP_SMEM))) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(prep_pw, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(PREP_SMEM))) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(CHAIN_SMEM))) != cudaSuccess) return err;
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    unsigned char *recs = static_cast<unsigned char *>(workspace);
    // the unit flags follow every record of the call
    unsigned char *flags = recs + static_cast<size_t>(total_chunks(cu_host + entry_base, num_seqs)) * p.H * REC_BYTES;
    int64_t ch_done = 0;   // chunks (not chunk-heads) of the sequences already launched
    std::vector<int32_t> ord;
    // tensor maps over the rows of this call (every row any of its chunks reads lies below
    // the last sequence's end)
    const int64_t rows = std::max<int64_t>(cu_host[entry_base + num_seqs], 1);
    CUtensorMap tm_qkv, tm_g;
    if ((err = encode_rows_map(&tm_qkv, p.qkv, 2 * static_cast<int64_t>(p.H) * K + static_cast<int64_t>(p.H) * V,
                               rows, p.ld_qkv)) != cudaSuccess) return err;
    if ((err = encode_rows_map(&tm_g, p.rg, static_cast<int64_t>(p.H) * K, rows, p.ld_g)) != cudaSuccess) return err;
    for (int64_t s0 = 0; s0 < num_seqs; s0 += kMaxSeqs) {
        const int64_t ns = std::min<int64_t>(kMaxSeqs, num_seqs - s0);
        Args a;
        a.tm_qkv = tm_qkv;
        a.tm_g = tm_g;
        a.p = p;
        a.cu = cu;
        a.entry_base = entry_base + s0;
        a.num_seqs = static_cast<int32_t>(ns);
        a.pf_stride = 2 * sms;
        a.rec = recs + static_cast<size_t>(ch_done) * p.H * REC_BYTES;
        a.flags = flags;
        a.flag0 = static_cast<int32_t>(ch_done * p.H);
        const int32_t *cuh = cu_host + entry_base + s0;
        a.cb[0] = 0;
        for (int64_t i = 0; i < ns; i++)
            a.cb[i + 1] = a.cb[i] + static_cast<int32_t>((static_cast<int64_t>(cuh[i + 1]) - cuh[i] + C - 1) / C);
        for (int64_t i = 0; i <= ns; i++) a.rs[i] = cuh[i];
        ord.resize(static_cast<size_t>(ns));
        std::iota(ord.begin(), ord.end(), 0);
        std::stable_sort(ord.begin(), ord.end(), [cuh](int32_t x, int32_t y) {
            return (cuh[x + 1] - cuh[x]) > (cuh[y + 1] - cuh[y]);
        });
        for (int64_t i = 0; i < ns; i++) a.order[i] = ord[static_cast<size_t>(i)];
        const int64_t nch = a.cb[ns];
        if (nch > 0) {
            const int64_t units = nch * p.H;
            if ((err = launch_pdl(prep, dim3(static_cast<unsigned>(units)), dim3(PT), PREP_SMEM, stream, a)) !=
                cudaSuccess) return err;
            if (after_prep && s0 == 0 && (err = cudaEventRecord(after_prep, stream)) != cudaSuccess) return err;
            // the units marked by the first pass (none, usually: its CTAs find that and end)
            const int64_t g = std::min<int64_t>(units, 2 * static_cast<int64_t>(sms));
            if ((err = launch_pdl(prep_pw, dim3(static_cast<unsigned>(g)), dim3(PT), PREP_SMEM, stream, a)) !=
                cudaSuccess) return err;
        } else if (after_prep && s0 == 0 && (err = cudaEventRecord(after_prep, stream)) != cudaSuccess) {
            return err;
        }
        // every sequence gets a chain CTA: empty ones check their slot and return
        if ((err = launch_pdl(chain, dim3(static_cast<unsigned>(ns * p.H)), dim3(CT), CHAIN_SMEM, stream, a)) !=
            cudaSuccess) return err;
        ch_done += nch;
    }
    return cudaSuccess;
}

cudaError_t launch_chunk_prefill(const Params &p, int K, int V, const int32_t *cu,
                                 const int32_t *cu_host, int64_t entry_base, int64_t num_seqs,
                                 int, void *workspace, size_t, cudaStream_t stream)
{
    if (num_seqs <= 0) return cudaSuccess;
    if (!chunk_dims(K, V))  // other head sizes take the token-recurrent kernel
        return launch_recurrent(p, K, V, 2, 1, cu, entry_base, num_seqs, stream);
    return launch_chunk_path(p, K, V, cu, cu_host, entry_base, num_seqs, workspace, stream);
}

// Mixed batch: the decodes (entries [0, num_decodes), one row each) take the packed-decode
// kernel, the prefills the chunk path.
// The side stream a mixed batch hands its decodes to, and its two events: one set per
// device, created on first use (lowest stream priority, no timing) and kept.
namespace {
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t after_prep = nullptr, join = nullptr;
};
constexpr int kMaxSideDevices = 64;
SideStream g_side[kMaxSideDevices];
std::mutex g_side_mutex;   // guards the creation and every hand-over ... join sequence
}  // namespace

static cudaError_t side_stream_locked(SideStream **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxSideDevices) return cudaErrorInvalidDevice;
    SideStream &ss = g_side[dev];
    if (!ss.s) {
        int lo = 0, hi = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithPriority(&ss.s, cudaStreamNonBlocking, lo)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&ss.after_prep, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &ss;
    return cudaSuccess;
}

cudaError_t launch_mixed(const Params &p, int K, int V, const int32_t *cu, const int32_t *cu_host,
                         int64_t num_decodes, int64_t num_prefills, void *workspace, cudaStream_t stream)
{
    if (num_decodes > 0 && num_prefills > 0 && chunk_dims(K, V)) {
        // The decodes run beside the prefill chains: a chain CTA holds a whole SM and the
        // chains of a batch rarely fill the GPU, so the (HBM-bound) decodes go to a
        // low-priority side stream that starts once the prep kernel is done, takes the SMs
        // the chains leave, and is joined back before the call returns.
        std::lock_guard<std::mutex> lock(g_side_mutex);
        SideStream *ss = nullptr;
        cudaError_t e = side_stream_locked(&ss);
        if (e != cudaSuccess) return e;
        if ((e = launch_chunk_path(p, K, V, cu, cu_host, num_decodes, num_prefills, workspace, stream,
                                   ss->after_prep)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(ss->s, ss->after_prep, 0)) != cudaSuccess) return e;
        if ((e = launch_decode(p, K, V, cu_host[0], num_decodes, ss->s)) != cudaSuccess) return e;
        if ((e = cudaEventRecord(ss->join, ss->s)) != cudaSuccess) return e;
        return cudaStreamWaitEvent(stream, ss->join, 0);
    }
    if (num_decodes > 0) {
        cudaError_t e = launch_decode(p, K, V, cu_host[0], num_decodes, stream);
        if (e != cudaSuccess) return e;
    }
    return launch_chunk_prefill(p, K, V, cu, cu_host, num_decodes, num_prefills, 64, workspace, 0, stream);
}

}  // namespace kda
