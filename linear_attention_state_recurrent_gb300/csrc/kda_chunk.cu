// Chunked varlen prefill on tcgen05 tensor cores (K = V = 128, chunk C = 64).
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
//                 tensor cores, the triangular solve and [Aqk; Kd^T] T diag(beta) on the
//                 tensor cores. It writes one record per (chunk, head) to the workspace:
//                 [K^G; Q^G] (fp16), gamma (fp32) and [M1; M2] (fp16), each already in the
//                 shared-memory layout the chain's MMAs read.
//   chain_kernel  one CTA per (sequence, head) chain (one per SM): the state stays in
//                 tensor memory, transposed (lane = value column j, column = key channel);
//                 per chunk two products
//                   P = S^T [K^G; Q^G]^T                 M=128 N=128 K=128  fp16
//                   [O^T | S^T] += Y^T [M1; M2]^T         M=128 N=192 K=64   fp16
//                 with S^T pre-scaled by gamma, the records streamed in by bulk copies two
//                 chunks ahead.
// A chunk where some channel decays by more than 40 nats within half a 16-row block (or
// 80 within a block) leaves the tensor-core Gram path: the prep CTA lists it and
// exact_kernel recomputes its record in fp32 on the CUDA cores.
//
// The decay-weighted Gram matrices are split into 16-row blocks s = 0..3 with prefixes
// P_s = b at the last row before block s. Off-diagonal blocks are computed in fp16 with
// a reference point between the two rows, so both factors are <= 1 (a factor that
// underflows only drops a term that is itself below 2^-24):
//   block (1,0): reference P_1;  blocks (2|3, 0|1): reference P_2;  block (3,2): P_3,
//   X_off = OFFA OFFB^T  with OFFA = [K^e; Q^e] rows (16..31 @P_1, 32..63 @P_2, and
//   48..63 @P_3 on lanes 0..15) and OFFB = [rows 0..31 @P_2; rows 0..15 @P_1; rows
//   32..47 @P_3]  (M=128 N=64 K=128, A in tensor memory).
// Diagonal blocks use the block's eighth row as reference, whose factors reach e^{40},
// in tf32:  X_diag = [K^L; Q^L] (K^R)^T  (M=128 N=64, K=128 in two channel halves, A in
// tensor memory).
//
// fp16 (11-bit significand, round to nearest) carries the same precision as tf32 with
// round to nearest; bf16 operands would exceed the 2e-3 relative error bar.
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
constexpr int PT = 256;          // prep / exact threads
constexpr int CT = 256;          // chain threads
constexpr int kMaxSeqs = 1024;   // sequences per launch (the host splits larger calls)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kHalfSpan2 = 40.f * kLog2e;    // largest half-block decay of the tf32 path (log2 units)
constexpr float kBlockSpan2 = 80.f * kLog2e;   // largest block decay of the factored path

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
constexpr uint32_t SM_G = 0;            // bf16 [64][128] raw_g, 16-byte chunks XOR-swizzled by row
constexpr uint32_t SM_BH = 16384;       // fp32 [64][64]  b (log2 units) of the current channel half, swizzled
constexpr uint32_t SM_OFFB = 32768;     // fp16 [64][128] off-diagonal B operand (SBO 2048)
constexpr uint32_t SM_DIAGB = 49152;    // tf32 [64][64]  K^R of the current channel half (SBO 2048)
constexpr uint32_t SM_SB = 65536;       // fp16 [192][64] Aqk rows 0..63, Kd^T rows 64..191 (SBO 1040)
constexpr uint32_t SM_TAB = SM_SB + 24 * SBO_SB;   // fp32 [4 blocks][8][64] per-(block, channel) constants
constexpr uint32_t SM_TOT = SM_TAB + 8192;         // fp32 [4][64] block sums of g
constexpr uint32_t SM_NRM = SM_TOT + 1024;         // fp32 [2][128] half-row |k|^2, |q|^2
constexpr uint32_t SM_BETA = SM_NRM + 1024;        // fp32 [64]
constexpr uint32_t SM_MBAR = SM_BETA + 256;        // mbarrier of the MMAs (two committing threads)
constexpr uint32_t SM_TMEMP = SM_MBAR + 8;
constexpr uint32_t SM_WAITOK = SM_TMEMP + 4;
constexpr uint32_t PREP_SMEM = SM_WAITOK + 4;
static_assert(SM_MBAR % 8 == 0, "mbarrier alignment");
static_assert(2 * (PREP_SMEM + 1024) <= 233472, "two prep CTAs per SM");
// solve-phase aliases over SM_G .. SM_DIAGB (dead once the Gram products are done)
constexpr uint32_t SM_AMAT = 0;        // fp32 [64][68]
constexpr uint32_t SM_TMAT = 17408;    // fp32 [64][68]
constexpr uint32_t SM_XTMP = 34816;    // fp32 scratch (<= 4608 B)
constexpr uint32_t SM_TT = 40960;      // fp16 [64][64] (T diag(beta))^T, K-major SBO 1024
constexpr int AP = 68;                 // fp32 row pitch of AMAT / TMAT
static_assert(SM_TT + 8192 <= SM_SB, "solve scratch overlaps SB");

// ---- prep tensor memory columns (256) ----
constexpr uint32_t TM_XOFF = 0;     // 64 columns
constexpr uint32_t TM_XDIAG = 64;   // 64 columns
constexpr uint32_t TM_OFFA = 128;   // fp16 A operand of X_off, packed pairs (64 columns)
constexpr uint32_t TM_DIAGA = 192;  // tf32 A operand of X_diag, current channel half (64 columns)
constexpr uint32_t TM_W1 = 0;       // [Aqk; Kd^T rows 0..63] T diag(beta)   (after assembly)
constexpr uint32_t TM_W2 = 64;      // Kd^T T diag(beta)

// per-(block, channel) constants (log2 units for prefixes)
enum Tab { kP0 = 0, kP1 = 1, kTL = 2, kTR = 3, kE = 4, kD4 = 5, kDa = 6 };

struct Args {
    Params p;
    const int32_t *cu;         // device cu_seqlens (entries)
    int64_t entry_base;        // first entry of this launch
    int32_t num_seqs;
    int32_t num_decodes;       // (unused by the prefill kernels)
    unsigned char *rec;        // records of this launch: (chunk, head) at (cb + j) * H + h
    uint32_t *flag_count;      // chunks that left the tensor-core Gram path
    uint32_t *flag_list;
    int32_t cb[kMaxSeqs + 1];  // chunk prefix over the launch's sequences
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
__device__ __forceinline__ uint4 pack4_tf32(const float *v)
{
    return make_uint4(tc::to_tf32(v[0]), tc::to_tf32(v[1]), tc::to_tf32(v[2]), tc::to_tf32(v[3]));
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
    return static_cast<uint32_t>(r * 256 + ((((c >> 2) ^ (r & 15))) << 4) + (c & 3) * 4);
}
// byte offset of fp16 element (row, k) of SB (K = 64, padded block stride SBO_SB)
__device__ __forceinline__ uint32_t sb_offset(int row, int k)
{
    return static_cast<uint32_t>((row >> 3) * SBO_SB + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}
__device__ __forceinline__ uint32_t tab_off(int s, int k, int c) { return static_cast<uint32_t>(((s * 8 + k) * 64 + c) * 4); }

// Copies rows [0, 64) of one 128-wide bf16 column block (base + row*ld) into a staged tile
// with NTH threads; rows at or past `nrows` are zero-filled (their source is not read).
template <int NTH>
__device__ __forceinline__ void stage_rows(uint32_t tile, const uint16_t *base, int64_t ld, int nrows, int tid)
{
#pragma unroll
    for (int x = 0; x < 1024 / NTH; x++) {
        const int id = tid + NTH * x, r = id >> 4, ch = id & 15;
        const bool ok = r < nrows;
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

// ---------------------------------------------------------------------------
// T = (I + A)^-1 for the strictly lower 64x64 A in AMAT (fp32, pitch AP) by 16x16
// diagonal-block inverses and two levels of block doubling (256 threads). Each level
// writes its final entries of T diag(beta), transposed and in fp16, to the operand tile
// at `tbt` (row m, K = k holds T[k][m] beta_m); the six zero blocks of the transpose are
// written during the first level, so the tile is complete (and fenced for the async
// proxy) when the solve returns. The fp32 T keeps only what later levels read.
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
    // level 2: within each 32-block p, X = A_10 T_00 then T_10 = -T_11 X (16x16)
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const int id = tid + 256 * it, p = id >> 8, r = (id >> 4) & 15, j = id & 15, o = 32 * p;
        float x = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m++) x += A[(o + 16 + r) * AP + o + m] * T[(o + m) * AP + o + j];
        X[(p * 16 + r) * 17 + j] = x;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 2; it++) {
        const int id = tid + 256 * it, p = id >> 8, r = (id >> 4) & 15, j = id & 15, o = 32 * p;
        float y = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m++)
            if (m <= r) y += T[(o + 16 + r) * AP + o + 16 + m] * X[(p * 16 + m) * 17 + j];
        T[(o + 16 + r) * AP + o + j] = -y;
        st_shared_u16(tbt + tc::core_offset(o + j, o + 16 + r, 64, 2), f16_bits(-y * beta[o + j]));
    }
    __syncthreads();
    // level 3: X = A_ba T_a (32x32), T_ba = -T_b X; 2x2 output tiles
    {
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
    {
        const int r = (tid >> 4) * 2, j = (tid & 15) * 2;
        float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
        for (int m = 0; m <= r + 1; m++) {       // T_b is lower triangular: m <= row
            const float t0 = (m <= r) ? T[(32 + r) * AP + 32 + m] : 0.f;
            const float t1 = T[(33 + r) * AP + 32 + m];
            const float2 x = *reinterpret_cast<const float2 *>(X + m * 36 + j);
            y00 += t0 * x.x; y01 += t0 * x.y;
            y10 += t1 * x.x; y11 += t1 * x.y;
        }
        // T_ba is final and read by no later level: only its scaled fp16 transpose is
        // stored, rows 32 + r, 33 + r of columns j, j + 1 as K pairs of rows j, j + 1
        const float bj0 = beta[j], bj1 = beta[j + 1];
        st_shared_u32(tbt + tc::core_offset(j, 32 + r, 64, 2), tc::pack_f16x2(-y00 * bj0, -y10 * bj0));
        st_shared_u32(tbt + tc::core_offset(j + 1, 32 + r, 64, 2), tc::pack_f16x2(-y01 * bj1, -y11 * bj1));
    }
    tc::fence_proxy_async();   // the transpose is read by the products issued after the barrier
    __syncthreads();
}

// ---------------------------------------------------------------------------
// prep_kernel: one CTA of 256 threads per (chunk, head); two CTAs per SM.
//
// Thread roles: TMEM lane l = 32 (warp & 3) + lane and channel quarter sub = warp >> 2.
// Lanes 0..63 are the K side (key row r = l), lanes 64..127 the Q side (query row
// r = l - 64); in a channel half a thread covers channels 32 sub .. 32 sub + 31.
// The gate pass uses channel c = tid & 63 of the half and row block tid >> 6.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(PT, 2) prep_kernel(const __grid_constant__ Args a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    const Params &p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int cgi = static_cast<int>(blockIdx.x / H), h = static_cast<int>(blockIdx.x % H);
    int lo = 0, hi = a.num_seqs - 1;   // the sequence: the last s with cb[s] <= cgi
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cb[mid] <= cgi) lo = mid; else hi = mid - 1;
    }
    const int64_t e = a.entry_base + lo;
    const int64_t row0 = static_cast<int64_t>(a.cu[e]) + static_cast<int64_t>(cgi - a.cb[lo]) * C;
    const int64_t rem = static_cast<int64_t>(a.cu[e + 1]) - row0;
    const int n = static_cast<int>(rem < C ? rem : C);
    unsigned char *rec = a.rec + static_cast<size_t>(blockIdx.x) * REC_BYTES;
    const int64_t HK = static_cast<int64_t>(H) * KD;

    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t mbar = sbase + SM_MBAR;
    float *tab = reinterpret_cast<float *>(smem + SM_TAB);
    float *tot = reinterpret_cast<float *>(smem + SM_TOT);
    float *nrm = reinterpret_cast<float *>(smem + SM_NRM);
    float *betas = reinterpret_cast<float *>(smem + SM_BETA);

    // ---- stage raw_g, start the norm pass ----
    stage_rows<PT>(sbase + SM_G, p.rg + row0 * p.ld_g + static_cast<int64_t>(h) * KD, p.ld_g, n, tid);
    cp_async_commit();
    if (tid == 0) tc::mbar_init(mbar, 2);   // two issuing threads commit to every MMA stage
    if (warp == 0) tc::tmem_alloc<256>(sbase + SM_TMEMP);
    const int l = 32 * (warp & 3) + lane, sub = warp >> 2;
    const bool kside = l < 64;
    const int r = l & 63, s = r >> 4;
    // own row: [half][16 bf16 pairs] = channels 64 hf + 32 sub .. + 31
    uint4 xr[2][4];
    {
        const uint16_t *src = p.qkv + (row0 + r) * p.ld_qkv + (kside ? HK : 0) + static_cast<int64_t>(h) * KD + 32 * sub;
        float ss = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; hf++)
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++) {
                const uint4 v = r < n ? __ldg(reinterpret_cast<const uint4 *>(src + 64 * hf + 8 * q4)) : make_uint4(0u, 0u, 0u, 0u);
                xr[hf][q4] = v;
                float f[8];
                unpack_bf16x8(v, f);
#pragma unroll
                for (int o = 0; o < 8; o++) ss += f[o] * f[o];
            }
        nrm[sub * 128 + l] = ss;
    }
    if (tid < C) betas[tid] = tid < n ? sigmoid_f(bf16_to_f32(p.rb[(row0 + tid) * p.ld_beta + h])) : 0.f;
    const float expA = __expf(__ldg(p.A_log + h));
    cp_async_wait_all();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SM_TMEMP);
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    // rows past the chunk hold zeros; their norm factor is 0 so that eps = 0 gives no NaN
    auto norm_of = [&](int lane_idx, int row) -> float {
        const float f = (lane_idx < 64 ? 1.f : p.scale) * rsqrtf(nrm[lane_idx] + nrm[128 + lane_idx] + p.eps);
        return row < n ? f : 0.f;
    };
    const float rn = norm_of(l, r);
    uint32_t phase = 0;
    bool ok = true;

    // ---- gate pass over one channel half: b (log2 units) into SM_BH, the constants
    // table, gamma into the record; returns whether the chunk leaves the tf32 path ----
    auto gate_half = [&](int hf) -> bool {
        const int c = tid & 63, sg = tid >> 6, cg = 64 * hf + c;
        const float dtb = p.dt_bias ? __ldg(p.dt_bias + h * KD + cg) : 0.f;
        const uint16_t *gt = reinterpret_cast<const uint16_t *>(smem + SM_G);
        float v[16];
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const int row = 16 * sg + j;
            const float x = bf16_to_f32(gt[(st_off(row, cg >> 3) >> 1) + (cg & 7)]) + dtb;
            const float g = row < n ? kLog2e * gate_log_decay_fast(x, expA, p.has_lb, p.lb) : 0.f;
            acc += g;
            v[j] = acc;
        }
        tot[sg * 64 + c] = acc;
        __syncthreads();
        float P0 = 0.f, P4 = 0.f;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const float t = tot[q * 64 + c];
            if (q < sg) P0 += t;
            P4 += t;
        }
        const float P1 = P0 + acc;
        float *bh = reinterpret_cast<float *>(smem + SM_BH);
#pragma unroll
        for (int j = 0; j < 16; j++) bh[bh_off(16 * sg + j, c) >> 2] = P0 + v[j];
        const float m2 = P0 + v[7];
        tab[tab_off(sg, kP0, c) >> 2] = P0;
        tab[tab_off(sg, kP1, c) >> 2] = P1;
        tab[tab_off(sg, kTL, c) >> 2] = ex2(P0 - m2);
        tab[tab_off(sg, kTR, c) >> 2] = ex2(m2 - P1);
        tab[tab_off(sg, kE, c) >> 2] = ex2(P0);
        tab[tab_off(sg, kD4, c) >> 2] = ex2(P4 - P1);
        tab[tab_off(sg, kDa, c) >> 2] = sg == 0 ? ex2(tot[64 + c]) : (sg == 3 ? ex2(tot[128 + c]) : 1.f);
        if (sg == 3) reinterpret_cast<float *>(rec + REC_GAM)[cg] = ex2(P4);
        const int fl = (v[0] - v[7] > kHalfSpan2) || (v[7] - v[15] > kHalfSpan2) || (-acc > kBlockSpan2);
        return __syncthreads_or(fl) != 0;
    };

    // ---- operand generation over one channel half ----
    auto gen_half = [&](int hf) {
        const uint32_t bh = sbase + SM_BH, tb = sbase + SM_TAB;
        const bool extra = r < 16;       // this lane also holds the off-diagonal row 48 + r
        uint4 xe[4];
        float rne = 0.f;
        if (extra) {
            const int re = 48 + r;
            const uint16_t *src = p.qkv + (row0 + re) * p.ld_qkv + (kside ? HK : 0) + static_cast<int64_t>(h) * KD +
                                  64 * hf + 32 * sub;
#pragma unroll
            for (int q4 = 0; q4 < 4; q4++)
                xe[q4] = re < n ? __ldg(reinterpret_cast<const uint4 *>(src + 8 * q4)) : make_uint4(0u, 0u, 0u, 0u);
            rne = norm_of(l + 48, re);
        }
        const int row_g = kside ? r : 64 + r;     // record row of K^G / Q^G
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int cl = 32 * sub + 8 * u;      // channel within the half
            const int c = 64 * hf + cl;           // channel within the head
            float x[8], b2[8], t[8], e1[8], v8[8];
            unpack_bf16x8(xr[hf][u], x);
#pragma unroll
            for (int o = 0; o < 8; o++) x[o] *= rn;
            {
                const float4 lo4 = ld_shared_f4(bh + bh_off(r, cl)), hi4 = ld_shared_f4(bh + bh_off(r, cl + 4));
                b2[0] = lo4.x; b2[1] = lo4.y; b2[2] = lo4.z; b2[3] = lo4.w;
                b2[4] = hi4.x; b2[5] = hi4.y; b2[6] = hi4.z; b2[7] = hi4.w;
            }
            auto tab8 = [&](int blk, int k, float *dst) {
                const float4 lo4 = ld_shared_f4(tb + tab_off(blk, k, cl)), hi4 = ld_shared_f4(tb + tab_off(blk, k, cl + 4));
                dst[0] = lo4.x; dst[1] = lo4.y; dst[2] = lo4.z; dst[3] = lo4.w;
                dst[4] = hi4.x; dst[5] = hi4.y; dst[6] = hi4.z; dst[7] = hi4.w;
            };
            tab8(s, kP0, t);
#pragma unroll
            for (int o = 0; o < 8; o++) e1[o] = ex2(b2[o] - t[o]);   // e^{b - P_s} <= 1
            // K^L / Q^L (tf32) -> tensor memory, lane l, column of the channel in the half
            tab8(s, kTL, t);
            {
                uint32_t d8[8];
#pragma unroll
                for (int o = 0; o < 8; o++) d8[o] = tc::to_tf32(x[o] * e1[o] * t[o]);
                tc::tmem_st8u(tlane + TM_DIAGA + cl, d8);
            }
            // K^G / Q^G = x e^{b} -> the record
            tab8(s, kE, t);
#pragma unroll
            for (int o = 0; o < 8; o++) v8[o] = x[o] * e1[o] * t[o];
            *reinterpret_cast<uint4 *>(rec + REC_KQG + tc::core_offset(row_g, c, 128, 2)) = pack8_f16(v8);
            // off-diagonal A operand (fp16 pairs -> tensor memory)
            if (!extra) {
                if (r >= 48) {   // rows 48..63 against rows 0..31: reference P_2 = P_3 - (block 2's decay)
                    tab8(3, kDa, t);
#pragma unroll
                    for (int o = 0; o < 8; o++) v8[o] = x[o] * e1[o] * t[o];
                } else {
#pragma unroll
                    for (int o = 0; o < 8; o++) v8[o] = x[o] * e1[o];
                }
            } else {             // row 48 + r against block 2: reference P_3
                float xx[8], be[8];
                unpack_bf16x8(xe[u], xx);
                const float4 lo4 = ld_shared_f4(bh + bh_off(48 + r, cl)), hi4 = ld_shared_f4(bh + bh_off(48 + r, cl + 4));
                be[0] = lo4.x; be[1] = lo4.y; be[2] = lo4.z; be[3] = lo4.w;
                be[4] = hi4.x; be[5] = hi4.y; be[6] = hi4.z; be[7] = hi4.w;
                tab8(3, kP0, t);
#pragma unroll
                for (int o = 0; o < 8; o++) v8[o] = xx[o] * rne * ex2(be[o] - t[o]);
            }
            {
                uint32_t a4[4];
#pragma unroll
                for (int o = 0; o < 4; o++) a4[o] = tc::pack_f16x2(v8[2 * o], v8[2 * o + 1]);
                tc::tmem_st4u(tlane + TM_OFFA + (c >> 1), a4);
            }
            if (kside) {
                // F = e^{P_{s+1} - b} <= 1; k F is the key row against later references
                tab8(s, kP1, t);
                float kf[8];
#pragma unroll
                for (int o = 0; o < 8; o++) kf[o] = x[o] * ex2(t[o] - b2[o]);
                // K^R (tf32) -> SM_DIAGB row r
                tab8(s, kTR, t);
#pragma unroll
                for (int o = 0; o < 8; o++) v8[o] = kf[o] * t[o];
                st_shared_u4(sbase + SM_DIAGB + tc::core_offset(r, cl, 64, 4), pack4_tf32(v8));
                st_shared_u4(sbase + SM_DIAGB + tc::core_offset(r, cl + 4, 64, 4), pack4_tf32(v8 + 4));
                // rows of the off-diagonal B operand
                const uint32_t ob = sbase + SM_OFFB;
                if (s == 0) {
                    tab8(0, kDa, t);
#pragma unroll
                    for (int o = 0; o < 8; o++) v8[o] = kf[o] * t[o];
                    st_shared_u4(ob + tc::core_offset(r, c, 128, 2), pack8_f16(v8));
                    st_shared_u4(ob + tc::core_offset(32 + r, c, 128, 2), pack8_f16(kf));
                } else if (s == 1) {
                    st_shared_u4(ob + tc::core_offset(r, c, 128, 2), pack8_f16(kf));
                } else if (s == 2) {
                    st_shared_u4(ob + tc::core_offset(16 + r, c, 128, 2), pack8_f16(kf));
                }
                // Kd^T = (k F e^{b_last - P_{s+1}})^T -> SB rows 64 + c
                tab8(s, kD4, t);
#pragma unroll
                for (int o = 0; o < 8; o++)
                    st_shared_u16(sbase + SM_SB + sb_offset(64 + c + o, r), f16_bits(kf[o] * t[o]));
            }
        }
    };

    // ================= channel half 0 =================
    bool flagged = gate_half(0);
    if (!flagged) {
        gen_half(0);
        tc::tmem_st_wait();
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0 || tid == 32) {
            tc::fence_after_sync();
            if (tid == 32)
                tc::gemm_ta_tf32<64, 64>(tmem + TM_XDIAG, tmem + TM_DIAGA, sbase + SM_DIAGB, SBO64_TF32, false);
            tc::commit(mbar);
        }
        // ================= channel half 1 =================
        flagged = gate_half(1);
        // the half-0 diagonal product reads SM_DIAGB and TM_DIAGA, which half 1 rewrites
        ok &= cta_wait(mbar, phase, smem + SM_WAITOK);
        phase ^= 1;
    }
    if (flagged || !ok) {
        if (tid == 0) {
            if (!ok) {
                if (p.err) atomicOr(p.err, kErrTimeout);
            } else {
                const uint32_t slot = atomicAdd(a.flag_count, 1u);
                a.flag_list[slot] = blockIdx.x;
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::tmem_dealloc<256>(tmem);
        return;
    }
    gen_half(1);
    tc::tmem_st_wait();
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 || tid == 32) {
        tc::fence_after_sync();
        if (tid == 0)
            tc::gemm_ta<64, 128>(tmem + TM_XOFF, tmem + TM_OFFA, sbase + SM_OFFB, SBO128_F16, false);
        else
            tc::gemm_ta_tf32<64, 64>(tmem + TM_XDIAG, tmem + TM_DIAGA, sbase + SM_DIAGB, SBO64_TF32, true);
        tc::commit(mbar);
    }
    ok &= cta_wait(mbar, phase, smem + SM_WAITOK);
    phase ^= 1;

    // ================= row assembly: A (fp32, with beta) and Aqk (fp16 into SB) =================
    if (ok) {
        const int qd = warp & 3;          // lane quadrant: 0/1 K rows 0..31/32..63, 2/3 Q rows
        const bool hiq = (qd & 1) != 0;   // rows 32..63 (blocks 2, 3)
        const float beta_r = kside ? betas[r] : 1.f;
        float *amat = reinterpret_cast<float *>(smem + SM_AMAT);
        auto put = [&](int row, int k4, const float *v) {   // 16 entries of row `row`, columns 16 k4 ..
            if (kside) {
                const float br = betas[row];
                float *dst = amat + row * AP + 16 * k4;
#pragma unroll
                for (int u = 0; u < 16; u += 4)
                    *reinterpret_cast<float4 *>(dst + u) = make_float4(v[u] * br, v[u + 1] * br, v[u + 2] * br, v[u + 3] * br);
            } else {
                st_shared_u4(sbase + SM_SB + sb_offset(row, 16 * k4), pack8_f16(v));
                st_shared_u4(sbase + SM_SB + sb_offset(row, 16 * k4 + 8), pack8_f16(v + 8));
            }
        };
        (void)beta_r;
#pragma unroll
        for (int kk = 0; kk < 2; kk++) {
            const int k4 = 2 * sub + kk;
            float v[16], w[16];
            // warp-uniform sources of this segment
            uint32_t src0 = 0xffffffffu, src1 = 0xffffffffu;
            if (!hiq) {
                if (k4 == 0) { src0 = TM_XDIAG + 0; src1 = TM_XOFF + 32; }
                else if (k4 == 1) src0 = TM_XDIAG + 16;
                else if (k4 == 2) src1 = TM_XOFF + 48;    // rows 48 + r, block (3, 2), lanes r < 16
            } else {
                if (k4 == 0) src0 = TM_XOFF + 0;
                else if (k4 == 1) src0 = TM_XOFF + 16;
                else if (k4 == 2) src0 = TM_XDIAG + 32;
                else src0 = TM_XDIAG + 48;
            }
            if (src0 != 0xffffffffu) tc::tmem_ld16(tlane + src0, v);
            if (src1 != 0xffffffffu) tc::tmem_ld16(tlane + src1, w);
            tc::tmem_ld_wait();
            float o[16];
            bool write_own = true;
            if (k4 > s) {
#pragma unroll
                for (int u = 0; u < 16; u++) o[u] = 0.f;
            } else if (k4 == s) {     // diagonal block: strictly lower for A, lower for Aqk
#pragma unroll
                for (int u = 0; u < 16; u++) {
                    const int i = 16 * k4 + u;
                    o[u] = (kside ? (i < r) : (i <= r)) ? v[u] : 0.f;
                }
            } else if (s == 1) {      // block (1, 0)
#pragma unroll
                for (int u = 0; u < 16; u++) o[u] = w[u];
            } else if (k4 < 2) {      // blocks (2|3, 0|1)
#pragma unroll
                for (int u = 0; u < 16; u++) o[u] = v[u];
            } else {                  // block (3, 2): written by lane r - 48
                write_own = false;
            }
            if (write_own) put(r, k4, o);
            if (!hiq && k4 == 2 && r < 16) put(48 + r, 2, w);
        }
    }
    tc::fence_proxy_async();   // the Aqk rows of SB are read by the last products
    __syncthreads();

    // ================= T = (I + A)^-1, then [Aqk; Kd^T] T diag(beta) =================
    if (ok) {
        solve_T(smem, tid, sbase + SM_TT, betas);
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
    // ================= [M1; M2] -> the record =================
    if (ok) {
        float v[2][16];
        tc::tmem_ld16(tlane + TM_W2 + 32 * sub, v[0]);
        tc::tmem_ld16(tlane + TM_W2 + 32 * sub + 16, v[1]);
        tc::tmem_ld_wait();
        unsigned char *mm = rec + REC_MM;
#pragma unroll
        for (int q = 0; q < 4; q++)
            *reinterpret_cast<uint4 *>(mm + tc::core_offset(64 + l, 32 * sub + 8 * q, 64, 2)) = pack8_f16(&v[q >> 1][8 * (q & 1)]);
        if (kside) {   // lanes 0..63 of the first product: M1 rows
            tc::tmem_ld16(tlane + TM_W1 + 32 * sub, v[0]);
            tc::tmem_ld16(tlane + TM_W1 + 32 * sub + 16, v[1]);
            tc::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; q++)
                *reinterpret_cast<uint4 *>(mm + tc::core_offset(l, 32 * sub + 8 * q, 64, 2)) = pack8_f16(&v[q >> 1][8 * (q & 1)]);
        }
    } else if (tid == 0 && p.err) {
        atomicOr(p.err, kErrTimeout);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc<256>(tmem);
}

// ---------------------------------------------------------------------------
// exact_kernel: the record of every (chunk, head) that prep_kernel listed, in fp32 on the
// CUDA cores with pairwise exponentials (no factoring, so no range limit on the decay).
// One CTA of 256 threads per listed record, grid-stride over the list.
// ---------------------------------------------------------------------------
constexpr uint32_t EX_KH = 0;            // fp32 [64][128] k^ (then Kd)
constexpr uint32_t EX_QH = 32768;        // fp32 [64][128] q^
constexpr uint32_t EX_BB = 65536;        // fp32 [64][128] b (natural log units)
constexpr uint32_t EX_AM = 98304;        // fp32 [64][68] A
constexpr uint32_t EX_TM = EX_AM + 17408;   // fp32 [64][68] T
constexpr uint32_t EX_AQ = EX_TM + 17408;   // fp32 [64][68] Aqk
constexpr uint32_t EX_BETA = EX_AQ + 17408; // fp32 [64]
constexpr uint32_t EX_NRM = EX_BETA + 256;  // fp32 [2][64]
constexpr uint32_t EXACT_SMEM = EX_NRM + 512;

__global__ void __launch_bounds__(PT, 1) exact_kernel(const __grid_constant__ Args a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    const Params &p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    float *KH = reinterpret_cast<float *>(smem + EX_KH);
    float *QH = reinterpret_cast<float *>(smem + EX_QH);
    float *BB = reinterpret_cast<float *>(smem + EX_BB);
    float *AM = reinterpret_cast<float *>(smem + EX_AM);
    float *TM = reinterpret_cast<float *>(smem + EX_TM);
    float *AQ = reinterpret_cast<float *>(smem + EX_AQ);
    float *bet = reinterpret_cast<float *>(smem + EX_BETA);
    float *nq = reinterpret_cast<float *>(smem + EX_NRM);
    const uint32_t count = *reinterpret_cast<volatile uint32_t *>(a.flag_count);
    for (uint32_t idx = blockIdx.x; idx < count; idx += gridDim.x) {
        const uint32_t bid = a.flag_list[idx];
        const int cgi = static_cast<int>(bid / H), h = static_cast<int>(bid % H);
        int lo = 0, hi = a.num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cb[mid] <= cgi) lo = mid; else hi = mid - 1;
        }
        const int64_t e = a.entry_base + lo;
        const int64_t row0 = static_cast<int64_t>(a.cu[e]) + static_cast<int64_t>(cgi - a.cb[lo]) * C;
        const int64_t rem = static_cast<int64_t>(a.cu[e + 1]) - row0;
        const int n = static_cast<int>(rem < C ? rem : C);
        unsigned char *rec = a.rec + static_cast<size_t>(bid) * REC_BYTES;
        const int64_t HK = static_cast<int64_t>(H) * KD;
        __syncthreads();   // the previous record's reads of shared memory are done
        // raw q, k
        for (int i = tid; i < C * KD; i += PT) {
            const int rr = i >> 7, c = i & 127;
            const uint16_t *row = p.qkv + (row0 + rr) * p.ld_qkv + static_cast<int64_t>(h) * KD + c;
            QH[i] = rr < n ? bf16_to_f32(row[0]) : 0.f;
            KH[i] = rr < n ? bf16_to_f32(row[HK]) : 0.f;
        }
        if (tid < C) bet[tid] = tid < n ? sigmoid_f(bf16_to_f32(p.rb[(row0 + tid) * p.ld_beta + h])) : 0.f;
        __syncthreads();
        // norms: warp w handles rows w, w + 8, ...
        for (int rr = warp; rr < C; rr += PT / 32) {
            float sq = 0.f, sk = 0.f;
            for (int c = lane; c < KD; c += 32) {
                sq += QH[rr * KD + c] * QH[rr * KD + c];
                sk += KH[rr * KD + c] * KH[rr * KD + c];
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            if (lane == 0) {
                nq[rr] = rr < n ? p.scale * rsqrtf(sq + p.eps) : 0.f;
                nq[64 + rr] = rr < n ? rsqrtf(sk + p.eps) : 0.f;
            }
        }
        __syncthreads();
        for (int i = tid; i < C * KD; i += PT) {
            QH[i] *= nq[i >> 7];
            KH[i] *= nq[64 + (i >> 7)];
        }
        // gate and cumulative decay: thread c < 128 walks the rows
        if (tid < KD) {
            const float expA = expf(__ldg(p.A_log + h));
            const float dtb = p.dt_bias ? __ldg(p.dt_bias + h * KD + tid) : 0.f;
            float acc = 0.f;
            for (int rr = 0; rr < C; rr++) {
                if (rr < n)
                    acc += gate_log_decay(bf16_to_f32(p.rg[(row0 + rr) * p.ld_g + static_cast<int64_t>(h) * KD + tid]) + dtb,
                                          expA, p.has_lb, p.lb);
                BB[rr * KD + tid] = acc;
            }
            reinterpret_cast<float *>(rec + REC_GAM)[tid] = expf(acc);
        }
        __syncthreads();
        // A and Aqk pairwise: warp per pair (rr, i), i <= rr, 4 channels per lane
        for (int pr = warp; pr < C * (C + 1) / 2; pr += PT / 32) {
            int rr = static_cast<int>((sqrtf(8.f * pr + 1.f) - 1.f) * 0.5f);
            if ((rr + 1) * (rr + 2) / 2 <= pr) rr++;
            if (rr * (rr + 1) / 2 > pr) rr--;
            const int i = pr - rr * (rr + 1) / 2;
            float sa = 0.f, sq = 0.f;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int c = 4 * lane + q;
                const float ex = expf(BB[rr * KD + c] - BB[i * KD + c]) * KH[i * KD + c];
                sa += KH[rr * KD + c] * ex;
                sq += QH[rr * KD + c] * ex;
            }
            sa = warp_sum(sa);
            sq = warp_sum(sq);
            if (lane == 0) {
                AM[rr * AP + i] = i < rr ? bet[rr] * sa : 0.f;
                AQ[rr * AP + i] = sq;
            }
        }
        __syncthreads();
        // T = (I + A)^-1, column j by forward substitution
        if (tid < C) {
            const int j = tid;
            for (int rr = 0; rr < C; rr++) {
                float t = 0.f;
                if (rr == j) t = 1.f;
                else if (rr > j) {
                    for (int m = j; m < rr; m++) t -= AM[rr * AP + m] * TM[m * AP + j];
                }
                TM[rr * AP + j] = t;
            }
        }
        // K^G, Q^G (record) and Kd = k^ e^{b_last - b} (in place of k^)
        for (int i = tid; i < C * KD; i += PT) {
            const int rr = i >> 7, c = i & 127;
            const float g = expf(BB[i]);
            reinterpret_cast<uint16_t *>(rec + REC_KQG)[tc::core_offset(rr, c, 128, 2) >> 1] = f16_bits(KH[i] * g);
            reinterpret_cast<uint16_t *>(rec + REC_KQG)[tc::core_offset(64 + rr, c, 128, 2) >> 1] = f16_bits(QH[i] * g);
        }
        __syncthreads();
        for (int i = tid; i < C * KD; i += PT) KH[i] *= expf(BB[(C - 1) * KD + (i & 127)] - BB[i]);
        __syncthreads();
        // M1[i][m] = beta_m sum_r Aqk[i][r] T[r][m];  M2[c][m] = beta_m sum_r Kd[r][c] T[r][m]
        for (int o = tid; o < 192 * C; o += PT) {
            const int row = o >> 6, m = o & 63;
            float acc = 0.f;
            if (row < C) {
                for (int rr = m; rr <= row; rr++) acc += AQ[row * AP + rr] * TM[rr * AP + m];
            } else {
                const int c = row - C;
                for (int rr = m; rr < C; rr++) acc += KH[rr * KD + c] * TM[rr * AP + m];
            }
            reinterpret_cast<uint16_t *>(rec + REC_MM)[tc::core_offset(row, m, 64, 2) >> 1] = f16_bits(acc * bet[m]);
        }
    }
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

__global__ void __launch_bounds__(CT, 1) chain_kernel(const __grid_constant__ Args a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    const Params &p = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int rank = static_cast<int>(blockIdx.x / H), h = static_cast<int>(blockIdx.x % H);
    const int sq = a.order[rank];
    const int64_t e = a.entry_base + sq;
    const int64_t row0 = a.cu[e], row1 = a.cu[e + 1];
    const int64_t slot = load_slot(p, e);
    const int j = 32 * (warp & 3) + lane, sub = warp >> 2;
    if (slot >= p.num_slots) {      // flagged before the length check: empty sequences too
        if (tid == 0 && p.err) atomicOr(p.err, kErrSlotRange);
        for (int64_t t = row0 + (tid >> 6); t < row1; t += CT / 64) {
            uint32_t *o = reinterpret_cast<uint32_t *>(p.out + t * p.ld_out + static_cast<int64_t>(h) * VD);
            o[tid & 63] = 0u;
        }
        return;
    }
    if (row1 <= row0) return;
    const bool has_state = slot >= 0;
    const bool writable = has_state && slot != p.null_slot;
    float *tile = has_state ? p.pool + slot * p.slot_stride + static_cast<int64_t>(h) * KD * VD : nullptr;
    const int nch = static_cast<int>((row1 - row0 + C - 1) / C);
    const unsigned char *rec0 = a.rec + (static_cast<size_t>(a.cb[sq]) * H + h) * REC_BYTES;
    const size_t rec_step = static_cast<size_t>(H) * REC_BYTES;
    const int64_t HK = static_cast<int64_t>(H) * KD;

    const uint32_t sbase = tc::smem_addr(smem);
    const uint32_t bar = sbase + CH_BAR;   // kq[0], kq[1], mm[0], mm[1], mma
    if (tid == 0) {
        for (int i = 0; i < 5; i++) tc::mbar_init(bar + 8 * i, 1);
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
        stage_rows<CT>(sbase + CH_VT + (c & 1) * 16384, p.qkv + r0 * p.ld_qkv + 2 * HK + static_cast<int64_t>(h) * VD,
                       p.ld_qkv, nn, tid);
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
#pragma unroll
        for (int u = 0; u < 16; u++) v[u] = has_state ? tile[static_cast<int64_t>(c + u) * VD + j] : 0.f;
        tc::tmem_st16(tlane + TC_S + c, v);
    }
    tc::tmem_st_wait();

    bool ok = true;
    uint32_t phc = 0;
    int nprev = 0;
    int64_t prev0 = row0;
    auto store_o = [&](const float (&ov)[2][16], int64_t cs, int nrows) {
        uint16_t *orow = p.out + cs * p.ld_out + static_cast<int64_t>(h) * VD + j;
#pragma unroll
        for (int q = 0; q < 2; q++)
#pragma unroll
            for (int u = 0; u < 16; u++) {
                const int rr = 32 * sub + 16 * q + u;
                if (rr < nrows) orow[static_cast<int64_t>(rr) * p.ld_out] = f32_to_bf16(ov[q][u]);
            }
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
        float ov[2][16];
        if (c > 0) {   // O^T of the previous chunk, read before P overwrites it
            tc::tmem_ld16(tlane + TC_PQ + 32 * sub, ov[0]);
            tc::tmem_ld16(tlane + TC_PQ + 32 * sub + 16, ov[1]);
        }
        {
            const float *gam = reinterpret_cast<const float *>(smem + CH_KQ + b * CH_KQ_STRIDE + REC_GAM);
#pragma unroll
            for (int cc = 0; cc < 64; cc += 16) {
                float v[16];
                const int cidx = 64 * sub + cc;
                tc::tmem_ld16(tlane + TC_S + cidx, v);
                tc::tmem_ld_wait();
                uint32_t pk8[8];
#pragma unroll
                for (int i = 0; i < 8; i++) pk8[i] = tc::pack_f16x2(v[2 * i], v[2 * i + 1]);
                tc::tmem_st8u(tlane + TC_AS + (cidx >> 1), pk8);
#pragma unroll
                for (int u = 0; u < 16; u += 4) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(gam + cidx + u);
                    v[u] *= g4.x; v[u + 1] *= g4.y; v[u + 2] *= g4.z; v[u + 3] *= g4.w;
                }
                tc::tmem_st16(tlane + TC_S + cidx, v);
            }
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            tc::gemm_ta<128, 128>(tmem + TC_PK, tmem + TC_AS, sbase + CH_KQ + b * CH_KQ_STRIDE, SBO128_F16, false);
            tc::commit(bar + 32);
        }
        if (c > 0) store_o(ov, prev0, nprev);
        // ---- P done: the record's first part is free for chunk c + 2 ----
        cp_async_wait_group<1>();   // this chunk's V tile (the newer group may fly)
        ok &= cta_wait(bar + 32, phc, smem + CH_WAITOK);
        phc ^= 1;
        if (!ok) break;
        if (c + 2 < nch) {
            if (tid == 0) issue_kq(c + 2);
            kq_pending[b] = c + 2;
        }
        // ---- Y^T = (V - K^G S)^T -> fp16 pairs in TMEM ----
        {
            const uint16_t *vt = reinterpret_cast<const uint16_t *>(smem + CH_VT + b * 16384);
#pragma unroll
            for (int q = 0; q < 2; q++) {
                float v[16];
                const int r0 = 32 * sub + 16 * q;
                tc::tmem_ld16(tlane + TC_PK + r0, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; u++) {
                    const int rr = r0 + u;
                    v[u] = bf16_to_f32(vt[(st_off(rr, j >> 3) >> 1) + (j & 7)]) - v[u];
                }
                uint32_t pk8[8];
#pragma unroll
                for (int i = 0; i < 8; i++) pk8[i] = tc::pack_f16x2(v[2 * i], v[2 * i + 1]);
                tc::tmem_st8u(tlane + TC_AY + (r0 >> 1), pk8);
            }
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncthreads();
        // the V tile of this chunk is consumed: stage chunk c + 2's
        if (c + 2 < nch) stage_v(c + 2);
        cp_async_commit();
        bool mm_ok = true;
        if (tid == 0) {
            mm_ok = tc::mbar_wait(bar + 16 + 8 * b, par);
            if (mm_ok) {
                tc::fence_after_sync();
                tc::gemm_ta<192, 64>(tmem + TC_PQ, tmem + TC_AY, sbase + CH_MM + b * REC_B_BYTES, SBO64_F16, true);
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
        float ov[2][16];
        tc::tmem_ld16(tlane + TC_PQ + 32 * sub, ov[0]);
        tc::tmem_ld16(tlane + TC_PQ + 32 * sub + 16, ov[1]);
        tc::tmem_ld_wait();
        store_o(ov, prev0, nprev);
        if (writable) {
#pragma unroll
            for (int cc = 0; cc < 64; cc += 16) {
                float v[16];
                const int cidx = 64 * sub + cc;
                tc::tmem_ld16(tlane + TC_S + cidx, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; u++) tile[static_cast<int64_t>(cidx + u) * VD + j] = v[u];
            }
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

// Workspace of a K = V = 128 prefill: a flag counter (256 bytes), the list of chunks that
// take the exact path (4 bytes per (chunk, head), rounded up to 256), then one record per
// (chunk, head).
static int64_t total_chunks(const int32_t *cu_host, int64_t num_seqs)
{
    int64_t t = 0;
    for (int64_t s = 0; s < num_seqs; s++) t += (static_cast<int64_t>(cu_host[s + 1]) - cu_host[s] + chunk::C - 1) / chunk::C;
    return t;
}

static size_t list_bytes(int64_t chunk_heads) { return (static_cast<size_t>(chunk_heads) * 4 + 255) / 256 * 256; }

size_t chunk_workspace_bytes(const int32_t *cu_host, int64_t num_seqs, int H, int K, int V, int)
{
    if (K != chunk::KD || V != chunk::VD || num_seqs <= 0) return 0;
    const int64_t ch = total_chunks(cu_host, num_seqs) * H;
    if (ch == 0) return 0;
    return 256 + list_bytes(ch) + static_cast<size_t>(ch) * chunk::REC_BYTES;
}

// The prefill chains of entries [entry_base, entry_base + num_seqs): per launch of at most
// kMaxSeqs sequences, the prep pass, the exact pass over the chunks prep listed, and the
// chains (longest sequence first).
static cudaError_t launch_chunk_path(const Params &p, const int32_t *cu, const int32_t *cu_host,
                                     int64_t entry_base, int64_t num_seqs, void *workspace,
                                     cudaStream_t stream)
{
    using namespace chunk;
    static_assert(sizeof(Args) < 32000, "kernel parameter space");
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(PREP_SMEM))) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(exact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(EXACT_SMEM))) != cudaSuccess) return err;
    if ((err = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(CHAIN_SMEM))) != cudaSuccess) return err;
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    const int64_t all_ch = total_chunks(cu_host + entry_base, num_seqs) * p.H;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    uint32_t *counter = reinterpret_cast<uint32_t *>(ws);
    uint32_t *list = reinterpret_cast<uint32_t *>(ws + 256);
    unsigned char *recs = ws + 256 + list_bytes(all_ch);
    int64_t ch_done = 0;   // chunks (not chunk-heads) of the sequences already launched
    std::vector<int32_t> ord;
    for (int64_t s0 = 0; s0 < num_seqs; s0 += kMaxSeqs) {
        const int64_t ns = std::min<int64_t>(kMaxSeqs, num_seqs - s0);
        Args a;
        a.p = p;
        a.cu = cu;
        a.entry_base = entry_base + s0;
        a.num_seqs = static_cast<int32_t>(ns);
        a.num_decodes = 0;
        a.flag_count = counter;
        a.flag_list = list;
        a.rec = recs + static_cast<size_t>(ch_done) * p.H * REC_BYTES;
        const int32_t *cuh = cu_host + entry_base + s0;
        a.cb[0] = 0;
        for (int64_t i = 0; i < ns; i++)
            a.cb[i + 1] = a.cb[i] + static_cast<int32_t>((static_cast<int64_t>(cuh[i + 1]) - cuh[i] + C - 1) / C);
        ord.resize(static_cast<size_t>(ns));
        std::iota(ord.begin(), ord.end(), 0);
        std::stable_sort(ord.begin(), ord.end(), [cuh](int32_t x, int32_t y) {
            return (cuh[x + 1] - cuh[x]) > (cuh[y + 1] - cuh[y]);
        });
        for (int64_t i = 0; i < ns; i++) a.order[i] = ord[static_cast<size_t>(i)];
        const int64_t nch = a.cb[ns];
        if (nch > 0) {
            if ((err = cudaMemsetAsync(counter, 0, sizeof(uint32_t), stream)) != cudaSuccess) return err;
            prep_kernel<<<static_cast<unsigned>(nch * p.H), PT, PREP_SMEM, stream>>>(a);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
            exact_kernel<<<static_cast<unsigned>(std::min<int64_t>(nch * p.H, sms)), PT, EXACT_SMEM, stream>>>(a);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        }
        // every sequence gets a chain CTA: empty ones check their slot and return
        chain_kernel<<<static_cast<unsigned>(ns * p.H), CT, CHAIN_SMEM, stream>>>(a);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        ch_done += nch;
    }
    return cudaSuccess;
}

cudaError_t launch_chunk_prefill(const Params &p, int K, int V, const int32_t *cu,
                                 const int32_t *cu_host, int64_t entry_base, int64_t num_seqs,
                                 int, void *workspace, size_t, cudaStream_t stream)
{
    if (num_seqs <= 0) return cudaSuccess;
    if (K != chunk::KD || V != chunk::VD)  // other head sizes take the token-recurrent kernel
        return launch_recurrent(p, K, V, 2, 1, cu, entry_base, num_seqs, stream);
    return launch_chunk_path(p, cu, cu_host, entry_base, num_seqs, workspace, stream);
}

// Mixed batch: the decodes (entries [0, num_decodes), one row each) take the packed-decode
// kernel, the prefills the chunk path.
cudaError_t launch_mixed(const Params &p, int K, int V, const int32_t *cu, const int32_t *cu_host,
                         int64_t num_decodes, int64_t num_prefills, void *workspace, cudaStream_t stream)
{
    if (num_decodes > 0) {
        cudaError_t e = launch_recurrent(p, K, V, 2, 1, cu, 0, num_decodes, stream);
        if (e != cudaSuccess) return e;
    }
    return launch_chunk_prefill(p, K, V, cu, cu_host, num_decodes, num_prefills, 64, workspace, 0, stream);
}

}  // namespace kda
