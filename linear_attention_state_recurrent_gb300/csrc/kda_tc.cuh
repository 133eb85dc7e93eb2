// Blackwell (sm_103a) building blocks written as inline PTX: tcgen05 MMA with
// operands in shared memory and accumulators in tensor memory (TMEM), TMEM
// allocation and loads/stores, mbarriers with bounded waits, and the operand
// layout the MMAs read.
//
// Operand layout: K-major, no swizzle. A tile of R rows x Kd elements is a grid of
// 8-row x 16-byte "core matrices" (8 fp16 or 4 tf32 per core row), each stored as
// 128 contiguous bytes; core (rg, kc) sits at ((rg * (Kd*esz/16)) + kc) * 128 bytes.
// In the shared-memory descriptor the leading byte offset (next core along K) is 128
// and the stride byte offset (next 8-row group) is Kd*esz*8. One MMA consumes 32
// bytes of K per row (K = 16 fp16 or 8 tf32), i.e. two cores: the next K step starts
// 256 bytes further.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (row, k) in a K-major no-swizzle tile with Kd columns of
// `esz`-byte elements.
__host__ __device__ constexpr uint32_t core_offset(int row, int k, int Kd, int esz)
{
    return static_cast<uint32_t>((((row >> 3) * (Kd * esz / 16)) + (k * esz) / 16) * 128 +
                                 (row & 7) * 16 + (k * esz) % 16);
}

// Shared-memory matrix descriptor (no swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    return d;
}

// Instruction descriptor: fp32 accumulate, K-major A and B, dense.
// fmt: 0 = fp16 (kind::f16), 2 = tf32 (kind::tf32).
__host__ __device__ constexpr uint32_t instr_desc(int fmt, int M, int N)
{
    return (1u << 4) | (static_cast<uint32_t>(fmt) << 7) | (static_cast<uint32_t>(fmt) << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// D[M=128, N] (+)= A[128, Kd] * B[N, Kd]^T over Kd, issued as Kd/kstep MMAs.
// a_sbo / b_sbo: stride byte offsets of the two tiles.
template <int FMT, int N, int KD>
__device__ __forceinline__ void gemm(uint32_t d_tmem, uint32_t a_saddr, uint32_t a_sbo,
                                     uint32_t b_saddr, uint32_t b_sbo, bool accumulate)
{
    constexpr int KSTEP = FMT == 0 ? 16 : 8;
    constexpr uint32_t ID = instr_desc(FMT, 128, N);
#pragma unroll
    for (int ks = 0; ks < KD / KSTEP; ks++) {
        const uint64_t da = smem_desc(a_saddr + ks * 256, 128, a_sbo);
        const uint64_t db = smem_desc(b_saddr + ks * 256, 128, b_sbo);
        const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
        if (FMT == 0) mma_f16(d_tmem, da, db, ID, acc);
        else mma_tf32(d_tmem, da, db, ID, acc);
    }
}

// D[M=128, N] (+)= A[128, Kd] * B[N, Kd]^T with A in tensor memory (fp16 packed two per
// 32-bit column: column c holds k = 2c in the low and 2c+1 in the high half; one K step
// of 16 spans 8 columns) and B in shared memory.
template <int N, int KD>
__device__ __forceinline__ void gemm_ta(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_saddr, uint32_t b_sbo,
                                        bool accumulate)
{
    constexpr uint32_t ID = instr_desc(0, 128, N);
#pragma unroll
    for (int ks = 0; ks < KD / 16; ks++) {
        const uint64_t db = smem_desc(b_saddr + ks * 256, 128, b_sbo);
        const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                     " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                     :: "r"(d_tmem), "r"(a_tmem + ks * 8), "l"(db), "r"(ID), "r"(acc));
    }
}

// Two independent accumulators over the two K halves of one product (A in tensor memory,
// fp16 pairs; B in shared memory): D0 = A[:, :Kd/2] B[:, :Kd/2]^T and
// D1 = A[:, Kd/2:] B[:, Kd/2:]^T, their K steps issued alternately so that the two
// accumulation chains overlap in the tensor pipe. D = D0 + D1.
// NH = 1: the first K half only (D1 untouched).
template <int N, int KD, int NH = 2>
__device__ __forceinline__ void gemm_ta_split(uint32_t d0, uint32_t d1, uint32_t a_tmem, uint32_t b_saddr,
                                              uint32_t b_sbo)
{
    constexpr uint32_t ID = instr_desc(0, 128, N);
    constexpr int HS = KD / 32;   // K steps of 16 per half
#pragma unroll
    for (int ks = 0; ks < HS; ks++) {
        const uint32_t acc = ks > 0 ? 1u : 0u;
#pragma unroll
        for (int hh = 0; hh < NH; hh++) {
            const int kk = hh * HS + ks;
            const uint64_t db = smem_desc(b_saddr + kk * 256, 128, b_sbo);
            asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                         " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                         :: "r"(hh ? d1 : d0), "r"(a_tmem + kk * 8), "l"(db), "r"(ID), "r"(acc));
        }
    }
}

// D[M=128, N] (+)= A[128, Kd] * B[N, Kd]^T in tf32 with A in tensor memory (one 32-bit
// column per K element: one K step of 8 spans 8 columns) and B in shared memory.
template <int N, int KD>
__device__ __forceinline__ void gemm_ta_tf32(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_saddr, uint32_t b_sbo,
                                             bool accumulate)
{
    constexpr uint32_t ID = instr_desc(2, 128, N);
#pragma unroll
    for (int ks = 0; ks < KD / 8; ks++) {
        const uint64_t db = smem_desc(b_saddr + ks * 256, 128, b_sbo);
        const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                     " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n"
                     :: "r"(d_tmem), "r"(a_tmem + ks * 8), "l"(db), "r"(ID), "r"(acc));
    }
}

__device__ __forceinline__ void commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(mbar) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Makes generic-proxy shared-memory writes visible to the tensor core's async proxy.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(mbar), "r"(count));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Waits for the mbarrier phase with the given parity; gives up after ~2 s and
// returns false instead of spinning forever.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity)
{
    uint64_t start = 0;
    for (uint32_t it = 0;; it++) {
        uint32_t ok;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                     " selp.u32 %0, 1, 0, p;\n}\n" : "=r"(ok) : "r"(mbar), "r"(parity) : "memory");
        if (ok) return true;
        if (it == 0) start = global_ns();
        else if ((it & 255u) == 0 && global_ns() - start > 2000000000ull) return false;
    }
}

// Arms an mbarrier for one arrival that also expects `bytes` of asynchronous copies.
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(mbar), "r"(bytes) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to
// this CTA's shared memory; completion is counted on `mbar` in bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}

// 2-D tensor copy (TMA) of one box, described by a tensor map in kernel parameter space,
// from global to this CTA's shared memory; completion is counted on `mbar` in bytes. x is
// the inner (element) coordinate, y the outer (row) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t mbar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(mbar) : "memory");
}

// Brings a tensor map (kernel parameter space) into the descriptor cache ahead of its first use.
__device__ __forceinline__ void prefetch_tensormap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

// Prefetch of one tensor-map box into L2.
__device__ __forceinline__ void tma_prefetch_2d(const void *tmap, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 :: "l"(tmap), "r"(x), "r"(y) : "memory");
}

// TMEM allocation by one full warp; the base address is written to *dst (smem).
template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_saddr)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_saddr), "r"(NCOLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(NCOLS) : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-collective; the warp
// reads lanes 32*(warp%4) .. +31).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                    "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                    "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                    "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                    "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                    "r"(__float_as_uint(v[15]))
                 : "memory");
}

// 8 consecutive 32-bit columns of this thread's TMEM lane (warp-collective)
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                    "r"(v[6]), "r"(v[7])
                 : "memory");
}

// 4 consecutive 32-bit columns of this thread's TMEM lane (warp-collective)
__device__ __forceinline__ void tmem_st4u(uint32_t taddr, const uint32_t (&v)[4])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]) : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// fp32 -> tf32 bit pattern, round to nearest (ties away from zero).
__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t u;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(x));
    return u;
}

// Two fp32 -> packed fp16x2 (round to nearest even); `lo` goes to the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t u;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(u) : "f"(hi), "f"(lo));
    return u;
}

}  // namespace tc
}  // namespace kda
