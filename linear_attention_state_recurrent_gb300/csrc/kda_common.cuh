// Device helpers shared by the KDA kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kda {

// Kernel-side view of the per-call arguments (filled by the host entry points).
struct Params {
    const uint16_t *qkv;  int64_t ld_qkv;
    const uint16_t *rg;   int64_t ld_g;
    const uint16_t *rb;   int64_t ld_beta;
    const float *A_log;   const float *dt_bias;
    int has_lb;           float lb;
    float scale;          float eps;
    float *pool;          int64_t num_slots;   int64_t slot_stride;
    const int32_t *indices; int64_t index_stride; int null_slot;
    uint16_t *out;        int64_t ld_out;
    uint32_t *err;
    int H;
};

// The steps around the recurrence in the fused decode / spec-verify calls. conv_width 0 =
// no convolution; gate == nullptr = no gated RMSNorm.
struct TailParams {
    const uint16_t *conv_w;   const uint16_t *conv_b;
    uint16_t *conv_state;     int64_t conv_slot_stride;  int conv_width;
    const uint16_t *gate;     int64_t ld_gate;
    const float *norm_w;      float norm_eps;
};

constexpr uint32_t kErrSlotRange = 1u;
constexpr uint32_t kErrTimeout = 2u;   // a bounded wait on the tensor cores gave up
constexpr uint32_t kErrRange = 4u;     // a value the chunked path carries in fp16 left its range

__device__ __forceinline__ float bf16_to_f32(uint16_t b)
{
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// fp32 -> bf16 bits, round to nearest even (the hardware conversion, one instruction)
__device__ __forceinline__ uint16_t f32_to_bf16(float f)
{
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// Two fp32 values to packed bf16 (lo in the low half), round to nearest even, one
// hardware conversion.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float softplus_f(float x)
{
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

__device__ __forceinline__ float sigmoid_f(float y)
{
    return 1.f / (1.f + expf(-y));
}

// Per-channel log-decay g <= 0 of the fused gate: -e^{A_log} softplus(x), or
// lower_bound * sigmoid(e^{A_log} x) when a lower bound is set; x = raw_g + dt_bias.
__device__ __forceinline__ float gate_log_decay(float x, float expA, int has_lb, float lb)
{
    return has_lb ? lb * sigmoid_f(expA * x) : -expA * softplus_f(x);
}

// The same gate with the fast hardware exp/log (used inside the chunk kernel, where the
// gate is evaluated for every (row, channel) of every chunk). Absolute error of
// log(1 + e^{-|x|}) stays below ~1e-7, far inside the tolerance of the products that
// consume g.
__device__ __forceinline__ float gate_log_decay_fast(float x, float expA, int has_lb, float lb)
{
    if (has_lb) return lb * __fdividef(1.f, 1.f + __expf(-expA * x));
    return -expA * (fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x))));
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 16-byte asynchronous global -> shared copy (L2 only); `valid` false zero-fills the
// destination without reading the source.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// waits until at most N of this thread's most recent cp.async groups are still pending
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Slot of entry e: indices[e * index_stride] widened to 64 bits.
__device__ __forceinline__ int64_t load_slot(const Params &p, int64_t e)
{
    return static_cast<int64_t>(__ldg(p.indices + e * p.index_stride));
}

}  // namespace kda
