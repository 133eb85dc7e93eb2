// kda_chunk_prefill_no_alloc: the chunked prefill for callers that cannot allocate device
// memory at call time, with its intra-chunk records in a fixed device array of this
// library instead of a caller-provided workspace.
//
// Who needs it: code that runs where cudaMalloc is not allowed or not wanted, e.g. a host
// thread inside a framework whose memory is owned by a caching pool it may not bypass, an
// engine that fixes its device footprint when it loads and must not grow afterwards, or a
// plugin handed only its inputs and outputs with no allocator. They pass inputs and
// outputs as for kda_chunk_prefill; the scratch comes from `g_prefill_scratch` below.
//
// The array is a file-scope __device__ variable, so every GPU on which this library's code
// is loaded holds KDA_NO_ALLOC_SCRATCH_BYTES of it until the process exits. Host code
// cannot use the array's name as a device address: on a call's first use of a device this
// file asks the runtime for the address (cudaGetSymbolAddress, with that device current)
// and keeps it for later calls on the same device.
#include <atomic>
#include <mutex>

#include "kda.h"
#include "kda_launch.h"

static_assert(KDA_NO_ALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");

// The prefill's intra-chunk records (one per (chunk of 64 rows, head)) and their flags.
// A call's kernels write every record byte and flag before they read it, so nothing in
// the array has to start at zero, and what a previous call left there is never read.
static __device__ __align__(256) unsigned char g_prefill_scratch[KDA_NO_ALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kScratchBytes = KDA_NO_ALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// The device address of g_prefill_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void **addr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_addr[dev].load(std::memory_order_relaxed);
        if (!p) {
            e = cudaGetSymbolAddress(&p, g_prefill_scratch);
            if (e != cudaSuccess) return e;
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *addr = p;
    return cudaSuccess;
}

}  // namespace

extern "C" {

int kda_chunk_prefill_no_alloc(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                               int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                               const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                               int64_t num_seqs, int32_t chunk_size, const kda_heads *heads,
                               const kda_state *state, uint16_t *out, int64_t ld_out,
                               uint32_t *err_flags, void *stream)
{
    // The size check is host-only and comes before any CUDA call. A size of 0 means either
    // that no scratch is needed (no sequences, or head sizes that take the token-recurrent
    // kernel) or invalid arguments, which kda_chunk_prefill then reports.
    size_t need = 0;
    if (num_seqs > 0 && heads && cu_seqlens_host)
        need = kda_chunk_prefill_workspace_bytes(cu_seqlens_host, num_seqs, heads, chunk_size);
    if (need > kScratchBytes)
        return kda::set_error(KDA_ERR_WORKSPACE,
                              "kda_chunk_prefill_no_alloc: these sequences need %zu bytes of scratch, "
                              "beyond the fixed %zu bytes (KDA_NO_ALLOC_SCRATCH_BYTES); split the call "
                              "or use kda_chunk_prefill with a workspace",
                              need, kScratchBytes);
    void *scratch = nullptr;
    if (need > 0) {
        const cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess)
            return kda::set_error(KDA_ERR_CUDA, "kda_chunk_prefill_no_alloc: scratch address: %s",
                                  cudaGetErrorString(e));
    }
    // argument checks, the workspace check and the launches are kda_chunk_prefill's
    return kda_chunk_prefill(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, cu_seqlens,
                             cu_seqlens_host, num_seqs, chunk_size, heads, state, scratch,
                             need > 0 ? kScratchBytes : 0, out, ld_out, err_flags, stream);
}

}  // extern "C"
