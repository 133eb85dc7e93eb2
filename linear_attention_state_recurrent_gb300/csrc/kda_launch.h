// Internal launcher declarations (host side), shared by the entry points.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kda_common.cuh"

namespace kda {

cudaError_t launch_gate(const Params &p, int K, int64_t N, float *g_out, float *beta_out,
                        cudaStream_t stream);

// mode: 0 = one row per entry (row e), 1 = T rows per entry (rows e*T ..), 2 = rows
// [cu[e], cu[e+1]). Entries entry_base .. entry_base + num_entries - 1.
cudaError_t launch_recurrent(const Params &p, int K, int V, int mode, int T, const int32_t *cu,
                             int64_t entry_base, int64_t num_entries, cudaStream_t stream);

// Single-token decode: entries 0 .. num_entries - 1 (their slots), entry e at row
// row_base + e.
cudaError_t launch_decode(const Params &p, int K, int V, int64_t row_base, int64_t num_entries,
                          cudaStream_t stream);

// Spec-verify: T consecutive rows per request.
cudaError_t launch_spec(const Params &p, int K, int V, int T, int64_t num_reqs, cudaStream_t stream);
constexpr int kSpecCkptMaxT = 16;   // longest request the checkpointing verify kernel takes
cudaError_t launch_spec_checkpoints(const Params &p, int K, int V, int T, int64_t num_reqs,
                                    const int32_t *num_accepted, cudaStream_t stream);

// Fused layer tail (conv -> recurrence -> gated norm): T (1..16) consecutive rows per entry.
cudaError_t launch_fused(const Params &p, const TailParams &tp, int K, int V, int T,
                         int64_t num_entries, cudaStream_t stream);

// Chunked prefill over entries entry_base .. entry_base + num_seqs - 1 (rows from cu).
size_t chunk_workspace_bytes(const int32_t *cu_host, int64_t num_seqs, int H, int K, int V,
                             int chunk_size);
cudaError_t launch_chunk_prefill(const Params &p, int K, int V, const int32_t *cu,
                                 const int32_t *cu_host, int64_t entry_base, int64_t num_seqs,
                                 int chunk_size, void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

// Sets the message kda_last_error returns (printf-style) and returns `status`.
int set_error(int status, const char *fmt, ...);

// The bounded-wait self-test (one CTA waits on an mbarrier nothing arrives at).
cudaError_t launch_bounded_wait_selftest(uint32_t *err, cudaStream_t stream);

// Mixed batch: decodes are entries [0, num_decodes) (length 1) and take the packed-decode
// kernel; prefills are the next num_prefills entries and take the chunk path.
cudaError_t launch_mixed(const Params &p, int K, int V, const int32_t *cu, const int32_t *cu_host,
                         int64_t num_decodes, int64_t num_prefills, void *workspace,
                         cudaStream_t stream);

}  // namespace kda
