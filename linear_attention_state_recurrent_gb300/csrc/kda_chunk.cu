// Chunked varlen prefill.
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {

size_t chunk_workspace_bytes(const int32_t *, int64_t, int, int, int, int) { return 0; }

cudaError_t launch_chunk_prefill(const Params &p, int K, int V, const int32_t *cu,
                                 const int32_t *, int64_t entry_base, int64_t num_seqs, int,
                                 void *, size_t, cudaStream_t stream)
{
    return launch_recurrent(p, K, V, 2, 1, cu, entry_base, num_seqs, stream);
}

}  // namespace kda
