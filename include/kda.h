/*
 * kda.h — C ABI of libkda: the Kimi Delta Attention (KDA) gated delta-rule
 * recurrence on one NVIDIA GB300 (sm_103a).
 *
 * The operation (the "KDA recurrence" of the Kimi-K3 pages; vLLM PR #60683
 * "specialized decode for Kimi-K3 on MI355X", section Purpose, and the packed
 * decode call of vLLM PR #51682, section "key source excerpts"), per token t of a
 * sequence and per head h, with channels c < K and value columns j < V:
 *
 *   x_c   = raw_g[t, h*K + c] + dt_bias[h*K + c]
 *   g_c   = -exp(A_log[h]) * softplus(x_c)                  if !has_lower_bound
 *         =  lower_bound * sigmoid(exp(A_log[h]) * x_c)      if  has_lower_bound
 *   alpha = exp(g)                          (per-channel decay, in (0, 1])
 *   beta  = sigmoid(raw_beta[t, h])
 *   q^    = scale * q / sqrt(|q|^2 + l2_eps),   k^ = k / sqrt(|k|^2 + l2_eps)
 *   S_t   = (I - beta k^ k^T) Diag(alpha) S_{t-1} + beta k^ v^T      (K x V, fp32)
 *   o_t   = S_t^T q^                                                  (V, bf16 out)
 *
 * The pages name the gate's inputs (raw_g, A_log, dt_bias, lower_bound) but print
 * no gate formula; the one above is this library's documented reading.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller. The library
 *    allocates nothing, keeps no state between calls, never synchronises the
 *    stream, and enqueues its kernels on `stream` (a cudaStream_t; NULL = legacy
 *    default stream). kda_packed_decode, kda_spec_verify,
 *    kda_spec_verify_checkpoints, kda_fused_decode and kda_fused_spec_verify can be
 *    captured in a CUDA graph.
 *  - bf16 values are passed as uint16_t bit patterns.
 *  - mixed_qkv: bf16 [N, ld_qkv]; row t = [ q (H*K) | k (H*K) | v (H*V) ], each
 *    part head-major ([H][K] or [H][V]). raw_g: bf16 [N, ld_g], H*K used.
 *    raw_beta: bf16 [N, ld_beta], H used. out: bf16 [N, ld_out], H*V written.
 *  - State pool: fp32, slot s and head h at pool + s*slot_stride + h*K*V, row-major
 *    [K][V] (V contiguous). slot_stride >= H*K*V may exceed it (a slot can carry
 *    more than the KDA state; the vLLM kernel takes it as stride_state_token =
 *    initial_state.stride(0), PR #51682). Updated in place.
 *  - State indices: the slot of entry i is indices[i * index_stride] (int32). The
 *    view may be strided — e.g. column 0 of a [rows, 1 + num_speculative_blocks]
 *    block table — exactly as the vLLM kernel loads
 *    state_indices + i_n * stride_state_indices (PR #51682, implementation
 *    breakdown item 1). index_stride must be >= 1 (a non-positive stride is
 *    rejected: PR #51682's risk section notes that relaxing the check let such
 *    views through unchecked).
 *  - Slot semantics: 0 <= slot < num_slots is read and written back in place;
 *    slot == null_slot (if null_slot >= 0) is read but never written, so padded
 *    requests of a graph replay can share it (PR #60683, "Refusal and steps",
 *    CUDA graphs); slot < 0 starts from a zero state and writes nothing;
 *    slot >= num_slots is skipped: its output rows are written as zeros, nothing
 *    is read or written in the pool, and bit 0 (KDA_ERRFLAG_SLOT_RANGE) of
 *    *err_flags is set with an atomic OR (err_flags may be NULL). The device never
 *    traps. Two entries naming the same writable slot in one call is a caller
 *    error with an unspecified result.
 *  - Sizes: H >= 1, K and V in {32, 64, 128}. The pool must be 16-byte aligned and
 *    slot_stride a multiple of 4. One call is one launch: it covers at most
 *    (2^31 - 1) / (4 H) entries (sequences or requests); a larger batch returns
 *    KDA_ERR_UNSUPPORTED and is split by the caller.
 *  - Return value: KDA_OK, or an error code with a message in kda_last_error().
 *    All argument checks happen on the host before any launch; on error nothing
 *    is enqueued. A zero-sized call (N == 0 / no entries) returns KDA_OK and
 *    enqueues nothing.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_OK 0
#define KDA_ERR_INVALID_ARGUMENT 1 /* a pointer, size, stride or layout is not accepted */
#define KDA_ERR_UNSUPPORTED 2      /* valid request this build does not serve (e.g. K=96) */
#define KDA_ERR_WORKSPACE 3        /* workspace missing, too small or misaligned */
#define KDA_ERR_CUDA 4             /* a CUDA runtime call or launch failed */

#define KDA_ERRFLAG_SLOT_RANGE 1u /* bit 0 of *err_flags: a state index was >= num_slots */
#define KDA_ERRFLAG_TIMEOUT 2u    /* bit 1: a device-side wait gave up after ~2 s (results invalid) */
#define KDA_ERRFLAG_RANGE 4u      /* bit 2: a value the chunked prefill carries in fp16 (a state entry,
                                     V - K^G S or an intra-chunk operand) reached |x| >= 65504; the
                                     affected outputs and states are invalid (kda_chunk_prefill and
                                     kda_mixed_batch with K and V in {64, 128}) */

/* Per-layer head parameters shared by every call. */
typedef struct kda_heads {
    int32_t H, K, V;        /* heads, key dim, value dim */
    const float *A_log;     /* device fp32 [H]: log of the per-head decay rate */
    const float *dt_bias;   /* device fp32 [H*K], per channel; NULL = zeros */
    int32_t has_lower_bound;/* nonzero: bounded gate lower_bound * sigmoid(...) */
    float lower_bound;      /* used when has_lower_bound; must be finite and <= 0 */
    float scale;            /* multiplies q^ (commonly K^-1/2); finite */
    float l2_eps;           /* epsilon inside the q/k L2 norms; >= 0 (1e-6 typical) */
} kda_heads;

/* The state pool and the entry -> slot map of one call. */
typedef struct kda_state {
    float *pool;            /* device fp32 [num_slots, slot_stride], updated in place */
    int64_t num_slots;      /* >= 1 */
    int64_t slot_stride;    /* elements between slots, >= H*K*V, multiple of 4 */
    const int32_t *indices; /* device int32, entry i at indices[i*index_stride] */
    int64_t index_stride;   /* >= 1 */
    int32_t null_slot;      /* slot that is read but never written; -1 = none */
} kda_state;

/*
 * The two steps around the recurrence in the Kimi-K3 decode layer ("spec conv, KDA
 * recurrence, gated RMSNorm", vLLM PR #60683, section Purpose, whole-layer list), fused
 * into kda_fused_decode / kda_fused_spec_verify. The pages name the steps only; the
 * definitions below are this library's readings.
 *
 * Short causal convolution, depthwise over the C = 2*H*K + H*V channels of the q|k|v row
 * (mixed_qkv then holds the convolution's INPUTS), width W in 1..4:
 *   y_t[ch] = sum_{w<W} weight[ch*W + w] * hist[t + w][ch] + bias[ch],   x'_t = y_t * sigmoid(y_t)
 * where hist = [the W-1 stored previous inputs of the slot, oldest first; the call's rows].
 * After the call the slot's conv state holds the last W-1 rows of hist (bit-exact bf16).
 * The conv state shares the KDA state's slot index and slot rules (negative: zero history,
 * not written; null slot: read, not written; out of range: untouched).
 */
typedef struct kda_short_conv {
    const uint16_t *weight;   /* device bf16 [C][W]; 8-byte aligned */
    const uint16_t *bias;     /* device bf16 [C], or NULL; 8-byte aligned */
    uint16_t *state;          /* device bf16 conv-state pool of num_slots slots (the kda_state's):
                                 slot s at state + s*slot_stride, [W-1][C] row-major (oldest
                                 input first), updated in place; may be NULL when W == 1 */
    int64_t slot_stride;      /* bf16 elements between slots, >= (W-1)*C, multiple of 4 */
    int32_t width;            /* W, 1..4 */
} kda_short_conv;

/*
 * Gated RMSNorm of each (token, head)'s V outputs:
 *   o'_j = o_j / sqrt(mean_j o_j^2 + eps) * weight[j] * sigmoid(gate[t*ld_gate + h*V + j])
 */
typedef struct kda_gated_norm {
    const uint16_t *gate;     /* device bf16 [N, ld_gate], H*V used; 4-byte aligned */
    int64_t ld_gate;          /* >= H*V, even */
    const float *weight;      /* device fp32 [V] */
    float eps;                /* >= 0 */
} kda_gated_norm;

/* Message of the last failing call on this host thread ("" if none). */
const char *kda_last_error(void);

/* Name of a status code. */
const char *kda_status_string(int status);

/*
 * kda_gate — the fused decay gate and beta on their own: per token t < N, head h,
 * channel c, g_out[t*H*K + h*K + c] = g_c (fp32 log-decay, <= 0) and
 * beta_out[t*H + h] = sigmoid(raw_beta[t, h]). The gate inputs are the ones the
 * vLLM call passes (raw_g, raw_beta, A_log, dt_bias, lower_bound; PR #51682 test
 * call); "chunk_kda_with_fused_gate" (PR #50649, Purpose) fuses this step into the
 * chunk kernel, as every other call here does. K may be any value in 1..1024 here.
 */
int kda_gate(const uint16_t *raw_g, int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
             int64_t N, const kda_heads *heads, float *g_out, float *beta_out, void *stream);

/*
 * kda_packed_decode — one decode token per sequence (fused_recurrent_kda_packed_decode,
 * PR #51682, key source excerpts). Sequence n < num_seqs is row n of mixed_qkv /
 * raw_g / raw_beta / out; its state slot is indices[n*index_stride]. The slot's
 * state is updated in place and o is written to out row n.
 */
int kda_packed_decode(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                      int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                      int64_t num_seqs, const kda_heads *heads, const kda_state *state,
                      uint16_t *out, int64_t ld_out, uint32_t *err_flags, void *stream);

/*
 * kda_spec_verify — a pure spec-verify step (PR #60683, "Refusal and steps": whole
 * uniform requests, width a multiple of k+1, at most 8 rows each in the pages'
 * deployment). Request r < num_reqs owns rows [r*T, (r+1)*T), T = tokens_per_req
 * in 1..64, and slot indices[r*index_stride]; its state advances token by token
 * and is written back once after the last token. Outputs for every row.
 */
int kda_spec_verify(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                    int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                    int64_t num_reqs, int32_t tokens_per_req, const kda_heads *heads,
                    const kda_state *state, uint16_t *out, int64_t ld_out,
                    uint32_t *err_flags, void *stream);

/*
 * kda_spec_verify_checkpoints — a spec-verify step that keeps the state after every
 * draft token, so the next step can resume from whichever prefix the target model
 * accepted. Request r owns rows [r*T, (r+1)*T) (T = tokens_per_req in 1..16) and a
 * block-table row of at least T slots, indices[r*index_stride + c] for c < T
 * (index_stride >= T): the mamba-group block table of 1 + num_speculative_blocks
 * columns (vLLM PR #51682, PR body; T = k + 1). With a_r = num_accepted[r] (device
 * int32 [num_reqs], the previous step's accepted-token count; NULL = 1 for every
 * request; padded requests carry 1, PR #60683 "Refusal and steps", CUDA graphs):
 *   - the initial state is read from column a_r - 1;
 *   - the state after token t is written to column t, for every t < T;
 *   - outputs are written for every row, as kda_spec_verify.
 * Per column: a negative slot reads a zero state (read column) / is not written, the
 * null slot is read but never written, a slot >= num_slots is not written and sets
 * KDA_ERRFLAG_SLOT_RANGE. If the read column is out of range or a_r is outside
 * [1, T], the request's outputs are zero, nothing of it is read or written, and
 * KDA_ERRFLAG_SLOT_RANGE is set. Distinct requests must not share a written slot.
 * indices must hold at least (num_reqs - 1)*index_stride + T entries. Writes T x
 * the state bytes of kda_spec_verify. Can be captured in a CUDA graph.
 */
int kda_spec_verify_checkpoints(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                                int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                                int64_t num_reqs, int32_t tokens_per_req,
                                const int32_t *num_accepted, const kda_heads *heads,
                                const kda_state *state, uint16_t *out, int64_t ld_out,
                                uint32_t *err_flags, void *stream);

/*
 * kda_fused_decode — kda_packed_decode with the short convolution in front and the gated
 * RMSNorm behind, in one kernel (one CTA per (sequence, head)). conv == NULL skips the
 * convolution (mixed_qkv are then the recurrence's inputs, as in kda_packed_decode);
 * norm == NULL skips the norm. Outputs, KDA state and error word follow kda_packed_decode.
 * Layout requirements beyond kda_packed_decode's (the kernel moves 4 channels per load):
 * mixed_qkv and raw_g 8-byte aligned with ld_qkv and ld_g multiples of 4, dt_bias 16-byte
 * aligned, conv weight, bias and state 8-byte aligned with a conv slot_stride multiple of 4.
 * Can be captured in a CUDA graph.
 */
int kda_fused_decode(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                     int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta, int64_t num_seqs,
                     const kda_heads *heads, const kda_state *state, const kda_short_conv *conv,
                     const kda_gated_norm *norm, uint16_t *out, int64_t ld_out,
                     uint32_t *err_flags, void *stream);

/*
 * kda_fused_spec_verify — kda_spec_verify (T = tokens_per_req in 1..16 rows per request,
 * state read once and written once) with the convolution over the request's T rows in
 * front (its conv state advances by T inputs) and the gated RMSNorm behind. NULL conv /
 * norm skip those steps. Can be captured in a CUDA graph.
 */
int kda_fused_spec_verify(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                          int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                          int64_t num_reqs, int32_t tokens_per_req, const kda_heads *heads,
                          const kda_state *state, const kda_short_conv *conv,
                          const kda_gated_norm *norm, uint16_t *out, int64_t ld_out,
                          uint32_t *err_flags, void *stream);

/*
 * kda_selftest_bounded_wait — exercises the error path of the bounded waits that the
 * tensor-core kernels use on their mbarriers, without a fault: one CTA waits on an
 * mbarrier that nothing arrives at, gives up after ~2 s, sets KDA_ERRFLAG_TIMEOUT in
 * *err_flags (device uint32, required) and returns. The CUDA context stays usable; the
 * call is asynchronous like every other.
 */
int kda_selftest_bounded_wait(uint32_t *err_flags, void *stream);

/*
 * kda_chunk_prefill_workspace_bytes — device workspace kda_chunk_prefill needs for
 * these sequence lengths (cu_seqlens_host: host int32 [num_seqs+1]). Returns 0 on
 * invalid arguments (and sets kda_last_error) or when no workspace is needed.
 */
size_t kda_chunk_prefill_workspace_bytes(const int32_t *cu_seqlens_host, int64_t num_seqs,
                                         const kda_heads *heads, int32_t chunk_size);

/*
 * kda_chunk_prefill — chunked varlen prefill (chunk_kda_with_fused_gate with its
 * WY-form recompute_w_u and intra-/inter-chunk products, PR #50649 Purpose).
 * Sequence s < num_seqs owns rows [cu_seqlens[s], cu_seqlens[s+1]) and slot
 * indices[s*index_stride]; its state is read from the slot, advanced over every
 * row, and written back once. cu_seqlens (device) and cu_seqlens_host (host) must
 * hold the same non-decreasing, non-negative int32 values; the host copy sizes the
 * launch; mixed_qkv, raw_g, raw_beta and out must hold cu_seqlens[num_seqs] rows.
 * chunk_size must be 64. mixed_qkv, raw_g and out must be 16-byte aligned with ld_qkv,
 * ld_g and ld_out multiples of 8 (the tensor-core path moves them in 16-byte vectors).
 * `workspace` (device, 256-byte aligned, owned by the caller) must hold
 * kda_chunk_prefill_workspace_bytes(...) bytes: with K and V each 64 or 128 (the tensor-core
 * path, which works on 128 x 128 tiles with the channels or columns past 64 held at zero)
 * one 57,856-byte record per (chunk of 64 rows, head), then one flag byte per record
 * (rounded up to 16 bytes). The call's first kernel (the intra-chunk pass over every chunk
 * in parallel) writes the records and flags; the second redoes the records whose flag
 * is set: a channel half that decays by more than 80 nats within 16 rows, computed
 * pairwise in fp32. The third (the per-sequence state chain) reads them. The contents are
 * scratch between calls. It may be NULL when the size is 0 (K or V of 32: the
 * token-recurrent kernel).
 * Calls that share a workspace must not overlap on the device. On the tensor-core path the call is
 * three launches per 1024 sequences.
 * Zero-length sequences are allowed: their slot is left untouched (a slot >= num_slots is
 * still flagged).
 * Precision and range (tensor-core path): the products take fp16 / tf32 operands with
 * fp32 accumulation; the state and V - K^G S enter them in fp16, so state entries and values
 * must stay below 65504 in magnitude. Beyond that the call sets KDA_ERRFLAG_RANGE in
 * *err_flags and its results are invalid (the fp32 pool itself holds any value).
 * Bounded waits: a tensor-core wait that gives up (~2 s) sets KDA_ERRFLAG_TIMEOUT and leaves
 * that sequence's outputs and state unwritten; with err_flags == NULL neither condition is
 * reported, so pass an error word wherever results must be trusted.
 */
int kda_chunk_prefill(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                      int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                      const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                      int64_t num_seqs, int32_t chunk_size, const kda_heads *heads,
                      const kda_state *state, void *workspace, size_t workspace_bytes,
                      uint16_t *out, int64_t ld_out, uint32_t *err_flags, void *stream);

/*
 * kda_mixed_batch — a mixed decode + prefill batch (PR #50649, Purpose: the decodes
 * of a mixed batch must not go through the chunk kernel, which returned NaN for
 * length-1 sequences). Sequences 0..num_decodes-1 must have length 1 and take the
 * recurrent decode path; sequences num_decodes..num_decodes+num_prefills-1 take
 * the chunked prefill path. One cu_seqlens (device + host copies) and one strided
 * index view cover all of them, decodes first. The decodes run kda_packed_decode's kernel
 * (decode d on row cu_seqlens_host[0] + d, every decode being one row); the prefills run kda_chunk_prefill's
 * kernels on `stream`. When both are present and K, V are in {64, 128}, the decodes run on
 * a low-priority stream of the library that starts once the prefill's first kernel is done
 * (so that they take the SMs the prefill chains leave free) and is joined back into
 * `stream` within the call: everything enqueued on `stream` after the call sees all its
 * results. The library creates that stream and two events once per device, on the first
 * such call there (make it before any stream capture), keeps them until exit, and
 * serialises the enqueue of concurrent mixed calls from different host threads.
 * Otherwise the decodes run first on `stream`. Workspace as for kda_chunk_prefill over the
 * prefill sequences:
 * kda_chunk_prefill_workspace_bytes(cu_seqlens_host + num_decodes, num_prefills, ...).
 * The prefills' range limit and error bits are kda_chunk_prefill's.
 */
int kda_mixed_batch(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                    int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                    const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                    int64_t num_decodes, int64_t num_prefills, const kda_heads *heads,
                    const kda_state *state, void *workspace, size_t workspace_bytes,
                    uint16_t *out, int64_t ld_out, uint32_t *err_flags, void *stream);

/*
 * kda_chunk_prefill_no_alloc — kda_chunk_prefill for callers that cannot allocate device
 * memory when they call: a host thread of a framework whose device memory belongs to a
 * caching pool it must not bypass, an engine that fixes its footprint at load time, a
 * plugin handed only its inputs and outputs. (This entry point is a property of this
 * library's interface; the method's pages have no counterpart.)
 * Arguments, results, error bits and precision are kda_chunk_prefill's, without the
 * workspace: the intra-chunk records live in one fixed device array of
 * KDA_NO_ALLOC_SCRATCH_BYTES (64 MiB) inside the library, which every GPU that loads the
 * library's code holds until the process exits. The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).
 * - Size limit: the call needs kda_chunk_prefill_workspace_bytes(...) bytes of scratch, one
 *   57,856-byte record and one flag byte per (chunk of 64 rows, head) with K and V in
 *   {64, 128} (at most 1,159 chunk-heads, e.g. 36 chunks at H = 32). A larger request is rejected, before any CUDA call, with
 *   KDA_ERR_WORKSPACE and a message naming both sizes; split it or use kda_chunk_prefill.
 *   Other head sizes need no scratch.
 * - Set-up: the first call on a device that needs scratch looks up the array's device
 *   address on the current device (cudaGetSymbolAddress; this may load the library's device
 *   code) and keeps it. Make that first call on each device before any stream capture.
 * - Sharing: every call on a device uses the same array, which keeps the last call's
 *   records. Nothing in it has to start at zero (each call writes every record it reads),
 *   but calls whose kernels can overlap on the GPU (other streams, other threads) race on
 *   it: order them on one stream or serialise them.
 */
#define KDA_NO_ALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int kda_chunk_prefill_no_alloc(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                               int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                               const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                               int64_t num_seqs, int32_t chunk_size, const kda_heads *heads,
                               const kda_state *state, uint16_t *out, int64_t ld_out,
                               uint32_t *err_flags, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
