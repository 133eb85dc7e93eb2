// extern "C" entry points of libkda (declared in include/kda.h): host-side
// argument checks, then kernel launches on the caller's stream. Nothing here
// allocates device memory or synchronises; the only state kept between calls is the
// mixed batch's side stream and events (one set per device, kda_chunk.cu) and the
// no-allocation prefill's scratch address (kda_noalloc.cu).
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "kda.h"
#include "kda_launch.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int ok()
{
    g_last_error[0] = '\0';
    return KDA_OK;
}

int cuda_status(cudaError_t e, const char *what)
{
    if (e != cudaSuccess)
        return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }

int check_heads(const kda_heads *hd, bool gate_only)
{
    if (!hd) return fail(KDA_ERR_INVALID_ARGUMENT, "heads is NULL");
    if (hd->H < 1) return fail(KDA_ERR_INVALID_ARGUMENT, "H must be >= 1 (got %d)", hd->H);
    if (gate_only) {
        if (hd->K < 1 || hd->K > 1024)
            return fail(KDA_ERR_INVALID_ARGUMENT, "K must be in 1..1024 (got %d)", hd->K);
    } else {
        if (hd->K < 1 || hd->V < 1)
            return fail(KDA_ERR_INVALID_ARGUMENT, "K and V must be >= 1 (got %d, %d)", hd->K, hd->V);
        if (!supported_dim(hd->K) || !supported_dim(hd->V))
            return fail(KDA_ERR_UNSUPPORTED, "K and V must each be 32, 64 or 128 (got K=%d, V=%d)",
                        hd->K, hd->V);
    }
    if (!hd->A_log) return fail(KDA_ERR_INVALID_ARGUMENT, "A_log is NULL");
    if (hd->has_lower_bound && !(std::isfinite(hd->lower_bound) && hd->lower_bound <= 0.f))
        return fail(KDA_ERR_INVALID_ARGUMENT, "lower_bound must be finite and <= 0 (got %g)",
                    static_cast<double>(hd->lower_bound));
    if (!gate_only) {
        if (!std::isfinite(hd->scale))
            return fail(KDA_ERR_INVALID_ARGUMENT, "scale must be finite");
        if (!(hd->l2_eps >= 0.f) || !std::isfinite(hd->l2_eps))
            return fail(KDA_ERR_INVALID_ARGUMENT, "l2_eps must be finite and >= 0");
    }
    return KDA_OK;
}

// Row-tensor checks shared by every compute call.
int check_rows(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g, int64_t ld_g,
               const uint16_t *raw_beta, int64_t ld_beta, const uint16_t *out, int64_t ld_out,
               const kda_heads *hd)
{
    const int64_t H = hd->H, K = hd->K, V = hd->V;
    if (!mixed_qkv || !raw_g || !raw_beta || !out)
        return fail(KDA_ERR_INVALID_ARGUMENT, "mixed_qkv, raw_g, raw_beta and out must be non-NULL");
    if (ld_qkv < 2 * H * K + H * V)
        return fail(KDA_ERR_INVALID_ARGUMENT, "ld_qkv (%lld) < 2*H*K + H*V (%lld)",
                    (long long)ld_qkv, (long long)(2 * H * K + H * V));
    if (ld_g < H * K)
        return fail(KDA_ERR_INVALID_ARGUMENT, "ld_g (%lld) < H*K (%lld)", (long long)ld_g, (long long)(H * K));
    if (ld_beta < H)
        return fail(KDA_ERR_INVALID_ARGUMENT, "ld_beta (%lld) < H (%lld)", (long long)ld_beta, (long long)H);
    if (ld_out < H * V)
        return fail(KDA_ERR_INVALID_ARGUMENT, "ld_out (%lld) < H*V (%lld)", (long long)ld_out, (long long)(H * V));
    if (!aligned(out, 8) || (ld_out % 4) != 0)
        return fail(KDA_ERR_INVALID_ARGUMENT, "out must be 8-byte aligned with ld_out a multiple of 4");
    if (!aligned(mixed_qkv, 2) || !aligned(raw_g, 2) || !aligned(raw_beta, 2))
        return fail(KDA_ERR_INVALID_ARGUMENT, "bf16 inputs must be 2-byte aligned");
    return KDA_OK;
}

int check_state(const kda_state *st, const kda_heads *hd)
{
    if (!st) return fail(KDA_ERR_INVALID_ARGUMENT, "state is NULL");
    if (!st->pool || !st->indices)
        return fail(KDA_ERR_INVALID_ARGUMENT, "state->pool and state->indices must be non-NULL");
    if (st->num_slots < 1)
        return fail(KDA_ERR_INVALID_ARGUMENT, "num_slots must be >= 1 (got %lld)", (long long)st->num_slots);
    const int64_t hkv = static_cast<int64_t>(hd->H) * hd->K * hd->V;
    if (st->slot_stride < hkv)
        return fail(KDA_ERR_INVALID_ARGUMENT, "slot_stride (%lld) < H*K*V (%lld)",
                    (long long)st->slot_stride, (long long)hkv);
    if (st->slot_stride % 4 != 0 || !aligned(st->pool, 16))
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "the pool must be 16-byte aligned and slot_stride a multiple of 4");
    if (st->index_stride < 1)
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "index_stride must be >= 1 (got %lld): state_indices is a 1-D view with a positive stride",
                    (long long)st->index_stride);
    if (!aligned(st->indices, 4))
        return fail(KDA_ERR_INVALID_ARGUMENT, "indices must be 4-byte aligned");
    if (st->null_slot < -1 || st->null_slot >= st->num_slots)
        return fail(KDA_ERR_INVALID_ARGUMENT, "null_slot must be -1 or in [0, num_slots) (got %d)",
                    st->null_slot);
    return KDA_OK;
}

// One launch covers a call: its grid has at most four CTAs per (entry, head) (the 32-column
// V slices) and the grid's x dimension holds at most 2^31 - 1 blocks.
int check_entry_count(int64_t entries, const kda_heads *hd)
{
    const int64_t per_entry = static_cast<int64_t>(hd->H) * 4;
    if (entries > INT32_MAX / per_entry)
        return fail(KDA_ERR_UNSUPPORTED,
                    "%lld entries x %d heads exceed one launch (at most %lld entries at this H): split the call",
                    (long long)entries, hd->H, (long long)(INT32_MAX / per_entry));
    return KDA_OK;
}

kda::Params make_params(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                        int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                        const kda_heads *hd, const kda_state *st, uint16_t *out, int64_t ld_out,
                        uint32_t *err)
{
    kda::Params p{};
    p.qkv = mixed_qkv; p.ld_qkv = ld_qkv;
    p.rg = raw_g; p.ld_g = ld_g;
    p.rb = raw_beta; p.ld_beta = ld_beta;
    p.A_log = hd->A_log; p.dt_bias = hd->dt_bias;
    p.has_lb = hd->has_lower_bound ? 1 : 0; p.lb = hd->lower_bound;
    p.scale = hd->scale; p.eps = hd->l2_eps;
    if (st) {
        p.pool = st->pool; p.num_slots = st->num_slots; p.slot_stride = st->slot_stride;
        p.indices = st->indices; p.index_stride = st->index_stride; p.null_slot = st->null_slot;
    }
    p.out = out; p.ld_out = ld_out;
    p.err = err;
    p.H = hd->H;
    return p;
}

// Fills the fused-tail parameters; validates the optional conv / norm arguments.
int make_tail(const kda_short_conv *cv, const kda_gated_norm *nm, const kda_heads *hd,
              kda::TailParams *tp)
{
    *tp = kda::TailParams{};
    const int64_t C = 2 * static_cast<int64_t>(hd->H) * hd->K + static_cast<int64_t>(hd->H) * hd->V;
    if (cv) {
        if (cv->width < 1 || cv->width > 4)
            return fail(KDA_ERR_INVALID_ARGUMENT, "conv width must be in 1..4 (got %d)", cv->width);
        if (!cv->weight || (cv->width > 1 && !cv->state))
            return fail(KDA_ERR_INVALID_ARGUMENT, "conv weight and conv state must be non-NULL");
        if (cv->width > 1 && cv->slot_stride < (cv->width - 1) * C)
            return fail(KDA_ERR_INVALID_ARGUMENT, "conv slot_stride (%lld) < (W-1)*C (%lld)",
                        (long long)cv->slot_stride, (long long)((cv->width - 1) * C));
        if (!aligned(cv->weight, 8) || !aligned(cv->bias, 8) || !aligned(cv->state, 8) ||
            (cv->width > 1 && cv->slot_stride % 4 != 0))
            return fail(KDA_ERR_INVALID_ARGUMENT,
                        "conv weight, bias and state must be 8-byte aligned, "
                        "and the conv slot_stride a multiple of 4");
        tp->conv_w = cv->weight; tp->conv_b = cv->bias;
        tp->conv_state = cv->state; tp->conv_slot_stride = cv->slot_stride;
        tp->conv_width = cv->width;
    }
    if (nm) {
        if (!nm->gate || !nm->weight)
            return fail(KDA_ERR_INVALID_ARGUMENT, "norm gate and weight must be non-NULL");
        if (nm->ld_gate < static_cast<int64_t>(hd->H) * hd->V || (nm->ld_gate % 2) != 0 ||
            !aligned(nm->gate, 4))
            return fail(KDA_ERR_INVALID_ARGUMENT,
                        "norm gate must be 4-byte aligned with an even ld_gate >= H*V");
        if (!(nm->eps >= 0.f) || !std::isfinite(nm->eps))
            return fail(KDA_ERR_INVALID_ARGUMENT, "norm eps must be finite and >= 0");
        tp->gate = nm->gate; tp->ld_gate = nm->ld_gate;
        tp->norm_w = nm->weight; tp->norm_eps = nm->eps;
    }
    return KDA_OK;
}

int check_cu_host(const int32_t *cu_host, int64_t n)
{
    if (!cu_host) return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens_host is NULL");
    if (cu_host[0] < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens[0] must be >= 0");
    for (int64_t s = 0; s < n; s++)
        if (cu_host[s + 1] < cu_host[s])
            return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must be non-decreasing (at %lld)", (long long)s);
    return KDA_OK;
}

}  // namespace

extern "C" {

const char *kda_last_error(void) { return g_last_error; }

const char *kda_status_string(int status)
{
    switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    default: return "KDA_ERR_UNKNOWN";
    }
}

int kda_gate(const uint16_t *raw_g, int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
             int64_t N, const kda_heads *heads, float *g_out, float *beta_out, void *stream)
{
    int s = check_heads(heads, true);
    if (s) return s;
    if (N < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "N must be >= 0");
    if (!raw_g || !raw_beta || !g_out || !beta_out)
        return fail(KDA_ERR_INVALID_ARGUMENT, "raw_g, raw_beta, g_out and beta_out must be non-NULL");
    if (ld_g < static_cast<int64_t>(heads->H) * heads->K || ld_beta < heads->H)
        return fail(KDA_ERR_INVALID_ARGUMENT, "ld_g must be >= H*K and ld_beta >= H");
    if (N == 0) return ok();
    kda::Params p = make_params(nullptr, 0, raw_g, ld_g, raw_beta, ld_beta, heads, nullptr,
                                nullptr, 0, nullptr);
    return cuda_status(kda::launch_gate(p, heads->K, N, g_out, beta_out,
                                        static_cast<cudaStream_t>(stream)), "kda_gate launch");
}

int kda_packed_decode(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                      int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                      int64_t num_seqs, const kda_heads *heads, const kda_state *state,
                      uint16_t *out, int64_t ld_out, uint32_t *err_flags, void *stream)
{
    int s;
    if ((s = check_heads(heads, false))) return s;
    if ((s = check_rows(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, out, ld_out, heads))) return s;
    if ((s = check_state(state, heads))) return s;
    if (num_seqs < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "num_seqs must be >= 0");
    if ((s = check_entry_count(num_seqs, heads))) return s;
    if (num_seqs == 0) return ok();
    kda::Params p = make_params(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, heads, state,
                                out, ld_out, err_flags);
    return cuda_status(kda::launch_recurrent(p, heads->K, heads->V, 0, 1, nullptr, 0, num_seqs,
                                             static_cast<cudaStream_t>(stream)),
                       "kda_packed_decode launch");
}

int kda_spec_verify(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                    int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                    int64_t num_reqs, int32_t tokens_per_req, const kda_heads *heads,
                    const kda_state *state, uint16_t *out, int64_t ld_out,
                    uint32_t *err_flags, void *stream)
{
    int s;
    if ((s = check_heads(heads, false))) return s;
    if ((s = check_rows(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, out, ld_out, heads))) return s;
    if ((s = check_state(state, heads))) return s;
    if (num_reqs < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "num_reqs must be >= 0");
    if (tokens_per_req < 1 || tokens_per_req > 64)
        return fail(KDA_ERR_INVALID_ARGUMENT, "tokens_per_req must be in 1..64 (got %d)", tokens_per_req);
    if ((s = check_entry_count(num_reqs, heads))) return s;
    if (num_reqs == 0) return ok();
    kda::Params p = make_params(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, heads, state,
                                out, ld_out, err_flags);
    // Rows laid out for 8-byte channel loads take the one-CTA-per-head kernel (the fused
    // kernel with no conv and no norm); others the V-split spec kernel.
    if (tokens_per_req <= 16 && aligned(mixed_qkv, 8) && aligned(raw_g, 8) && ld_qkv % 4 == 0 &&
        ld_g % 4 == 0 && aligned(heads->dt_bias, 16)) {
        const kda::TailParams none{};
        return cuda_status(kda::launch_fused(p, none, heads->K, heads->V, tokens_per_req, num_reqs,
                                             static_cast<cudaStream_t>(stream)),
                           "kda_spec_verify launch");
    }
    return cuda_status(kda::launch_spec(p, heads->K, heads->V, tokens_per_req, num_reqs,
                                        static_cast<cudaStream_t>(stream)),
                       "kda_spec_verify launch");
}

int kda_spec_verify_checkpoints(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                                int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                                int64_t num_reqs, int32_t tokens_per_req,
                                const int32_t *num_accepted, const kda_heads *heads,
                                const kda_state *state, uint16_t *out, int64_t ld_out,
                                uint32_t *err_flags, void *stream)
{
    int s;
    if ((s = check_heads(heads, false))) return s;
    if ((s = check_rows(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, out, ld_out, heads))) return s;
    if ((s = check_state(state, heads))) return s;
    if (num_reqs < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "num_reqs must be >= 0");
    if (tokens_per_req < 1 || tokens_per_req > kda::kSpecCkptMaxT)
        return fail(KDA_ERR_INVALID_ARGUMENT, "tokens_per_req must be in 1..%d (got %d)",
                    kda::kSpecCkptMaxT, tokens_per_req);
    if (state->index_stride < tokens_per_req)
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "index_stride (%lld) must be >= tokens_per_req (%d): one slot per token",
                    static_cast<long long>(state->index_stride), tokens_per_req);
    if (num_accepted && !aligned(num_accepted, 4))
        return fail(KDA_ERR_INVALID_ARGUMENT, "num_accepted must be 4-byte aligned");
    if ((s = check_entry_count(num_reqs, heads))) return s;
    if (num_reqs == 0) return ok();
    kda::Params p = make_params(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, heads, state,
                                out, ld_out, err_flags);
    return cuda_status(kda::launch_spec_checkpoints(p, heads->K, heads->V, tokens_per_req,
                                                    num_reqs, num_accepted,
                                                    static_cast<cudaStream_t>(stream)),
                       "kda_spec_verify_checkpoints launch");
}

static int fused_common(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                        int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                        int64_t num_entries, int32_t T, const kda_heads *heads,
                        const kda_state *state, const kda_short_conv *conv,
                        const kda_gated_norm *norm, uint16_t *out, int64_t ld_out,
                        uint32_t *err_flags, void *stream, const char *name)
{
    int s;
    if ((s = check_heads(heads, false))) return s;
    if ((s = check_rows(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, out, ld_out, heads))) return s;
    if ((s = check_state(state, heads))) return s;
    if (num_entries < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "the entry count must be >= 0");
    if (T < 1 || T > 16)
        return fail(KDA_ERR_INVALID_ARGUMENT, "tokens_per_req must be in 1..16 (got %d)", T);
    if (!aligned(mixed_qkv, 8) || !aligned(raw_g, 8) || ld_qkv % 4 != 0 || ld_g % 4 != 0)
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "mixed_qkv and raw_g must be 8-byte aligned with ld_qkv and ld_g multiples of 4");
    if (!aligned(heads->dt_bias, 16))
        return fail(KDA_ERR_INVALID_ARGUMENT, "dt_bias must be 16-byte aligned");
    kda::TailParams tp;
    if ((s = make_tail(conv, norm, heads, &tp))) return s;
    if ((s = check_entry_count(num_entries, heads))) return s;
    if (num_entries == 0) return ok();
    kda::Params p = make_params(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, heads, state,
                                out, ld_out, err_flags);
    return cuda_status(kda::launch_fused(p, tp, heads->K, heads->V, T, num_entries,
                                         static_cast<cudaStream_t>(stream)), name);
}

int kda_fused_decode(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                     int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta, int64_t num_seqs,
                     const kda_heads *heads, const kda_state *state, const kda_short_conv *conv,
                     const kda_gated_norm *norm, uint16_t *out, int64_t ld_out,
                     uint32_t *err_flags, void *stream)
{
    return fused_common(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, num_seqs, 1, heads,
                        state, conv, norm, out, ld_out, err_flags, stream, "kda_fused_decode launch");
}

int kda_fused_spec_verify(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                          int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                          int64_t num_reqs, int32_t tokens_per_req, const kda_heads *heads,
                          const kda_state *state, const kda_short_conv *conv,
                          const kda_gated_norm *norm, uint16_t *out, int64_t ld_out,
                          uint32_t *err_flags, void *stream)
{
    return fused_common(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, num_reqs,
                        tokens_per_req, heads, state, conv, norm, out, ld_out, err_flags, stream,
                        "kda_fused_spec_verify launch");
}

int kda_selftest_bounded_wait(uint32_t *err_flags, void *stream)
{
    if (!err_flags) return fail(KDA_ERR_INVALID_ARGUMENT, "err_flags is NULL");
    return cuda_status(kda::launch_bounded_wait_selftest(err_flags, static_cast<cudaStream_t>(stream)),
                       "kda_selftest_bounded_wait launch");
}

size_t kda_chunk_prefill_workspace_bytes(const int32_t *cu_seqlens_host, int64_t num_seqs,
                                         const kda_heads *heads, int32_t chunk_size)
{
    if (check_heads(heads, false)) return 0;
    if (num_seqs < 0) { fail(KDA_ERR_INVALID_ARGUMENT, "num_seqs must be >= 0"); return 0; }
    if (num_seqs == 0) return 0;
    if (check_cu_host(cu_seqlens_host, num_seqs)) return 0;
    if (chunk_size != 64) { fail(KDA_ERR_UNSUPPORTED, "chunk_size must be 64"); return 0; }
    return kda::chunk_workspace_bytes(cu_seqlens_host, num_seqs, heads->H, heads->K, heads->V,
                                      chunk_size);
}

static int chunk_common(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                        int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                        const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                        int64_t num_decodes, int64_t num_prefills, int32_t chunk_size,
                        const kda_heads *heads, const kda_state *state, void *workspace,
                        size_t workspace_bytes, uint16_t *out, int64_t ld_out,
                        uint32_t *err_flags, void *stream, const char *name)
{
    int s;
    if ((s = check_heads(heads, false))) return s;
    if ((s = check_rows(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, out, ld_out, heads))) return s;
    if ((s = check_state(state, heads))) return s;
    if (num_decodes < 0 || num_prefills < 0)
        return fail(KDA_ERR_INVALID_ARGUMENT, "sequence counts must be >= 0");
    if (chunk_size != 64) return fail(KDA_ERR_UNSUPPORTED, "chunk_size must be 64 (got %d)", chunk_size);
    if (!aligned(mixed_qkv, 16) || !aligned(raw_g, 16) || !aligned(out, 16) || (ld_qkv % 8) != 0 ||
        (ld_g % 8) != 0 || (ld_out % 8) != 0)
        return fail(KDA_ERR_INVALID_ARGUMENT,
                    "%s: mixed_qkv, raw_g and out must be 16-byte aligned with ld_qkv, ld_g and ld_out "
                    "multiples of 8", name);
    const int64_t n = num_decodes + num_prefills;
    if ((s = check_entry_count(n, heads))) return s;
    if (n == 0) return ok();
    if (!cu_seqlens) return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens is NULL");
    if ((s = check_cu_host(cu_seqlens_host, n))) return s;
    for (int64_t d = 0; d < num_decodes; d++)
        if (cu_seqlens_host[d + 1] - cu_seqlens_host[d] != 1)
            return fail(KDA_ERR_INVALID_ARGUMENT,
                        "decode sequence %lld of the mixed batch has length %d (must be 1)",
                        (long long)d, cu_seqlens_host[d + 1] - cu_seqlens_host[d]);
    const size_t need = kda::chunk_workspace_bytes(cu_seqlens_host + num_decodes, num_prefills,
                                                   heads->H, heads->K, heads->V, chunk_size);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
        return fail(KDA_ERR_WORKSPACE, "%s needs a 256-byte aligned workspace of %zu bytes (got %zu)",
                    name, need, workspace ? workspace_bytes : (size_t)0);
    kda::Params p = make_params(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, heads, state,
                                out, ld_out, err_flags);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(kda::launch_mixed(p, heads->K, heads->V, cu_seqlens, cu_seqlens_host,
                                         num_decodes, num_prefills, workspace, st),
                       "mixed batch launch");
}

int kda_chunk_prefill(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                      int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                      const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                      int64_t num_seqs, int32_t chunk_size, const kda_heads *heads,
                      const kda_state *state, void *workspace, size_t workspace_bytes,
                      uint16_t *out, int64_t ld_out, uint32_t *err_flags, void *stream)
{
    return chunk_common(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, cu_seqlens,
                        cu_seqlens_host, 0, num_seqs, chunk_size, heads, state, workspace,
                        workspace_bytes, out, ld_out, err_flags, stream, "kda_chunk_prefill");
}

int kda_mixed_batch(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                    int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                    const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                    int64_t num_decodes, int64_t num_prefills, const kda_heads *heads,
                    const kda_state *state, void *workspace, size_t workspace_bytes,
                    uint16_t *out, int64_t ld_out, uint32_t *err_flags, void *stream)
{
    return chunk_common(mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, cu_seqlens,
                        cu_seqlens_host, num_decodes, num_prefills, 64, heads, state, workspace,
                        workspace_bytes, out, ld_out, err_flags, stream, "kda_mixed_batch");
}

}  // extern "C"

int kda::set_error(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}
