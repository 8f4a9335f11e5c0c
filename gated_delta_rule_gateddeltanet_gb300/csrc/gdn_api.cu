// The C ABI of libgdn.so: argument checks, planning and kernel dispatch.
//
// Argument rules follow the validation list of "Add GatedDeltaNet evaluation
// export for Qwen hybrid models" (Dependency: scalar-per-head dt_bias, forced
// plans, supported dtypes, update-rule inputs, state alias) and the dtype
// contract of the same page (What changed: FP16 and FP32 I/O, BF16 rejected,
// FP32 gates and state).  Everything that the host can check is checked
// here, before any launch; data-dependent checks happen in the kernels.
#include <math.h>
#include <stdint.h>

#include "gdn_internal.cuh"

namespace {

bool valid_head_dim(int d) { return d == 32 || d == 64 || d == 128; }

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Plans that put every sequence on a chunked kernel.
bool forced_chunked(const gdn_forward_args *a) {
    return a->plan == GDN_PLAN_CHUNKED || a->plan == GDN_PLAN_CHUNKED_SPLIT;
}

// Whether the split plan splits anything at these head sizes.
bool splits(const gdn_forward_args *a) {
    return a->plan == GDN_PLAN_CHUNKED_SPLIT && gdn::chunked_wy_splits(a->head_dim_k, a->head_dim_v);
}

// Workspace of the two-phase chunked evaluation for these arguments.
size_t two_phase_bytes(const gdn_forward_args *a) {
    return gdn::chunked_wy_workspace_bytes(a->num_seqs, a->total_tokens, a->num_k_heads, a->num_v_heads, splits(a),
                                           a->io_dtype == GDN_F16 ? 2 : 4);
}

// Host-side checks shared by gdn_forward and gdn_forward_workspace_size.
gdn_status check_sizes(const gdn_forward_args *a) {
    if (!a) return GDN_ERR_NULL;
    if (a->io_dtype == GDN_BF16) return GDN_ERR_DTYPE;
    if (a->io_dtype != GDN_F32 && a->io_dtype != GDN_F16) return GDN_ERR_DTYPE;
    if (a->gate_mode != GDN_GATES_RAW && a->gate_mode != GDN_GATES_PRECOMPUTED) return GDN_ERR_ARG;
    if (a->plan != GDN_PLAN_AUTO && a->plan != GDN_PLAN_RECURRENT && a->plan != GDN_PLAN_CHUNKED &&
        a->plan != GDN_PLAN_CHUNKED_SPLIT)
        return GDN_ERR_ARG;
    if (a->num_seqs < 0 || a->num_seqs > 65535 || a->total_tokens < 0) return GDN_ERR_SHAPE;
    if (a->num_k_heads <= 0 || a->num_v_heads <= 0 || a->num_v_heads % a->num_k_heads != 0)
        return GDN_ERR_SHAPE;
    if (!valid_head_dim(a->head_dim_k) || !valid_head_dim(a->head_dim_v)) return GDN_ERR_SHAPE;
    if (a->state_update_capacity < 0 || a->max_seqlen < 0) return GDN_ERR_SHAPE;
    if (a->num_seqs > 0 && a->num_state_slots < 1) return GDN_ERR_SHAPE;
    if (a->num_seqs > 0 && !a->state_slots && a->num_state_slots < a->num_seqs) return GDN_ERR_SHAPE;
    const int64_t qk_min = (int64_t)a->num_k_heads * a->head_dim_k;
    const int64_t v_min = (int64_t)a->num_v_heads * a->head_dim_v;
    if ((a->q_stride != 0 && a->q_stride < qk_min) || (a->k_stride != 0 && a->k_stride < qk_min) ||
        (a->v_stride != 0 && a->v_stride < v_min))
        return GDN_ERR_SHAPE;
    if (!(a->scale >= 0.f) || isinf(a->scale)) return GDN_ERR_SHAPE;
    if (forced_chunked(a) && !gdn::chunked_wy_supported(a->head_dim_k, a->head_dim_v)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// Whether these sizes may use the chunked kernel (and so need workspace).
bool wants_chunked(const gdn_forward_args *a) {
    if (a->num_seqs == 0 || a->plan == GDN_PLAN_RECURRENT) return false;
    if (!gdn::chunked_wy_supported(a->head_dim_k, a->head_dim_v)) return false;
    const int longest = a->max_seqlen > 0 && a->max_seqlen < a->total_tokens ? a->max_seqlen : a->total_tokens;
    return forced_chunked(a) || longest > gdn::recurrent_max_len(a->head_dim_k, a->head_dim_v);
}

// The chunked kernel moves q, k, v rows with bulk copies and writes output
// rows in 16-byte pieces.
bool chunked_aligned(const gdn_forward_args *a, const gdn::ForwardParams &p) {
    const size_t esz = p.io_f16 ? 2 : 4;
    return aligned16(a->q) && aligned16(a->k) && aligned16(a->v) && aligned16(a->output) &&
           (p.q_stride * esz) % 16 == 0 &&
           (p.k_stride * esz) % 16 == 0 && (p.v_stride * esz) % 16 == 0;
}

// Checks a forward call completely (sizes, pointers, alignment) and resolves
// it into kernel parameters.  dense_S >= 0: rank-4 inputs of dense_S tokens
// per sequence (cu_seqlens unused); -1: packed inputs.  Returns GDN_OK with
// *out filled, or the error.
gdn_status resolve_forward(const gdn_forward_args *a, int dense_S, gdn::ForwardParams *out) {
    const gdn_status st = check_sizes(a);
    if (st != GDN_OK) return st;
    if (a->num_seqs == 0) return GDN_OK;
    if (dense_S < 0 && !a->cu_seqlens) return GDN_ERR_NULL;
    if (a->total_tokens > 0 && (!a->q || !a->k || !a->v || !a->a || !a->b || !a->output)) return GDN_ERR_NULL;
    if (a->gate_mode == GDN_GATES_RAW && (!a->A_log || !a->dt_bias)) return GDN_ERR_NULL;
    if (a->state_update_capacity > 0 && !a->state_update) return GDN_ERR_NULL;
    if ((a->final_state && !aligned16(a->final_state)) || (a->initial_state && !aligned16(a->initial_state)))
        return GDN_ERR_ALIGN;

    gdn::ForwardParams p{};
    p.B = a->num_seqs;
    p.T = a->total_tokens;
    p.Hk = a->num_k_heads;
    p.Hv = a->num_v_heads;
    p.dk = a->head_dim_k;
    p.dv = a->head_dim_v;
    p.r = p.Hv / p.Hk;
    p.num_slots = a->num_state_slots;
    p.io_f16 = a->io_dtype == GDN_F16;
    p.gate_raw = a->gate_mode == GDN_GATES_RAW;
    p.scale = a->scale > 0.f ? a->scale : 1.0f / sqrtf((float)p.dk);
    p.cap = a->state_update_capacity;
    p.W = (long long)p.Hv + (long long)p.Hk * p.dk + (long long)p.Hv * p.dv;
    p.q_stride = a->q_stride ? a->q_stride : (long long)p.Hk * p.dk;
    p.k_stride = a->k_stride ? a->k_stride : (long long)p.Hk * p.dk;
    p.v_stride = a->v_stride ? a->v_stride : (long long)p.Hv * p.dv;
    p.q = a->q;
    p.k = a->k;
    p.v = a->v;
    p.a = a->a;
    p.b = a->b;
    p.A_log = a->A_log;
    p.dt_bias = a->dt_bias;
    p.cu = dense_S < 0 ? a->cu_seqlens : nullptr;
    p.dense_S = dense_S < 0 ? 0 : dense_S;
    p.slots = a->state_slots;
    p.init = a->initial_state;
    p.final_state = a->final_state;
    p.out = a->output;
    p.caps = p.cap > 0 ? a->state_update : nullptr;
    p.status = a->status;
    p.max_len = 0x7fffffff;
    p.min_len = 0;
    p.max_len_hint = a->max_seqlen;

    *out = p;
    return GDN_OK;
}

}  // namespace

namespace gdn {
// Workspace of the single-kernel chunked evaluation (the chain list only), or
// 0 when these arguments never reach a chunked kernel.
gdn_status single_kernel_workspace_size(const gdn_forward_args *args, size_t *bytes) {
    if (!bytes) return GDN_ERR_NULL;
    const gdn_status st = check_sizes(args);
    if (st != GDN_OK) return st;
    const bool single = chunked_supported(args->head_dim_k, args->head_dim_v);
    *bytes = wants_chunked(args) && single ? chunked_workspace_bytes(args->num_seqs) : 0;
    return GDN_OK;
}
}  // namespace gdn

namespace {

gdn_status forward_impl(const gdn_forward_args *a, int dense_S, gdn_stream_t stream) {
    gdn::ForwardParams p{};
    const gdn_status st = resolve_forward(a, dense_S, &p);
    if (st != GDN_OK || a->num_seqs == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
#ifdef GDN_DEBUG_CHECKS
    if (p.final_state &&
        gdn::debug_check_distinct_slots(p.slots, nullptr, p.B, p.num_slots, p.status, s) != cudaSuccess)
        return GDN_ERR_CUDA;
#endif
    bool chunked = wants_chunked(a);
    if (chunked && !chunked_aligned(a, p)) {
        if (forced_chunked(a)) return GDN_ERR_ALIGN;
        chunked = false;  // the automatic plan keeps every sequence on the recurrent kernel
    }
    const bool d128 = gdn::chunked_supported(a->head_dim_k, a->head_dim_v);
    if (chunked && !d128 && !forced_chunked(a) &&
        (!a->workspace || (reinterpret_cast<uintptr_t>(a->workspace) & 15u) || a->workspace_bytes < two_phase_bytes(a)))
        chunked = false;  // head sizes 32 / 64 have only the two-phase form: without its workspace
                          // the automatic plan keeps every sequence on the recurrent kernels
    if (chunked) {
        // A workspace of gdn_forward_workspace_size bytes runs the two-phase
        // chunked evaluation; one that only holds the chain list runs the
        // single-kernel one (same results up to rounding, slower; dk = dv = 128).
        // The split plan has no single-kernel form.
        if (!a->workspace || (reinterpret_cast<uintptr_t>(a->workspace) & 15u)) return GDN_ERR_WORKSPACE;
        const bool split = splits(a);
        const bool two_phase = a->workspace_bytes >= two_phase_bytes(a);
        if (!two_phase && (a->plan == GDN_PLAN_CHUNKED_SPLIT || !d128 ||
                           a->workspace_bytes < gdn::chunked_workspace_bytes(a->num_seqs)))
            return GDN_ERR_WORKSPACE;
        const int auto_max = gdn::recurrent_max_len(a->head_dim_k, a->head_dim_v);
        const int min_len = forced_chunked(a) ? -1 : auto_max;
        const cudaError_t e = two_phase ? gdn::launch_chunked_wy(p, min_len, split, a->workspace, s)
                                        : gdn::launch_chunked(p, min_len, a->workspace, s);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        if (forced_chunked(a)) return GDN_OK;
        p.max_len = auto_max;
    }
    if (gdn::launch_recurrent(p, s) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // namespace

extern "C" {

const char *gdn_status_string(gdn_status status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL: return "a required pointer is NULL";
        case GDN_ERR_DTYPE: return "unsupported I/O dtype (FP16 and FP32 only; BF16 is rejected)";
        case GDN_ERR_SHAPE: return "inconsistent or unsupported sizes";
        case GDN_ERR_ALIGN: return "a state pointer is not 16-byte aligned";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_CUDA: return "CUDA launch error";
        case GDN_ERR_UNSUPPORTED: return "the forced plan does not support these sizes";
        case GDN_ERR_ARG: return "invalid argument value (unknown enum, cu_seqlens given to the rank-4 call, or overlapping buffers)";
    }
    return "unknown status";
}

gdn_status gdn_forward_workspace_size(const gdn_forward_args *args, size_t *bytes) {
    if (!bytes) return GDN_ERR_NULL;
    const gdn_status st = check_sizes(args);
    if (st != GDN_OK) return st;
    *bytes = wants_chunked(args) ? two_phase_bytes(args) : 0;
    return GDN_OK;
}

gdn_status gdn_forward(const gdn_forward_args *a, gdn_stream_t stream) { return forward_impl(a, -1, stream); }

gdn_status gdn_forward_dense(const gdn_forward_args *args, int32_t seq_len, gdn_stream_t stream) {
    if (!args) return GDN_ERR_NULL;
    if (args->cu_seqlens) return GDN_ERR_ARG;  // rank-4 inputs carry their lengths in seq_len
    if (seq_len < 0 || (int64_t)args->num_seqs * seq_len != (int64_t)args->total_tokens) return GDN_ERR_SHAPE;
    gdn_forward_args a = *args;
    // every sequence has seq_len tokens: a tighter bound than the caller's hint
    if (a.max_seqlen == 0 || a.max_seqlen > seq_len) a.max_seqlen = seq_len;
    return forward_impl(&a, seq_len, stream);
}

gdn_status gdn_state_transpose(const float *src, float *dst, int64_t num_matrices, int32_t rows, int32_t cols,
                               gdn_stream_t stream) {
    if (num_matrices < 0 || rows < 0 || cols < 0) return GDN_ERR_SHAPE;
    if (num_matrices == 0 || rows == 0 || cols == 0) return GDN_OK;
    if (!src || !dst) return GDN_ERR_NULL;
    const int64_t bytes = num_matrices * (int64_t)rows * cols * 4;
    const char *s0 = reinterpret_cast<const char *>(src), *d0 = reinterpret_cast<const char *>(dst);
    if (s0 < d0 + bytes && d0 < s0 + bytes) return GDN_ERR_ARG;  // source and destination overlap
    if (gdn::launch_transpose(src, dst, num_matrices, rows, cols, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status gdn_replay_prefix(float *state_banks, int32_t num_slots, int32_t num_requests, int32_t num_k_heads,
                             int32_t num_v_heads, int32_t head_dim_k, int32_t head_dim_v,
                             const int32_t *src_slots, const int32_t *dst_slots, const float *state_update,
                             int32_t capacity, const int32_t *accept_len, int32_t *status,
                             gdn_stream_t stream) {
    if (num_requests < 0 || num_requests > 65535 || capacity < 0) return GDN_ERR_SHAPE;
    if (num_k_heads <= 0 || num_v_heads <= 0 || num_v_heads % num_k_heads != 0) return GDN_ERR_SHAPE;
    if (!valid_head_dim(head_dim_k) || !valid_head_dim(head_dim_v)) return GDN_ERR_SHAPE;
    if (num_requests == 0) return GDN_OK;
    if (num_slots < 1) return GDN_ERR_SHAPE;
    if (!state_banks || !src_slots || !dst_slots || !accept_len) return GDN_ERR_NULL;
    if (capacity > 0 && !state_update) return GDN_ERR_NULL;
    if (!aligned16(state_banks)) return GDN_ERR_ALIGN;
    gdn::ReplayParams p{};
    p.R = num_requests;
    p.Hk = num_k_heads;
    p.Hv = num_v_heads;
    p.dk = head_dim_k;
    p.dv = head_dim_v;
    p.r = num_v_heads / num_k_heads;
    p.num_slots = num_slots;
    p.cap = capacity;
    p.W = (long long)p.Hv + (long long)p.Hk * p.dk + (long long)p.Hv * p.dv;
    p.banks = state_banks;
    p.src = src_slots;
    p.dst = dst_slots;
    p.n = accept_len;
    p.caps = state_update;
    p.status = status;
#ifdef GDN_DEBUG_CHECKS
    if (gdn::debug_check_distinct_slots(dst_slots, src_slots, num_requests, num_slots, status,
                                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GDN_ERR_CUDA;
#endif
    if (gdn::launch_replay(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status varlen_causal_conv_with_state(const gdn_conv_args *a, gdn_stream_t stream) {
    if (!a) return GDN_ERR_NULL;
    if (a->io_dtype != GDN_F32 && a->io_dtype != GDN_F16) return GDN_ERR_DTYPE;
    if (a->activation != GDN_ACT_NONE && a->activation != GDN_ACT_SILU) return GDN_ERR_ARG;
    const int vec = a->io_dtype == GDN_F16 ? 8 : 4;
    const size_t esz = a->io_dtype == GDN_F16 ? 2 : 4;
    if (a->num_seqs < 0 || a->num_seqs > 65535 || a->total_tokens < 0 || a->channels <= 0 ||
        a->channels % vec != 0 || a->kernel_size < 2 || a->kernel_size > 4 || a->state_update_capacity < 0)
        return GDN_ERR_SHAPE;
    if ((a->x_stride != 0 && a->x_stride < a->channels) || a->max_seqlen < 0) return GDN_ERR_SHAPE;
    if (a->num_seqs == 0) return GDN_OK;
    if (a->num_state_slots < 1 || (!a->state_slots && a->num_state_slots < a->num_seqs)) return GDN_ERR_SHAPE;
    if (!a->cu_seqlens || !a->weight || !a->final_state) return GDN_ERR_NULL;
    if (a->total_tokens > 0 && (!a->x || !a->output)) return GDN_ERR_NULL;
    if (a->state_update_capacity > 0 && !a->state_update) return GDN_ERR_NULL;
    const int64_t xs = a->x_stride ? a->x_stride : a->channels;
    if (!aligned16(a->x) || !aligned16(a->output) || (a->state_update_capacity > 0 && !aligned16(a->state_update)) ||
        !aligned16(a->final_state) || (a->initial_state && !aligned16(a->initial_state)) ||
        (xs * (int64_t)esz) % 16 != 0)
        return GDN_ERR_ALIGN;
    gdn::ConvParams p{};
    p.B = a->num_seqs;
    p.T = a->total_tokens;
    p.C = a->channels;
    p.K = a->kernel_size;
    p.num_slots = a->num_state_slots;
    p.io_f16 = a->io_dtype == GDN_F16;
    p.silu = a->activation == GDN_ACT_SILU;
    p.cap = a->state_update_capacity;
    p.x_stride = xs;
    p.x = a->x;
    p.w = a->weight;
    p.bias = a->bias;
    p.cu = a->cu_seqlens;
    p.slots = a->state_slots;
    p.capture_count = a->capture_count;
    p.state_in = a->initial_state;
    p.state_out = a->final_state;
    p.out = a->output;
    p.values = p.cap > 0 ? a->state_update : nullptr;
    p.status = a->status;
    // as many tokens per CTA as keep the grid within about one wave of 4 CTAs
    // per SM (at most 64): small batches are latency-bound, so a second
    // partial wave costs a full CTA latency
    const long long cblocks = (a->channels / 4 + 255) / 256;  // the kernel's threads own 4 channels
    long long tpc = ((long long)a->total_tokens * cblocks + 607) / 608;
    p.tokens_per_cta = (int)(tpc < 1 ? 1 : (tpc > 64 ? 64 : tpc));
    // Sequences of at most one token always lie inside one token block, where the
    // conv kernel writes their state itself; empty ones keep an in-place state.
    p.skip_state_kernel = a->max_seqlen == 1 && a->initial_state == a->final_state;
    p.max_len_hint = a->max_seqlen;
#ifdef GDN_DEBUG_CHECKS
    if (gdn::debug_check_distinct_slots(p.slots, nullptr, p.B, p.num_slots, p.status,
                                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GDN_ERR_CUDA;
#endif
    if (gdn::launch_conv(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status causal_conv_replay_prefix(void *conv_states, int32_t num_slots, int32_t num_requests, int32_t channels,
                                     int32_t kernel_size, int32_t io_dtype, const int32_t *src_slots,
                                     const int32_t *dst_slots, const void *state_update, int32_t capacity,
                                     const int32_t *accept_len, int32_t *status, gdn_stream_t stream) {
    if (io_dtype != GDN_F32 && io_dtype != GDN_F16) return GDN_ERR_DTYPE;
    const int vec = io_dtype == GDN_F16 ? 8 : 4;
    if (num_requests < 0 || num_requests > 65535 || capacity < 0 || channels <= 0 || channels % vec != 0 ||
        kernel_size < 2 || kernel_size > 4)
        return GDN_ERR_SHAPE;
    if (num_requests == 0) return GDN_OK;
    if (num_slots < 1) return GDN_ERR_SHAPE;
    if (!conv_states || !src_slots || !dst_slots || !accept_len) return GDN_ERR_NULL;
    if (capacity > 0 && !state_update) return GDN_ERR_NULL;
    if (capacity > 0 && !aligned16(state_update)) return GDN_ERR_ALIGN;
    gdn::ConvReplayParams p{};
    p.R = num_requests;
    p.C = channels;
    p.K = kernel_size;
    p.num_slots = num_slots;
    p.cap = capacity;
    p.io_f16 = io_dtype == GDN_F16;
    p.states = conv_states;
    p.values = state_update;
    p.src = src_slots;
    p.dst = dst_slots;
    p.n = accept_len;
    p.status = status;
#ifdef GDN_DEBUG_CHECKS
    if (gdn::debug_check_distinct_slots(dst_slots, src_slots, num_requests, num_slots, status,
                                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GDN_ERR_CUDA;
#endif
    if (gdn::launch_conv_replay(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // extern "C"
