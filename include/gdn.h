/*
 * gdn.h -- C ABI of libgdn.so, a GB300 (sm_103a) implementation of the
 * GatedDeltaNet (gated delta rule) recurrence used by the linear-attention
 * layers of Qwen hybrid models.
 *
 * Every entry point takes plain pointers and sizes.  Pointers documented as
 * "device" must be CUDA device (or managed) memory of the current device.
 * The caller owns every buffer: the library never allocates, frees or
 * synchronises, and launches its kernels on the stream it is given, in
 * stream order.  It keeps no state between calls and may be called from
 * several host threads at once.
 *
 * Kernels (all but the causal convolution's) are launched as programmatic
 * dependents of the kernel before them on the stream: their thread blocks may
 * be scheduled while that kernel finishes, but each waits for its completion
 * (and the visibility of its writes) before reading anything, so stream order
 * holds as with plain launches.  A caller's own kernel launched right after
 * a library call with programmatic stream serialization must itself wait
 * (griddepcontrol.wait or cudaGridDependencySynchronize) before reading the
 * library's outputs, which is that launch mode's rule; plainly launched
 * kernels are unaffected.
 *
 * Errors come in two kinds.
 *  - Argument errors that the host can see (NULL pointers, bad sizes, BF16,
 *    misalignment) return a non-zero gdn_status before anything is launched.
 *  - Errors that depend on device data (the packing in cu_seqlens, a state
 *    slot out of range, an accepted length out of range) cannot be seen by the
 *    host without a synchronisation.  The kernels skip the affected unit of
 *    work (a sequence or a request) and OR a GDN_DEVERR_* bit into the
 *    optional device word `status`; they never trap.  The caller zeroes that
 *    word and reads it when it chooses.
 *  - Preconditions that cost a launch to check (the requests of one call use
 *    distinct state slots) are checked only by the debug build of the library
 *    (libgdn_debug.so, compiled with GDN_DEBUG_CHECKS): a small kernel ahead
 *    of the call's work sets GDN_DEVERR_DUP_SLOT.  The release build assumes
 *    them.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same type as cudaStream_t); NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL */
    GDN_ERR_DTYPE = 2,       /* unsupported I/O dtype; BF16 is always rejected */
    GDN_ERR_SHAPE = 3,       /* inconsistent or unsupported sizes */
    GDN_ERR_ALIGN = 4,       /* a state pointer is not 16-byte aligned */
    GDN_ERR_WORKSPACE = 5,   /* workspace missing or smaller than gdn_forward_workspace_size */
    GDN_ERR_CUDA = 6,        /* the CUDA runtime reported an error at launch */
    GDN_ERR_UNSUPPORTED = 7, /* a forced plan that these sizes do not support */
    GDN_ERR_ARG = 8          /* an enum field holds an unknown value, or another argument value is
                                invalid for the call (see each entry point) */
} gdn_status;

/* I/O dtypes of q, k, v and output.  Gates and states are always FP32. */
enum { GDN_F32 = 0, GDN_F16 = 1, GDN_BF16 = 2 /* rejected */ };

/* How the `a` and `b` inputs are read. */
enum {
    GDN_GATES_RAW = 0,         /* raw a, b: g = exp(-exp(A_log) softplus(a + dt_bias)), beta = sigmoid(b) */
    GDN_GATES_PRECOMPUTED = 1  /* a = effective decay g in [0, 1], b = beta (activation "none") */
};

/* Which kernel evaluates a sequence. */
enum {
    GDN_PLAN_AUTO = 0,       /* per sequence: up to 32 tokens recurrent (256 when dk or dv
                                is below 128), longer ones chunked (the chunked kernels
                                need 16-byte aligned q, k, v and the workspace; head
                                sizes below 128 run them on zero-padded d = 128 tiles) */
    GDN_PLAN_RECURRENT = 1,  /* every sequence on the recurrent kernels: a one-token span
                                carries the state token by token, a longer span goes
                                four tokens at a time in closed form on the tensor cores
                                (tcgen05 at dk = dv = 128, warp tensor cores at smaller
                                heads), whatever else the batch holds, so a span gets
                                the same bits in any batch (a max_seqlen hint of 1
                                promises one-token spans: only the decode kernel runs) */
    GDN_PLAN_CHUNKED = 2,    /* every sequence on the tensor-core chunked kernels (head
                                sizes 32, 64, 128 in any combination; below 128 the
                                d = 128 operand tiles are zero-padded) */
    GDN_PLAN_CHUNKED_SPLIT = 3 /* GDN_PLAN_CHUNKED, and at dk = dv = 128 every sequence
                                of more than 1984 tokens (31 chunks) whose captured
                                tokens lie in its first half is evaluated as two halves
                                at once: for batches of a few long sequences, whose
                                (sequence, head) chains would leave most SMs idle.
                                Other head sizes run unsplit.
                                See "Sequence-parallel evaluation" below. */
};

/* Bits of the device status word. */
#define GDN_DEVERR_CU_SEQLENS 0x1  /* cu_seqlens not 0 = cu[0] <= ... <= cu[B] = T */
#define GDN_DEVERR_STATE_SLOT 0x2  /* state_slots[b] outside [0, num_state_slots) */
#define GDN_DEVERR_ACCEPT_LEN 0x4  /* accept_len[j] outside [0, capacity] */
#define GDN_DEVERR_REPLAY_SLOT 0x8 /* a replay source or destination slot out of range */
#define GDN_DEVERR_TIMEOUT 0x10    /* a bounded wait inside a kernel gave up (the unit is not written) */
#define GDN_DEVERR_CAPTURE_COUNT 0x20 /* conv: capture_count[b] outside [0, capacity] (nothing captured) */
#define GDN_DEVERR_DUP_SLOT 0x40   /* debug builds only (GDN_DEBUG_CHECKS): two requests of one call
                                      write the same state slot, or a replay writes a slot that
                                      another request of the call reads; the release build does
                                      not check this precondition (results are then undefined) */

/*
 * Arguments of gdn_forward.
 *
 * Source: "[CUDA] Add compact GatedDeltaNet operator" (Description) defines
 * the operator: packed ragged inputs, fused gate normalisation, native gate
 * arithmetic from raw A_log, and three outputs [output, final_state,
 * state_update], where the FP32 state_update capsule packs the decay, the
 * shared key and the delta of each token.  "Add GatedDeltaNet evaluation
 * export for Qwen hybrid models" (What changed, Dependency) fixes packed THD
 * Q/K/V with cumulative sequence lengths, the FP32 V-major state, the
 * precomputed-gate mode, scalar-per-head dt_bias, FP16/FP32 I/O with BF16
 * rejected, and an aliased (in-place) state.
 *
 * Per token t of sequence b and value head h (key head kh = h / (Hv / Hk)):
 *   qn = q / max(|q|, 1e-6), kn = k / max(|k|, 1e-6)
 *   S <- g S;  u = beta (v - S kn);  S <- S + u kn^T;  o = scale S qn
 * with S the dv x dk FP32 state (row i belongs to value channel i).
 *
 * Layouts (T = total_tokens, B = num_seqs, row-major, innermost last):
 *   q, k          [T, Hk, dk] io_dtype; token stride q_stride / k_stride
 *                 elements (0 = Hk*dk), heads contiguous inside a token
 *   v             [T, Hv, dv] io_dtype; token stride v_stride (0 = Hv*dv)
 *   a, b          [T, Hv] FP32, contiguous
 *   A_log, dt_bias [Hv] FP32 (RAW mode only; may be NULL in PRECOMPUTED mode)
 *   cu_seqlens    device [B+1] int32: sequence b owns tokens [cu[b], cu[b+1])
 *   state_slots   device [B] int32, or NULL for slot b = b
 *   initial_state device [num_state_slots, Hv, dv, dk] FP32, or NULL for zeros
 *   final_state   device, same shape; may equal initial_state (in place).
 *                 Only the slots named by the batch are written.  NULL: the
 *                 final states are not written at all -- for a speculative
 *                 verify pass whose accepted prefix is rebuilt later from the
 *                 committed state and the capsules ("Replay compact fixed
 *                 state for hybrid decoding", Summary), this saves the write
 *                 of every touched state.
 *   output        device [T, Hv, dv] io_dtype, contiguous
 *   state_update  device [B, capacity, W] FP32 with W = Hv + Hk*dk + Hv*dv, or
 *                 NULL when capacity = 0.  Row (b, i) describes token i of
 *                 sequence b for i < min(len_b, capacity):
 *                 [g for each value head | kn for each key head | u for each
 *                 value head (dv floats each)].  Rows past the sequence's
 *                 length are not written.
 *   status        device int32 or NULL (see above)
 *   workspace     device scratch of workspace_bytes (may be NULL when
 *                 gdn_forward_workspace_size reports 0)
 * Sequences in one call must use distinct state slots (checked by the debug
 * build: GDN_DEVERR_DUP_SLOT).
 */
typedef struct gdn_forward_args {
    int32_t num_seqs;              /* B >= 0 (at most 65535) */
    int32_t total_tokens;          /* T >= 0 */
    int32_t num_k_heads;           /* Hk >= 1 */
    int32_t num_v_heads;           /* Hv, a multiple of Hk */
    int32_t head_dim_k;            /* dk in {32, 64, 128} */
    int32_t head_dim_v;            /* dv in {32, 64, 128} */
    int32_t num_state_slots;       /* leading extent of the state pool */
    int32_t io_dtype;              /* GDN_F32 or GDN_F16 */
    int32_t gate_mode;             /* GDN_GATES_* */
    int32_t plan;                  /* GDN_PLAN_* */
    float scale;                   /* output scale; 0 means 1/sqrt(dk) */
    int32_t state_update_capacity; /* capsule rows per sequence; 0 = not emitted */
    int32_t max_seqlen;            /* upper bound on the longest sequence, 0 = unknown (T).
                                      A performance hint: under GDN_PLAN_AUTO a bound of
                                      at most 32 keeps every sequence on the recurrent
                                      kernel and skips the chunked launches, and a bound
                                      of 1 (decode) runs the decode kernel alone.  Results
                                      do not depend on it as long as it is a true bound. */
    int64_t q_stride;
    int64_t k_stride;
    int64_t v_stride;
    const void *q;
    const void *k;
    const void *v;
    const float *a;
    const float *b;
    const float *A_log;
    const float *dt_bias;
    const int32_t *cu_seqlens;
    const int32_t *state_slots;
    const float *initial_state;
    float *final_state;
    void *output;
    float *state_update;
    int32_t *status;
    void *workspace;
    size_t workspace_bytes;
} gdn_forward_args;

/*
 * Sequence-parallel evaluation (GDN_PLAN_CHUNKED_SPLIT).
 *
 * The chunked evaluation of the operator ("[CUDA] Add compact GatedDeltaNet
 * operator", Description: the tensor-core chunked-prefill path) passes the
 * state from chunk to chunk, so each (sequence, value head) chain is
 * sequential, and a single long prompt has only Hv chains, fewer than the
 * GPU's SMs.  Per value head, each token maps the state affinely,
 * S -> S g (I - beta kn kn^T) + beta v kn^T, so over the second half of a
 * sequence S_t = S1 A_t + B_t, with S1 the state entering that half.  The
 * split plan runs, at the same time, the first half from the initial state
 * (giving S1), and the second half twice: from a zero state (giving B_t and
 * the outputs scale B_t qn) and from the identity with v removed (giving A_t
 * and scale A_t qn; dk = dv).  Two further kernels add S1 (scale A_t qn) to the
 * second half's outputs and write S1 A + B as the final state.  The results
 * equal those of GDN_PLAN_CHUNKED up to floating-point rounding (the
 * correction is a tensor-core product with fp16 operands and FP32
 * accumulation, and second-half outputs are rounded twice to the I/O type).
 * Capsules: only tokens whose state is known exactly have a delta, so a
 * sequence is split only when its captured tokens (the first
 * state_update_capacity) all lie in the first half, which runs from the true
 * initial state; otherwise it runs whole.  A sequence of more than 1984
 * tokens is split when that holds, so whether it is split depends only on
 * its own length and the capacity, and a packed batch still gives bitwise
 * the results of its sequences run one at a time.
 * Restrictions: the workspace must be the one gdn_forward_workspace_size
 * reports for this plan (there is no single-kernel form; smaller workspaces
 * give GDN_ERR_WORKSPACE and gdn_forward_no_alloc GDN_ERR_UNSUPPORTED).
 */

/*
 * Bytes of device workspace gdn_forward needs for these arguments (sizes,
 * plan, io_dtype and max_seqlen only are read).  Non-zero exactly when a chunked
 * (tensor-core) kernel may run.  The size is that of the two-phase chunked
 * evaluation: a header (work counter, the longest-first work list and
 * per-sequence offsets: 4 (7 + 8B) bytes rounded up to 1 KiB) plus one record
 * per (64-token chunk, key head) of 32 KiB and one per (chunk, value head) of
 * 17,408 bytes, for at most
 * T/64 + B chunks -- about 1.36 MB per 64 tokens at Hk = 16, Hv = 48.
 * GDN_PLAN_CHUNKED_SPLIT adds three FP32 states per value head for each
 * sequence that can be split (at most min(B, T / 1985)) and T/2 + 64 rows of
 * Hv * dv io_dtype elements for the second halves' identity-run outputs.
 *
 * The records hold d = 128 operand tiles at every head size (smaller heads
 * are zero-padded), so the size does not depend on dk and dv.
 *
 * At dk = dv = 128, gdn_forward also accepts a smaller workspace of at least
 * (B + 2) int32 (rounded up to 256 bytes): it then runs the single-kernel
 * chunked evaluation, which keeps only the sequence list and work counter
 * there.  Both give the same results up to floating-point rounding; the
 * two-phase one is faster.  Other head sizes have only the two-phase form:
 * with a smaller workspace the automatic plan runs every sequence on the
 * recurrent kernels and a forced chunked plan returns GDN_ERR_WORKSPACE.  The workspace must be 16-byte aligned and not shared by calls
 * that overlap on the GPU.  Returns GDN_OK and writes *bytes, or an argument
 * error.
 */
gdn_status gdn_forward_workspace_size(const gdn_forward_args *args, size_t *bytes);

/*
 * Runs the gated delta rule over one packed batch (see gdn_forward_args) and
 * writes output, final_state and, when capacity > 0, state_update.
 * Asynchronous on `stream`.
 */
gdn_status gdn_forward(const gdn_forward_args *args, gdn_stream_t stream);

/*
 * gdn_forward on rank-4 (dense) inputs.
 *
 * Source: "[CUDA] Add compact GatedDeltaNet operator" (Description) supports
 * ragged and rank-4 inputs; "Add GatedDeltaNet evaluation export for Qwen
 * hybrid models" (Copilot overview, builder review) describes the dense
 * layout [B, S, ...] next to the packed token-major one.
 *
 * The batch is num_seqs sequences of exactly seq_len tokens each:
 *   q, k [B, S, Hk, dk], v [B, S, Hv, dv], a, b [B, S, Hv], output
 *   [B, S, Hv, dv] -- in memory the same as the packed layouts with
 *   T = B * S tokens, so strides and every other field mean what they mean
 *   for gdn_forward.  args->cu_seqlens must be NULL (GDN_ERR_ARG otherwise);
 *   args->total_tokens must equal num_seqs * seq_len (GDN_ERR_SHAPE).
 * The state is V-major [slots, Hv, dv, dk] as everywhere in this library;
 * callers that keep the dense export's K-major state [.., dk, dv] convert it
 * with gdn_state_transpose before and after the call.  Workspace: as
 * gdn_forward_workspace_size reports for these arguments.  Results are
 * bitwise those of gdn_forward with cu_seqlens = {0, S, 2S, ..., B S}.
 */
gdn_status gdn_forward_dense(const gdn_forward_args *args, int32_t seq_len, gdn_stream_t stream);

/*
 * dst[m] = src[m]^T for num_matrices row-major rows x cols FP32 matrices
 * (device pointers, packed one after another).  Converts recurrent states
 * between the K-major layout of the dense export, [.., dk, dv], and the
 * V-major layout of the packed operator, [.., dv, dk] ("Add GatedDeltaNet
 * evaluation export for Qwen hybrid models", builder review): K-major to
 * V-major is rows = dk, cols = dv; back is rows = dv, cols = dk.  src and dst
 * must not overlap (GDN_ERR_ARG).  Asynchronous on `stream`.
 */
gdn_status gdn_state_transpose(const float *src, float *dst, int64_t num_matrices, int32_t rows, int32_t cols,
                               gdn_stream_t stream);

/*
 * Replays an accepted prefix of capsules into an inactive state bank.
 *
 * Source: "Replay compact fixed state for hybrid decoding" (Summary, Key
 * changes): the engine captures packed per-token updates and replays only an
 * accepted prefix into inactive state banks before publishing them; the
 * capsule content is the decay, shared key and delta of "[CUDA] Add compact
 * GatedDeltaNet operator" (Description).
 *
 * For request j and every value head h:
 *   S = state_banks[src_slots[j], h]
 *   for i < accept_len[j]:  S <- g_i S + u_i kn_i^T   (capsule row (j, i))
 *   state_banks[dst_slots[j], h] = S
 * accept_len[j] = 0 copies the source state into the destination.
 *
 *   state_banks  device [num_slots, Hv, dv, dk] FP32 (V-major), 16-byte aligned
 *   src_slots, dst_slots, accept_len  device [num_requests] int32
 *   state_update device [num_requests, capacity, W] FP32 in the capsule layout
 *                of gdn_forward (W = Hv + Hk*dk + Hv*dv)
 *   status       device int32 or NULL: GDN_DEVERR_REPLAY_SLOT,
 *                GDN_DEVERR_ACCEPT_LEN (the request is skipped)
 * A destination may equal its own source (in place) but must not be any other
 * request's source or destination (the debug build checks this and sets
 * GDN_DEVERR_DUP_SLOT).
 */
gdn_status gdn_replay_prefix(float *state_banks, int32_t num_slots, int32_t num_requests,
                             int32_t num_k_heads, int32_t num_v_heads, int32_t head_dim_k,
                             int32_t head_dim_v, const int32_t *src_slots, const int32_t *dst_slots,
                             const float *state_update, int32_t capacity, const int32_t *accept_len,
                             int32_t *status, gdn_stream_t stream);

/*
 * gdn_forward for callers that cannot allocate device memory.  The onnxruntime
 * pull requests that define the operator have no counterpart to this call.
 *
 * Some hosts own all device memory through their own allocator and give an
 * operator only its declared inputs and outputs (an inference runtime's
 * custom-operator interface, a serving loop with a fixed memory plan), and
 * some paths cannot afford a cudaMalloc, which may synchronise the device.
 * This call behaves like gdn_forward but ignores args->workspace: long
 * sequences run on the single-kernel chunked evaluation, whose workspace (the
 * sequence list and work counter) comes from a fixed 16 KiB array compiled
 * into the library, which every GPU that loads the library keeps until exit.
 *
 *  - Batches of more than GDN_NO_ALLOC_MAX_SEQS sequences that need a
 *    workspace are rejected with GDN_ERR_WORKSPACE before anything runs.
 *  - plan = GDN_PLAN_CHUNKED_SPLIT is rejected with GDN_ERR_UNSUPPORTED: the
 *    split plan's workspace grows with the batch and it has no single-kernel
 *    form.
 *  - Head sizes below 128 have no single-kernel chunked form: the automatic
 *    plan then keeps every sequence on the recurrent kernels, and
 *    GDN_PLAN_CHUNKED returns GDN_ERR_WORKSPACE.
 *  - The first call on each device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 *    The address is kept for the life of the process, so the library must not
 *    be used after a cudaDeviceReset (or any other teardown of the device's
 *    primary context) in the same process.
 *  - All calls share the array (each call rewrites what it uses), so calls
 *    that overlap on the GPU, e.g. on two streams, race and must not be made.
 *  - No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define GDN_NO_ALLOC_MAX_SEQS 4094
gdn_status gdn_forward_no_alloc(const gdn_forward_args *args, gdn_stream_t stream);

/* Activation applied after the causal convolution. */
enum { GDN_ACT_NONE = 0, GDN_ACT_SILU = 1 };

/*
 * Arguments of varlen_causal_conv_with_state.
 *
 * Source: "[CUDA] Add compact GatedDeltaNet operator", embedded commit "Add
 * compact VarlenCausalConv state updates" (Description): packed token-major
 * input [num_tokens, channels], a per-request state of the kernel_size - 1
 * preceding inputs of every channel, three outputs [output, final_state,
 * state_update] where state_update holds only the appended input values,
 * [batch, state_update_capacity, channels], bounded by an optional
 * per-request capture_count; "Add GatedDeltaNet evaluation export for Qwen
 * hybrid models" (Copilot overview): fused depthwise conv1d + SiLU + carried
 * state.
 *
 * For token t of sequence b and channel c, with x_ext the sequence's state
 * (oldest first) followed by its tokens:
 *   y[t, c] = act(bias[c] + sum_{j<K} weight[c, j] * x_ext[t - (K-1) + j, c])
 *
 * Layouts (T = total_tokens, B = num_seqs, C = channels, K = kernel_size):
 *   x             device [T, C] io_dtype; token stride x_stride elements (0 = C)
 *   weight        device [C, K] FP32;  bias device [C] FP32 or NULL
 *   cu_seqlens    device [B+1] int32;  state_slots device [B] int32 or NULL
 *   capture_count device [B] int32 in [0, capacity], or NULL (capture up to
 *                 capacity tokens of every sequence)
 *   initial_state device [num_state_slots, C, K-1] io_dtype (oldest input
 *                 first), or NULL for zeros
 *   final_state   device, same shape; may equal initial_state (in place):
 *                 becomes the last K-1 inputs of (state, tokens)
 *   output        device [T, C] io_dtype
 *   state_update  device [B, capacity, C] io_dtype, or NULL when capacity = 0:
 *                 row (b, i) = input of token i of sequence b, for
 *                 i < min(len_b, capacity, capture_count[b]); other rows untouched
 * C must be a multiple of 8 (fp16) or 4 (fp32); x, output and state_update
 * 16-byte aligned; K in {2, 3, 4}.  Sequences must use distinct slots.
 */
typedef struct gdn_conv_args {
    int32_t num_seqs;
    int32_t total_tokens;
    int32_t channels;
    int32_t kernel_size;
    int32_t num_state_slots;
    int32_t io_dtype;              /* GDN_F32 or GDN_F16 */
    int32_t activation;            /* GDN_ACT_* */
    int32_t state_update_capacity; /* 0 = no capture */
    int32_t max_seqlen;            /* upper bound on the longest sequence, 0 = unknown.  A
                                      performance hint: a bound of 1 to 8 (decode steps,
                                      speculative drafts) runs one launch in which a thread
                                      carries whole sequences.  Results do not depend on
                                      it, bit for bit, even when a sequence exceeds it. */
    int64_t x_stride;
    const void *x;
    const float *weight;
    const float *bias;
    const int32_t *cu_seqlens;
    const int32_t *state_slots;
    const int32_t *capture_count;
    const void *initial_state;
    void *final_state;
    void *output;
    void *state_update;
    int32_t *status;
} gdn_conv_args;

/*
 * Runs the packed causal convolution (see gdn_conv_args); asynchronous on
 * `stream`.  Device-side data errors set GDN_DEVERR_CU_SEQLENS,
 * GDN_DEVERR_STATE_SLOT or GDN_DEVERR_CAPTURE_COUNT and skip the sequence.
 */
gdn_status varlen_causal_conv_with_state(const gdn_conv_args *args, gdn_stream_t stream);

/*
 * Replays an accepted prefix of captured conv inputs into an inactive state
 * bank: for request j, conv_states[dst_slots[j]] = the last K-1 entries of
 * (conv_states[src_slots[j]], state_update[j, 0 .. accept_len[j])).
 * Source: "Replay compact fixed state for hybrid decoding" (Summary, Key
 * changes): compact convolution values replayed into inactive banks.
 *   conv_states  device [num_slots, C, K-1] io_dtype
 *   state_update device [num_requests, capacity, C] io_dtype (the capture of
 *                varlen_causal_conv_with_state)
 *   src_slots, dst_slots, accept_len  device [num_requests] int32
 * accept_len[j] = 0 copies the source state.  A destination may equal its own
 * source but must not be another request's source or destination.
 */
gdn_status causal_conv_replay_prefix(void *conv_states, int32_t num_slots, int32_t num_requests, int32_t channels,
                                     int32_t kernel_size, int32_t io_dtype, const int32_t *src_slots,
                                     const int32_t *dst_slots, const void *state_update, int32_t capacity,
                                     const int32_t *accept_len, int32_t *status, gdn_stream_t stream);

/* A static, human-readable name for a status code. */
const char *gdn_status_string(gdn_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
