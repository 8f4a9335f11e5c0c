// Internal launch interface of libgdn.so (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Everything a forward kernel needs, resolved on the host from gdn_forward_args.
struct ForwardParams {
    int B, T, Hk, Hv, dk, dv, r, num_slots;
    int io_f16;        // 1: q, k, v, output are FP16; 0: FP32
    int gate_raw;      // 1: raw gate inputs; 0: precomputed g, beta
    float scale;
    int cap;           // capsule rows per sequence (0: none)
    long long W;       // capsule row width in floats
    long long q_stride, k_stride, v_stride;  // elements between tokens
    const void *q, *k, *v;
    const float *a, *b, *A_log, *dt_bias;
    const int32_t *cu, *slots;
    const float *init;
    float *final_state;
    void *out;
    float *caps;
    int32_t *status;
    // Sequences with more tokens than this are left to the chunked kernel.
    int max_len;
    // Sequences with fewer tokens than this are left to another kernel of the
    // same call (0: none); see launch_recurrent.
    int min_len;
    // The caller's bound on the longest sequence (gdn_forward_args.max_seqlen, 0: unknown).
    int max_len_hint;
    // Rank-4 [B, S, H, D] inputs: cu is null and sequence b owns tokens
    // [b S, (b + 1) S) with S = dense_S.  0 for packed inputs.
    int dense_S;
};

// Streaming multiprocessors of the current device, looked up once per device
// ordinal (persistent grids are sized from it; a process may drive GPUs with
// different SM counts).
inline int current_device_sms() {
    constexpr int kMaxDevices = 128;
    static int cached[kMaxDevices] = {};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < kMaxDevices && __atomic_load_n(&cached[dev], __ATOMIC_RELAXED) > 0)
        return __atomic_load_n(&cached[dev], __ATOMIC_RELAXED);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    if (dev < kMaxDevices) __atomic_store_n(&cached[dev], n, __ATOMIC_RELAXED);
    return n;
}

// First token of sequence b (b may be B: one past the last sequence).
__host__ __device__ __forceinline__ int seq_start(const int32_t *cu, int dense_S, int b) {
    return cu ? cu[b] : b * dense_S;
}

struct ReplayParams {
    int R, Hk, Hv, dk, dv, r, num_slots, cap;
    long long W;
    float *banks;
    const int32_t *src, *dst, *n;
    const float *caps;
    int32_t *status;
};

// Packed causal convolution (see gdn_conv.cu).
struct ConvParams {
    int B, T, C, K, num_slots, io_f16, silu, cap, tokens_per_cta;
    int skip_state_kernel;  // 1: no sequence straddles token blocks and the state is updated in place
    int max_len_hint;       // the caller's bound on the longest sequence (0: unknown)
    long long x_stride;
    const void *x;
    const float *w, *bias;
    const int32_t *cu, *slots, *capture_count;
    const void *state_in;
    void *state_out, *out, *values;
    int32_t *status;
};

struct ConvReplayParams {
    int R, C, K, num_slots, cap, io_f16;
    void *states;
    const void *values;
    const int32_t *src, *dst, *n;
    int32_t *status;
};

cudaError_t launch_conv(const ConvParams &p, cudaStream_t stream);

#ifdef GDN_DEBUG_CHECKS
// Debug builds: GDN_DEVERR_DUP_SLOT when two of the n requests write the same
// slot, or one writes a slot another reads (`read` may be null; see gdn_debug.cu).
cudaError_t debug_check_distinct_slots(const int32_t *written, const int32_t *read, int n, int num_slots,
                                       int32_t *status, cudaStream_t stream);
#endif
cudaError_t launch_conv_replay(const ConvReplayParams &p, cudaStream_t stream);

// Spans of at most p.max_len tokens: the CUDA-core decode kernel when the
// caller bounds every span to one token (a max_seqlen hint of 1), else at
// dk = dv = 128 the tcgen05 short-span kernel and at other head sizes the
// persistent mixed kernel (one-token spans on the decode kernel's arithmetic
// in both, longer ones four tokens at a time).  Without the hint, a batch with
// as many tokens as sequences may still hold multi-token spans next to empty
// ones: the decode kernel then takes the spans of at most one token and the
// short-span kernel the others, so that no span's bits depend on its batch.
cudaError_t launch_recurrent(const ForwardParams &p, cudaStream_t stream);
// Batches with a multi-token span at dk = dv = 128: the tcgen05 short-span
// kernel (gdn_verify.cu); one-token spans in it keep the decode kernel's bits.
bool verify_kernel_supported(const ForwardParams &p);
cudaError_t launch_verify(const ForwardParams &p, cudaStream_t stream);
// dst[m] = src[m]^T for `num` row-major rows x cols FP32 matrices.
cudaError_t launch_transpose(const float *src, float *dst, long long num, int rows, int cols, cudaStream_t stream);
cudaError_t launch_replay(const ReplayParams &p, cudaStream_t stream);

// Chunked tensor-core path: sequences with more than `min_len` tokens
// (min_len < 0: every sequence).  Needs chunked_workspace_bytes(B) of
// device workspace (the chain list and its work counter).  Single-kernel
// form: dk = dv = 128 only.
bool chunked_supported(int dk, int dv);
size_t chunked_workspace_bytes(int B);
cudaError_t launch_chunked(const ForwardParams &p, int min_len, void *workspace, cudaStream_t stream);

// Two-phase chunked path (a parallel per-chunk kernel, then the sequential
// state-passing kernel): faster, and needs chunked_wy_workspace_bytes of
// workspace for the per-chunk records (about 1.36 MB per 64 tokens at
// Hk = 16, Hv = 48, d = 128).  With `split`, every sequence of more than
// 31 * 64 tokens is evaluated as two segments at once (see
// gdn_chunked_wy.cu), which needs room for three states per split sequence
// and head and for the identity-run outputs (io_bytes per element); only
// dk = dv = 128 is split (other sizes run unsplit under that plan).  Head
// sizes 32, 64 and 128 in any combination (zero-padded operand tiles).
bool chunked_wy_supported(int dk, int dv);
bool chunked_wy_splits(int dk, int dv);
size_t chunked_wy_workspace_bytes(int B, int T, int Hk, int Hv, bool split, int io_bytes);
// Workspace of the single-kernel chunked evaluation for these arguments (0 if
// no chunked kernel can run); argument errors as gdn_forward_workspace_size.
gdn_status single_kernel_workspace_size(const gdn_forward_args *args, size_t *bytes);
cudaError_t launch_chunked_wy(const ForwardParams &p, int min_len, bool split, void *workspace,
                              cudaStream_t stream);

// Tensor map over a packed fp16 [T, row_elems] array with `stride` elements
// between tokens, boxes of box_y tokens x box_x elements, zero fill past T;
// with swizzle128 (box_x = 64) each box lands in shared memory in the
// 128-byte swizzled layout of a K-major MMA operand tile.
bool encode_rows_f16(CUtensorMap *map, const void *base, long long row_elems, long long stride, int T, int box_x,
                     int box_y, bool swizzle128);

// Tensor map over a dense row-major FP32 [rows, row_elems] array (no gaps
// between rows), boxes of box_y rows x box_x elements, zero fill past the
// last row; with swizzle128 (box_x = 32) each box lands in shared memory in
// the 128-byte swizzled layout (16-byte chunk c of row r at c ^ (r % 8)).
bool encode_rows_f32(CUtensorMap *map, const float *base, long long row_elems, long long rows, int box_x, int box_y,
                     bool swizzle128);

// Tensor map over a dense FP32 [rows, d] array whose boxes of box_rows rows
// land in shared memory as d / 32 consecutive tiles of box_rows x 32 floats in
// the 128-byte swizzled layout (one tensor copy instead of d / 32); false if
// the driver does not accept the view.
bool encode_state_tiles(CUtensorMap *map, const float *base, int d, long long rows, int box_rows);

// Tensor map over a packed FP32 [T, row_elems] array with `stride` elements
// between tokens (stride * 4 a multiple of 16), boxes of box_y tokens x box_x
// elements, zero fill past T.
bool encode_rows_f32_strided(CUtensorMap *map, const float *base, long long row_elems, long long stride, int T,
                             int box_x, int box_y);

// Sequences up to this many tokens stay on the recurrent kernel under the
// automatic plan; longer ones go to the chunked kernel.  Head sizes below
// 128 run the chunked kernels on d = 128 tiles zero-padded, while the
// recurrent kernels' cost falls with dk dv, so they keep sequences longer.
constexpr int RECURRENT_MAX_LEN = 32;
constexpr int RECURRENT_MAX_LEN_SMALL_HEADS = 256;
inline int recurrent_max_len(int dk, int dv) {
    return dk == 128 && dv == 128 ? RECURRENT_MAX_LEN : RECURRENT_MAX_LEN_SMALL_HEADS;
}

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// ---------------------------------------------------------------- dependent launches
//
// The kernels of the library (all but the causal convolution's token-block
// kernels, whose one-wave decode step measured slower so) are launched as programmatic
// dependents of the kernel before them on the stream (launch_dependent): a
// kernel's CTAs may become
// resident while that kernel's last CTAs finish, which hides the launch gap
// between consecutive kernels (back-to-back decode steps, the chunked path's
// plan -> prep -> scan, the speculative step's verify -> replay).  Every kernel
// starts with dependent_prologue(): it waits until the previous kernel has
// completed and its memory is visible (the ordering a plain launch gives).
// For a kernel launched without the attribute the wait returns at once.  No
// kernel releases its dependents early (griddepcontrol.launch_dependents):
// the next kernel is scheduled as this one's CTAs exit, which measured
// faster on back-to-back decode steps (67.3 vs 67.8 us) than a release at
// each CTA's start.
__device__ __forceinline__ void dependent_prologue() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

__device__ __forceinline__ void flag_error(int32_t *status, int bit) {
    if (status) atomicOr(status, bit);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// softplus(x) = log(1 + e^x), evaluated without overflow.
__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

// Effective decay and beta from one (token, value head)'s gate inputs: raw
// (a, b, A_log, dt_bias) or precomputed (a = g, b = beta).
__device__ __forceinline__ void gates_from(int raw, float av, float bv, float A_log, float dt_bias, float &g,
                                           float &beta) {
    if (raw) {
        g = expf(-expf(A_log) * softplus_f(av + dt_bias));
        beta = 1.f / (1.f + expf(-bv));
    } else {
        g = av;
        beta = bv;
    }
}

}  // namespace gdn
