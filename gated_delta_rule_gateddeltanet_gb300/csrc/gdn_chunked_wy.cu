// Two-phase chunked (WY / UT-transform) gated delta rule on the tcgen05 tensor
// cores: a parallel phase over every (64-token chunk, key head) and a
// sequential state-passing phase over every (sequence, value head) chain.
//
// Operator: "[CUDA] Add compact GatedDeltaNet operator" (Description) -- the
// tensor-core chunked prefill path of the GatedDeltaNet operator; same results
// as the token-by-token recurrence, evaluated 64 tokens at a time.
//
// Algebra, per (sequence, value head) chain and chunk of n <= 64 tokens, with
// S0 the dv x dk state entering the chunk, Gamma_r the within-chunk cumulative
// log decay and gamma_r = exp(Gamma_r):
//   A[r,s] = beta_r exp(Gamma_r - Gamma_s) (k_r . k_s)  (s < r);   T = (I + A)^-1
//   PD[r,s] = exp(Gamma_r - Gamma_s) (q_r . k_s)        (s <= r)
//   X = S0 K^T,  O' = S0 Q^T                            (dv x n)
//   R^T[i,s] = beta_s (v_s[i] - gamma_s X[i,s]);   U^T = R^T T^T   (the capsule deltas)
//   o_r = scale (gamma_r O'[:,r] + (U^T PD^T)[:,r])
//   S1 = gamma_last S0 + (U^T diag(exp(Gamma_last - Gamma))) K
// This follows from S_r = gamma_r S0 + sum_{s<=r} (gamma_r/gamma_s) u_s k_s^T
// and u_r = beta_r (v_r - g_r S_{r-1} k_r).  Only differences Gamma_r - Gamma_s
// with r >= s are exponentiated.
//
// Everything in the first two lines depends on the chunk's own inputs only,
// not on the state, so it leaves the sequential critical path:
//
//  wy_prep_kernel (one CTA per (chunk, key head), four CTAs per SM): L2-normal-
//    ises q and k into the [Q;K] fp16 operand tile, runs [Q;K] K^T on the
//    tensor cores (P = QK^T and G = KK^T, shared by the key head's value
//    heads), and for each of its value heads computes the gates, A, P o D and
//    the triangular inverse T.  It writes byte images of the operand tiles,
//    already in the swizzled shared-memory layout the MMAs read, to the
//    caller's workspace (one 32 KiB record per (chunk, key head), one 17 KiB
//    record per (chunk, value head)), plus the capsule's k and g.
//
//  wy_scan_kernel (persistent, one CTA per SM, chains longest-first): keeps the
//    FP32 state in tensor memory and, per chunk, loads the two records with
//    bulk copies (and v with a 2-D TMA copy) one chunk ahead, then runs three
//    dependent tensor-core steps:
//      MMA2  S0 [Q;K]^T     -> O', X                (128 x 128, K = dk)
//      MMA3  R^T T^T        -> U^T                  (128 x 64,  K = n)
//      MMA4  U^T PD^T       -> Y                    (128 x 64,  K = n)
//      MMA5  (U^T diag) K   accumulated onto gamma_last S0   (128 x 128, K = n)
//    with the CUDA-core work between them (fp16 state copy, R^T, U^T and its
//    decayed copy, capsule deltas, outputs) done by all 16 warps.
//
//  Split plan (sequence-parallel, for few long sequences): the scan runs each
//    long sequence as three chains per head (first half; second half from a
//    zero state; second half from the identity), and wy_out_correction_kernel
//    and wy_split_final_kernel combine them (see "Sequence-parallel
//    evaluation" below).
//
// Every MMA is kind::f16 (fp16 operands, FP32 accumulation in tensor memory)
// with the value dimension dv = 128 as M and both operands in the 128-byte
// swizzled layout, K-major except K in MMA5: its B operand is the [Q;K]
// tile's k rows read as an MN-major operand (dk along the 128-byte rows), so
// no transposed copy of K exists.  Numerics are those of the single-kernel chunked
// evaluation (same fp16 operand roundings), except that gamma scales the
// FP32 MMA result O' instead of an fp16 copy of Q.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "chunk_tiles.cuh"
#include "gdn_internal.cuh"
#include "ptx.cuh"

namespace gdn {
namespace {

using namespace ct;

constexpr int CH = 64;   // chunk length
// Operand tiles are sized for dk = dv = DH = 128.  Smaller head sizes (32, 64)
// run on the same tiles zero-padded: features past dk and state rows past dv
// are zero in every operand and in the tensor-memory state, so they add
// nothing to any product, and only the first dk / dv entries are read from
// or written to memory.
constexpr int DH = 128;
constexpr float EPS = 1e-6f;
constexpr float LOG_DECAY_FLOOR = -200.f;  // exp(-200) is 0 in fp32; keeps Gamma well-conditioned
constexpr long long WAIT_LIMIT = 4000000000LL;

// Workspace records (byte images of shared-memory operand tiles).
constexpr int KREC_BYTES = 32768;  // [Q;K] tile: 2 K-blocks (dk 0-63, 64-127) x 128 rows (64 q, 64 k) x 128 B
constexpr int VREC_T = 0;          // T, [64][64] fp16
constexpr int VREC_PD = 8192;      // P o D, [64][64] fp16
constexpr int VREC_F = 16384;      // per-token factors (fp32, 64 each): beta, beta*gamma, gamma, exp(Gamma_last - Gamma)
constexpr int F_BETA = 0, F_BG = CH, F_GAMMA = 2 * CH, F_DECAY = 3 * CH;
constexpr int VREC_BYTES = VREC_F + 4 * CH * 4;
static_assert(VREC_BYTES % 128 == 0, "records stay 128-byte aligned");

long long max_chunks(int B, int T) { return (long long)T / CH + B; }

// ---------------------------------------------------------------- plan

// Sequence-parallel evaluation (split plan).  A sequence of at least
// SPLIT_MIN chunks is cut at chunk c1 = ceil(nc / 2) into two segments whose
// chains run at the same time.  Per value head the state after token t of
// the second segment is affine in the state S1 entering it,
//     S_t = S1 A_t + B_t,
// because each token maps S -> S g (I - beta k k^T) + beta v k^T.  B_t is
// the chain run from a zero state, A_t the chain run from the identity with
// the v term removed (dk = dv), and the outputs inherit the same split:
//     o_t = o_t(zero) + S1 o_t(identity),   final = S1 A_last + B_last.
// So the second segment runs twice, from zero (its outputs go straight to the
// output buffer) and from the identity (outputs to a workspace buffer),
// while the first segment runs from the true initial state; two short
// kernels then add S1 o_t(identity) to the outputs and form the final state.
// Chain kinds in the work list:
constexpr int K_WHOLE = 0, K_FIRST = 1, K_ZERO = 2, K_IDENT = 3;
constexpr int SPLIT_MIN = 32;  // chunks: sequences of more than 31 * 64 tokens are split
constexpr int OC_ROWS = 128;   // tokens per tile of the output correction

// Workspace header (int32 words, B sequences):
//   [0] work counter of the scan, [1] E = work-list entries, [2] NS = split sequences
//   list[3B]    work entries, longest chain first: b * 4 + kind
//   cbase[B+1]  index of each sequence's first chunk in the record arrays
//   sidx[B]     split index of each sequence, or -1      (these four: split plan only)
//   sseq[B]     the sequence of each split index
//   tbase[B+1]  first correction tile of each split sequence (prefix over split indices)
//   obase[B+1]  first row of each split sequence's identity-run outputs
struct Header {
    int32_t *w, *list, *cbase, *sidx, *sseq, *tbase, *obase;
    __host__ __device__ Header(int32_t *ws, int B)
        : w(ws), list(ws + 4), cbase(ws + 4 + 3 * B), sidx(ws + 5 + 4 * B), sseq(ws + 5 + 5 * B),
          tbase(ws + 5 + 6 * B), obase(ws + 6 + 7 * B) {}
};
size_t header_bytes(int B) { return ((size_t)(7 + 8 * (size_t)B) * 4 + 1023) & ~size_t(1023); }
// Split sequences and their identity-run output rows that a workspace must hold.
long long max_split(int B, int T) { return std::min<long long>(B, (long long)T / (CH * (SPLIT_MIN - 1) + 1)); }
long long max_split_rows(int T) { return (long long)T / 2 + CH; }
constexpr size_t STATE_BYTES = (size_t)DH * DH * 4;

// Exclusive prefix over sequences b = 0 .. B-1 of value(b), in sequence
// order: put(b, prefix) for every b; returns the total.  All PLAN_NT threads
// call it; thread t owns the contiguous sequences [t * per, (t + 1) * per).
constexpr int PLAN_BINS = 1024;
constexpr int PLAN_NT = 1024;
template <typename V, typename P>
__device__ long long scan_sequences(int B, V value, P put, long long *wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (B + PLAN_NT - 1) / PLAN_NT;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    long long local = 0;
    for (int b = b0; b < b1; ++b) local += value(b);
    long long incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    long long run = incl - local + (warp > 0 ? wsum[warp - 1] : 0);
    for (int b = b0; b < b1; ++b) {
        put(b, run);
        run += value(b);
    }
    const long long total = wsum[PLAN_NT / 32 - 1];
    __syncthreads();  // every thread has read wsum before the next scan reuses it
    return total;
}

// Builds the header.  The work list is a counting sort of the chains on
// their length in chunks (lengths above 1022 share the first bin and are all
// scheduled first).  Sequences with a bad packing are left out (the recurrent
// kernel reports them); an empty sequence is listed (its final state is its
// initial state).  split = false: no sequence is split.  A sequence is split
// only when the tokens it captures (the first `cap`) all lie in its first
// segment, which runs from the true state and so yields the exact deltas.
__global__ void __launch_bounds__(PLAN_NT) wy_plan_kernel(const int32_t *cu, int dense_S, int B, int T, int min_len,
                                                          bool split, int cap, int32_t *ws, int32_t *status) {
    dependent_prologue();
    __shared__ int hist[PLAN_BINS];
    __shared__ long long wsum[PLAN_NT / 32];
    __shared__ int total;
    const int tid = threadIdx.x;
    const Header hd(ws, B);
    // chunks of sequence b on this path, or -1 when it is not
    auto chunks_of = [&](int b) -> int {
        const int lo = seq_start(cu, dense_S, b), hi = seq_start(cu, dense_S, b + 1);
        if (lo < 0 || hi < lo || hi > T || hi - lo <= min_len) return -1;
        return (hi - lo + CH - 1) / CH;
    };
    auto is_split = [&](int c) { return split && c >= SPLIT_MIN && cap <= CH * ((c + 1) / 2); };
    auto bin = [&](int c) { return PLAN_BINS - 1 - min(c, PLAN_BINS - 1); };
    for (int i = tid; i < PLAN_BINS; i += PLAN_NT) hist[i] = 0;
    __syncthreads();
    // a packing error is flagged here too: under the forced chunked plans no other
    // kernel sees the batch
    if (tid == 0 && cu && (cu[0] != 0 || cu[B] != T)) flag_error(status, GDN_DEVERR_CU_SEQLENS);
    for (int b = tid; b < B; b += PLAN_NT) {
        const int lo = seq_start(cu, dense_S, b), hi = seq_start(cu, dense_S, b + 1);
        if (lo < 0 || hi < lo || hi > T) flag_error(status, GDN_DEVERR_CU_SEQLENS);
        const int c = chunks_of(b);
        if (c < 0) continue;
        if (is_split(c)) {
            atomicAdd(&hist[bin((c + 1) / 2)], 1);
            atomicAdd(&hist[bin(c - (c + 1) / 2)], 2);
        } else {
            atomicAdd(&hist[bin(c)], 1);
        }
    }
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int i = 0; i < PLAN_BINS; ++i) {
            const int c = hist[i];
            hist[i] = run;
            run += c;
        }
        total = run;
    }
    __syncthreads();
    for (int b = tid; b < B; b += PLAN_NT) {
        const int c = chunks_of(b);
        if (c < 0) continue;
        if (is_split(c)) {
            const int c1 = (c + 1) / 2;
            hd.list[atomicAdd(&hist[bin(c1)], 1)] = b * 4 + K_FIRST;
            hd.list[atomicAdd(&hist[bin(c - c1)], 1)] = b * 4 + K_ZERO;
            hd.list[atomicAdd(&hist[bin(c - c1)], 1)] = b * 4 + K_IDENT;
        } else {
            hd.list[atomicAdd(&hist[bin(c)], 1)] = b * 4 + K_WHOLE;
        }
    }
    // per-sequence offsets (sequence order)
    const long long nch = scan_sequences(
        B, [&](int b) -> long long { return max(chunks_of(b), 0); },
        [&](int b, long long run) { hd.cbase[b] = (int32_t)run; }, wsum);
    if (!split) {  // nothing below is read when no sequence is split
        if (tid == 0) {
            hd.cbase[B] = (int32_t)nch;
            hd.w[0] = 0;
            hd.w[1] = total;
            hd.w[2] = 0;
        }
        return;
    }
    const long long ns = scan_sequences(
        B, [&](int b) -> long long { return is_split(chunks_of(b)) ? 1 : 0; },
        [&](int b, long long run) {
            const bool sp = is_split(chunks_of(b));
            hd.sidx[b] = sp ? (int32_t)run : -1;
            if (sp) hd.sseq[run] = b;
        },
        wsum);
    // tokens of each split sequence's second segment (from chunk c1 on)
    auto seg2 = [&](int b) -> long long {
        const int c = chunks_of(b);
        if (!is_split(c)) return 0;
        return (long long)seq_start(cu, dense_S, b + 1) - seq_start(cu, dense_S, b) - (long long)CH * ((c + 1) / 2);
    };
    const long long ntile = scan_sequences(
        B, [&](int b) -> long long { return (seg2(b) + OC_ROWS - 1) / OC_ROWS; },
        [&](int b, long long run) {
            if (hd.sidx[b] >= 0) hd.tbase[hd.sidx[b]] = (int32_t)run;
        },
        wsum);
    const long long nrow = scan_sequences(
        B, [&](int b) -> long long { return seg2(b); },
        [&](int b, long long run) {
            if (hd.sidx[b] >= 0) hd.obase[hd.sidx[b]] = (int32_t)run;
        },
        wsum);
    if (tid == 0) {
        hd.cbase[B] = (int32_t)nch;
        hd.tbase[ns] = (int32_t)ntile;
        hd.obase[ns] = (int32_t)nrow;
        hd.w[0] = 0;
        hd.w[1] = total;
        hd.w[2] = (int32_t)ns;
    }
}

// ---------------------------------------------------------------- triangular inverse

// In-place unit lower-triangular inverse: AT holds a 64 x 64 strictly lower A
// (fp32, row stride AS, zeros on and above the diagonal) and receives
// T = (I + A)^-1 in full.  The four 16 x 16 diagonal blocks come from forward
// substitution (one column per thread); the off-diagonal blocks from the block
// identity [[L11, 0], [L21, L22]]^-1 = [[T11, 0], [-T22 L21 T11, T22]], first
// inside the two 32 x 32 diagonal blocks, then for the lower-left quadrant
// (warp-level TF32 products, FP32 storage).  Each block of A is read (into the product M = L21 T11) before the block of
// T that replaces it is written.  256 threads; ends with a barrier.
// Row strides (floats): AS = 68 makes the warp-level product loads of the A / T
// blocks conflict-free (rows land 4 banks apart); MS = 40 does the same for the
// scratch M read as the right-hand factor.
constexpr int AS = 68, MS = 40;
__device__ void tri_inverse_inplace(float *AT, float *M, int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    float x[16];
    const int blk = tid >> 4, c = tid & 15, o = blk * 16;
    if (tid < 64) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc0 = 0.f, acc1 = 0.f;  // two partial sums shorten the dependency chain
#pragma unroll
            for (int s = 0; s < r; s += 2) {
                acc0 = fmaf(AT[(o + r) * AS + o + s], x[s], acc0);
                if (s + 1 < r) acc1 = fmaf(AT[(o + r) * AS + o + s + 1], x[s + 1], acc1);
            }
            x[r] = (r < c) ? 0.f : (r == c ? 1.f : -(acc0 + acc1));
        }
    }
    __syncthreads();  // every diagonal block of A is read before T overwrites it
    if (tid < 64) {
#pragma unroll
        for (int r = 0; r < 16; ++r) AT[(o + r) * AS + o + c] = x[r];
    }
    __syncthreads();
    // inside the 32 x 32 diagonal blocks (o = 0, 32): M = A21 T11, T21 = -T22 M
    if (warp < 4) {
        const int pr = warp >> 1, n0 = (warp & 1) * 8, ob = 32 * pr;
        warp_tile_16x8<16>(AT + (ob + 16) * AS + ob, AS, AT + ob * AS + ob + n0, AS, M + pr * 16 * MS + n0, MS, 1.f,
                           lane);
    }
    __syncthreads();
    if (warp < 4) {
        const int pr = warp >> 1, n0 = (warp & 1) * 8, ob = 32 * pr;
        warp_tile_16x8<16>(AT + (ob + 16) * AS + ob + 16, AS, M + pr * 16 * MS + n0, MS,
                           AT + (ob + 16) * AS + ob + n0, AS, -1.f, lane);
    }
    __syncthreads();
    // the lower-left 32 x 32 quadrant: M = A21 T11, T21 = -T22 M (one 16 x 8 tile per warp)
    {
        const int m0 = (warp >> 2) * 16, n0 = (warp & 3) * 8;
        warp_tile_16x8<32>(AT + (32 + m0) * AS, AS, AT + n0, AS, M + m0 * MS + n0, MS, 1.f, lane);
    }
    __syncthreads();
    {
        const int m0 = (warp >> 2) * 16, n0 = (warp & 3) * 8;
        warp_tile_16x8<32>(AT + (32 + m0) * AS + 32, AS, M + n0, MS, AT + (32 + m0) * AS + n0, AS, -1.f, lane);
    }
    __syncthreads();
}

// Gates of the 64 tokens [t0, t0 + 64) of value head h (one warp, two tokens
// per lane).  Raw mode: g = exp(-exp(A_log) softplus(a + dt_bias)),
// beta = sigmoid(b); precomputed mode: g = a, beta = b.  Log decays are
// floored at LOG_DECAY_FLOOR; tokens at or past `n` get g = 1, beta = 0 (no
// effect).  Writes the within-chunk cumulative log decay Gamma (in log2
// units, for the exponentials of A and P o D) and beta to
// shared memory, the scan kernel's per-token factors (beta, beta gamma,
// gamma = exp(Gamma), exp(Gamma_last - Gamma)) to the record at `fdst`, and
// the capsule decays.
__device__ __forceinline__ void chunk_gates(const ForwardParams &p, int t0, int n, int h, int b, int bos,
                                            float *Gam, float *Beta, float *fdst, int lane) {
    float lg[2], bt[2], gt[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int s = lane + 32 * u;
        lg[u] = 0.f;
        bt[u] = 0.f;
        gt[u] = 1.f;
        if (s < n) {
            const long long t = (long long)t0 + s;
            const float av = p.a[t * p.Hv + h], bv = p.b[t * p.Hv + h];
            if (p.gate_raw) {
                const float l = -expf(p.A_log[h]) * softplus_f(av + p.dt_bias[h]);
                gt[u] = expf(l);
                lg[u] = fmaxf(l, LOG_DECAY_FLOOR);
                bt[u] = 1.f / (1.f + expf(-bv));
            } else {
                gt[u] = av;
                lg[u] = av > 0.f ? fmaxf(logf(av), LOG_DECAY_FLOOR) : LOG_DECAY_FLOOR;
                bt[u] = bv;
            }
        }
    }
    float c[2] = {lg[0], lg[1]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, c[0], o);
        const float y1 = __shfl_up_sync(0xffffffffu, c[1], o);
        if (lane >= o) {
            c[0] += y0;
            c[1] += y1;
        }
    }
    c[1] += __shfl_sync(0xffffffffu, c[0], 31);
    const float l0 = __shfl_sync(0xffffffffu, c[0], (n - 1) & 31);
    const float l1 = __shfl_sync(0xffffffffu, c[1], (n - 1) & 31);
    const float Gl = n - 1 < 32 ? l0 : l1;  // Gamma of the chunk's last token
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int s = lane + 32 * u;
        const float gm = expf(c[u]);
        Gam[s] = c[u] * LOG2E;  // log2 units: the A and P o D exponentials are bare ex2
        Beta[s] = bt[u];
        fdst[F_BETA + s] = bt[u];
        fdst[F_BG + s] = bt[u] * gm;
        fdst[F_GAMMA + s] = gm;
        fdst[F_DECAY + s] = expf(Gl - c[u]);
        const int tl = t0 + s - bos;
        if (p.caps && s < n && tl < p.cap) p.caps[((long long)b * p.cap + tl) * p.W + h] = gt[u];
    }
}

// N consecutive floats (N a multiple of 4) from 16-byte aligned shared memory.
template <int N>
__device__ __forceinline__ void ld_fn(const float *src, float (&x)[N]) {
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
        const float4 v = reinterpret_cast<const float4 *>(src)[q];
        x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
    }
}

// Eight consecutive elements (k % 8 == 0) of one row of a swizzled fp16 tile: one 16-byte store.
__device__ __forceinline__ void st_h8(uint8_t *base, uint32_t off, const float *x) {
    uint4 v;
    __half2 h0 = __floats2half2_rn(x[0], x[1]), h1 = __floats2half2_rn(x[2], x[3]);
    __half2 h2 = __floats2half2_rn(x[4], x[5]), h3 = __floats2half2_rn(x[6], x[7]);
    v.x = *reinterpret_cast<uint32_t *>(&h0);
    v.y = *reinterpret_cast<uint32_t *>(&h1);
    v.z = *reinterpret_cast<uint32_t *>(&h2);
    v.w = *reinterpret_cast<uint32_t *>(&h3);
    *reinterpret_cast<uint4 *>(base + off) = v;
}

// ---------------------------------------------------------------- phase 1: per (chunk, key head)

constexpr int PT = 256;  // threads of the prep kernel
constexpr int GH = 8;    // value heads whose gates are computed together (one warp each)
// Shared memory of the prep kernel (offsets from a 1024-byte aligned base).
// The first 48 KiB hold the key-head record image ([Q;K] tile, then K^T
// tile); with fp16 I/O the raw q and k rows land there by 2-D TMA copies in
// the swizzled layout and are normalised in place.  Once the record's bulk
// store has read it, the same bytes hold A / T (fp32), the block-product
// scratch and the T and P o D tiles of one value head.
constexpr int P_AT = 0;                    // [64][AS] fp32
constexpr int P_M = 64 * AS * 4;           // [32][MS] fp32
constexpr int P_TPD = 23552;               // T and P o D tiles (1024-byte aligned), 16 KiB
constexpr int PREP_BYTES = P_TPD + VREC_F;  // the value-head phase's scratch (the record image is smaller)
constexpr int PREP_SMEM = PREP_BYTES + 1024;
static_assert(P_M + 32 * MS * 4 <= P_TPD && KREC_BYTES <= PREP_BYTES, "prep shared-memory layout");

template <typename TIO, bool PAD>
__global__ void __launch_bounds__(PT, 4)
    wy_prep_kernel(const ForwardParams p, const int32_t *ws, uint8_t *krec, uint8_t *vrec,
                   const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k) {
    dependent_prologue();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar, lbar;
    __shared__ uint32_t tmem_base;
    __shared__ __align__(16) float Gam_s[GH][CH];  // within-chunk cumulative log2 decay per value head
    __shared__ float Beta_s[GH][CH];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr bool STAGED = sizeof(TIO) == 2;
    const int dk_ = PAD ? p.dk : DH;  // PAD: head size 32 or 64 on the zero-padded tiles

    const int g = blockIdx.x / p.Hk, kh = blockIdx.x % p.Hk;
    const int32_t *cbase = Header(const_cast<int32_t *>(ws), p.B).cbase;
    if (g >= cbase[p.B]) return;  // past the last chunk (the grid is sized by an upper bound)
    int lo = 0, hi = p.B;         // the sequence b with cbase[b] <= g < cbase[b + 1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cbase[mid] <= g) lo = mid;
        else hi = mid;
    }
    const int b = lo;
    const int bos = seq_start(p.cu, p.dense_S, b), eos = seq_start(p.cu, p.dense_S, b + 1);
    const int t0 = bos + CH * (g - cbase[b]);
    const int n = min(CH, eos - t0);

    // fp16: the chunk's q rows (tile rows 0-63) and k rows (64-127), both
    // 64-element halves of each, by swizzled 2-D TMA copies; rows past the
    // sequence arrive too and are zeroed when normalising
    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::mbar_init(&lbar, 1);
        ptx::fence_mbar_init();
        if (STAGED) {
            // one 64-feature box per K-block that holds features of this head (the
            // features past dk that a box brings are zeroed when normalising)
            const int nkb = (dk_ + 63) / 64;
            ptx::mbar_arrive_expect_tx(&lbar, (uint32_t)(nkb * 2 * CH * 64 * 2));
            for (int kb = 0; kb < nkb; ++kb) {
                ptx::tma_load_2d(sm + kb * 16384, &map_q, kh * dk_ + kb * 64, t0, &lbar);
                ptx::tma_load_2d(sm + kb * 16384 + CH * 128, &map_k, kh * dk_ + kb * 64, t0, &lbar);
            }
        }
    }
    __syncwarp();
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base, 64);
        ptx::tmem_relinquish();
    }
    // gates of the first GH value heads while the rows are in flight
    auto gates_group = [&](int i0) {
        const int wi = warp, i = i0 + wi;
        if (wi < GH && i < p.r) {
            const int h = kh * p.r + i;
            chunk_gates(p, t0, n, h, b, bos, Gam_s[wi], Beta_s[wi],
                        reinterpret_cast<float *>(vrec + ((size_t)g * p.Hv + h) * VREC_BYTES + VREC_F), lane);
        }
    };
    gates_group(0);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tm = tmem_base;
    bool ok = true;
    if (STAGED) ok = ptx::mbar_wait_bounded(&lbar, 0, WAIT_LIMIT);
    ok = __syncthreads_and(ok);

    // ---- L2-normalised q and k rows of the [Q;K] tile (zero past the sequence)
    if (STAGED) {
        // in place: four lanes per token (32 features each, as four 16-byte
        // pieces of the swizzled row), warp w handles tokens 8w .. 8w+7
        const int s = warp * 8 + (lane >> 2), qp = lane & 3;
        const int tl = t0 + s - bos;
#pragma unroll 1
        for (int which = 0; ok && which < 2; ++which) {  // q rows, then k rows
            const int rrow = which * 64 + s;
            float x[32];
            float ss = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(sm + sw(rrow, 32 * qp + 8 * m, 128));
                const __half2 *hv = reinterpret_cast<const __half2 *>(&raw);
                const bool in_head = 32 * qp + 8 * m < dk_;  // dk is a multiple of 32
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(hv[e]);
                    x[8 * m + 2 * e] = in_head ? f.x : 0.f;
                    x[8 * m + 2 * e + 1] = in_head ? f.y : 0.f;
                }
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) ss = fmaf(x[e], x[e], ss);
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            const float inv = 1.f / fmaxf(sqrtf(ss), EPS);
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = s < n ? x[e] * inv : 0.f;  // rows past the sequence become zero
#pragma unroll
            for (int m = 0; m < 4; ++m) st_h8(sm, sw(rrow, 32 * qp + 8 * m, 128), x + 8 * m);
            if (which == 1 && p.caps && s < n && tl < p.cap && 32 * qp < dk_) {
                float *dst = p.caps + ((long long)b * p.cap + tl) * p.W + p.Hv + (long long)kh * dk_ + 32 * qp;
#pragma unroll
                for (int e = 0; e < 32; ++e) dst[e] = x[e];  // rows need not be 16-byte aligned
            }
        }
    } else {
        // from global memory: warp w handles tokens w, w + 8, ..., four at a time
        const TIO *qg = static_cast<const TIO *>(p.q);
        const TIO *kg = static_cast<const TIO *>(p.k);
#pragma unroll 1
        for (int round = 0; ok && round < 2; ++round) {
            float qv[4][4], kv[4][4], sq[4], sk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = warp + 8 * (u + 4 * round);
#pragma unroll
                for (int e = 0; e < 4; ++e) qv[u][e] = kv[u][e] = 0.f;
                if (s < n && lane * 4 < dk_) {
                    const long long t = (long long)t0 + s;
                    ld4<TIO>(qg + t * p.q_stride + (long long)kh * dk_ + lane * 4, qv[u]);
                    ld4<TIO>(kg + t * p.k_stride + (long long)kh * dk_ + lane * 4, kv[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                sq[u] = sk[u] = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sq[u] = fmaf(qv[u][e], qv[u][e], sq[u]);
                    sk[u] = fmaf(kv[u][e], kv[u][e], sk[u]);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    sq[u] += __shfl_xor_sync(0xffffffffu, sq[u], off);
                    sk[u] += __shfl_xor_sync(0xffffffffu, sk[u], off);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = warp + 8 * (u + 4 * round);
                const float iq = 1.f / fmaxf(sqrtf(sq[u]), EPS), ik = 1.f / fmaxf(sqrtf(sk[u]), EPS);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    qv[u][e] *= iq;
                    kv[u][e] *= ik;
                }
                const int c = lane * 4;
                st_h4(sm, sw(s, c, 128), qv[u][0], qv[u][1], qv[u][2], qv[u][3]);
                st_h4(sm, sw(64 + s, c, 128), kv[u][0], kv[u][1], kv[u][2], kv[u][3]);
                const int tl = t0 + s - bos;
                if (p.caps && s < n && tl < p.cap && c < dk_) {
                    float *dst = p.caps + ((long long)b * p.cap + tl) * p.W + p.Hv + (long long)kh * dk_ + c;
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = kv[u][e];  // rows need not be 16-byte aligned
                }
            }
        }
    }
    __syncthreads();
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    // ---- [Q;K] K^T on the tensor cores (P in lanes 0-63, G in lanes 64-127),
    //      and the key-head record to the workspace
    if (ok && tid == 0) {
        ptx::tc_fence_after();
        const uint32_t a_qk = ptx::smem_u32(sm);
        const uint32_t i64 = ptx::idesc_f16_f32(128, 64);
        for (int ks = 0; ks < dk_ / 16; ++ks) {  // features past dk are zero
            const uint32_t ko = (ks >> 2) * 16384 + (ks & 3) * 32;
            ptx::mma_f16(tm, ptx::sdesc_k_sw128(a_qk + ko), ptx::sdesc_k_sw128(a_qk + 64 * 128 + ko), i64, ks > 0);
        }
        ptx::mma_commit(&bar);
        ptx::bulk_s2g(krec + ((size_t)g * p.Hk + kh) * KREC_BYTES, sm, KREC_BYTES);
        ptx::bulk_commit();
    }
    const bool mma_issued = ok;
    if (ok) ok = ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);
    ptx::tc_fence_after();
    if (tid == 0) ptx::bulk_wait_read_all();  // the tile bytes may be reused from here on
    ok = __syncthreads_and(ok);

    // ---- per value head of this key head: A and P o D, T, record
    float *AT = reinterpret_cast<float *>(sm + P_AT);
    float *Mw = reinterpret_cast<float *>(sm + P_M);
    uint8_t *tpd = sm + P_TPD;
    const int quarter = warp & 3, c32 = (warp >> 2) * 32;
    const int row = quarter * 32 + lane;  // tensor-memory lane of this thread
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
#pragma unroll 1
    for (int i = 0; ok && i < p.r; ++i) {
        const int h = kh * p.r + i, wi = i % GH;
        if (i > 0 && wi == 0) {  // the next group of heads' gates
            gates_group(i);
            __syncthreads();
        }
        if ((quarter & 1) == 0 && c32 == 32) {  // rows 0-31, columns 32-63: above the diagonal, all zero
            const int r = row & 63;
            if (quarter >= 2) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(AT + r * AS + c32 + j) = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 32; j += 8) st_h8(tpd + VREC_PD, sw(r, c32 + j, 64), z);
            }
        } else {
            float v[32];
            ptx::tmem_ld32(tm + lane_sel + c32, v);
            const int r = row & 63;
            const float *Gm = Gam_s[wi];  // cumulative log2 decays: columns read 8 at a time (broadcast)
            const float Gr = Gm[r];
            if (quarter >= 2) {  // lanes 64-127: G = K K^T -> A (strictly lower)
                const float br = Beta_s[wi][r];
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    float gc[8], w[8];
                    ld_fn<8>(Gm + c32 + j, gc);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = c32 + j + e;
                        w[e] = (s < r) ? br * ex2_approx(Gr - gc[e]) * v[j + e] : 0.f;
                    }
                    // 16-byte stores: with the 68-float row stride a quarter-warp's 8 rows
                    // cover all 32 banks (single-float stores of one column hit 8)
                    float4 *dst = reinterpret_cast<float4 *>(AT + r * AS + c32 + j);
                    dst[0] = make_float4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_float4(w[4], w[5], w[6], w[7]);
                }
            } else {  // lanes 0-63: P = Q K^T -> P o D (lower, diagonal included)
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    float w[8], gc[8];
                    ld_fn<8>(Gm + c32 + j, gc);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = c32 + j + e;
                        w[e] = (s <= r) ? v[j + e] * ex2_approx(Gr - gc[e]) : 0.f;
                    }
                    st_h8(tpd + VREC_PD, sw(r, c32 + j, 64), w);
                }
            }
        }
        __syncthreads();
        tri_inverse_inplace(AT, Mw, tid);
        {  // T -> fp16 tile: thread (r, 16-column group)
            const int r = tid >> 2, s0 = (tid & 3) * 16;
#pragma unroll
            for (int j = 0; j < 16; j += 8) {
                float w[8];
                const float4 a = *reinterpret_cast<const float4 *>(AT + r * AS + s0 + j);
                const float4 c = *reinterpret_cast<const float4 *>(AT + r * AS + s0 + j + 4);
                w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
                w[4] = c.x; w[5] = c.y; w[6] = c.z; w[7] = c.w;
                st_h8(tpd + VREC_T, sw(r, s0 + j, 64), w);
            }
        }
        ptx::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            ptx::bulk_s2g(vrec + ((size_t)g * p.Hv + h) * VREC_BYTES, tpd, VREC_F);
            ptx::bulk_commit();
            ptx::bulk_wait_read_all();
        }
        __syncthreads();
    }
    if (!ok && tid == 0) {
        flag_error(p.status, GDN_DEVERR_TIMEOUT);
        if (mma_issued) ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);  // let the MMA drain before tensor memory is freed
        if (STAGED) ptx::mbar_wait_bounded(&lbar, 0, WAIT_LIMIT);      // and the row copies
    }
    if (tid == 0) ptx::bulk_wait_all();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tm, 64);
    }
}

// ---------------------------------------------------------------- phase 2: per (sequence, value head) chain

constexpr int NT = 512;  // 16 warps: four per tensor-memory lane quarter (32 warps measured slower)
// Columns a thread handles of a 64-column (CW) and of a 128-column (CS) region.
constexpr int CW = 64 / (NT / 128), CS = 2 * CW;
static_assert(CW % 8 == 0, "16-byte tile stores need 8-column pieces");
constexpr int TMEM_COLS = 512;
// Tensor-memory columns (128 lanes each).  MMA2's result is double-buffered
// so that chunk c - 1's outputs are read while chunk c's MMA2 runs.
constexpr uint32_t TM_S = 0;     // FP32 state S (dv lanes x dk columns)
constexpr uint32_t TM_OX = 128;  // two buffers of 128 columns: O' = S0 Q^T (64), then X = S0 K^T (64)
constexpr uint32_t TM_U = 384;   // U^T
constexpr uint32_t TM_Y = 448;   // U^T (P o D)^T

// Shared memory (offsets from a 1024-byte aligned base): two stages holding
// one chunk's inputs each, then the fp16 state copy and the R^T / U^T tile.
constexpr int S_KREC = 0;                   // key-head record: [Q;K] tile (k rows from byte 64 * 128 of each K-block)
constexpr int S_VREC = KREC_BYTES;          // value-head record: T, P o D, per-token factors
constexpr int S_V = S_VREC + VREC_BYTES;    // fp16 v rows of the chunk [64][128]; then U^T diag(decay) tile
constexpr int STAGE_BYTES = S_V + 16384;
constexpr int OFF_S16 = 2 * STAGE_BYTES;    // [128][128] fp16 S0 (two K-blocks)
constexpr int OFF_RT = OFF_S16 + 32768;     // [128][64] fp16 R^T, then U^T
constexpr int OFF_OT = OFF_RT + 16384;      // fp16 I/O: a full chunk's outputs [64 tokens][128] for one tensor store
constexpr int SCAN_SMEM = OFF_OT + 16384 + 1024;  // + slack for the 1024-byte alignment
static_assert(S_V % 1024 == 0 && STAGE_BYTES % 1024 == 0, "stage layout");
static_assert(SCAN_SMEM + 1024 <= 227 * 1024, "shared memory budget (dynamic + static)");

// SPLIT = false: every chain is a whole sequence (the work list holds no
// other kind), and the split-plan code is compiled out.
template <typename TIO, bool SPLIT, bool PAD>
__global__ void __launch_bounds__(NT, 1)
    wy_scan_kernel(const ForwardParams p, int32_t *ws, const uint8_t *krec, const uint8_t *vrec, float *split_states,
                   TIO *oid, const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                   const __grid_constant__ CUtensorMap map_oi, int out_tma) {
    dependent_prologue();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar;      // MMA completion
    __shared__ __align__(8) uint64_t lbar[2];  // stage loads
    __shared__ uint32_t tmem_base;
    __shared__ int item_s;
    __shared__ __align__(16) float gam_prev[CH];  // gamma of the chunk whose outputs are pending
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Tensor memory: a warp reaches only the 32 lanes of its quarter (warp % 4);
    // the NT / 128 warps of a quarter split the columns.
    const int quarter = warp & 3, cq = warp >> 2;
    const int row = quarter * 32 + lane;  // the tensor-memory lane (state / output row) of this thread
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int c16 = cq * CW, c32 = cq * CS;  // this thread's first column of a 64- / 128-column region

    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::mbar_init(&lbar[0], 1);
        ptx::mbar_init(&lbar[1], 1);
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tm = tmem_base;
    uint32_t phase = 0, lph[2] = {0u, 0u};
    bool pending[2] = {false, false};
    bool failed = false;
    constexpr bool STAGED = sizeof(TIO) == 2;
    // Shared-memory descriptors: a step of 16 elements along K adds 32 bytes,
    // i.e. 2 to the descriptor's address field (addresses stay below 256 KiB,
    // so the 14-bit field never carries).
    const uint64_t d_S16 = ptx::sdesc_k_sw128(ptx::smem_u32(sm + OFF_S16));
    const uint64_t d_RT = ptx::sdesc_k_sw128(ptx::smem_u32(sm + OFF_RT));
    constexpr uint32_t I64 = ptx::idesc_f16_f32(128, 64), I128 = ptx::idesc_f16_f32(128, 128);
    constexpr uint32_t I128_BMN = ptx::idesc_f16_f32(128, 128, true);  // B MN-major

    auto mma_wait = [&]() -> bool {
        const bool ok = ptx::mbar_wait_bounded(&bar, phase, WAIT_LIMIT);
        phase ^= 1u;
        ptx::tc_fence_after();
        return __syncthreads_and(ok);
    };
    auto mma_ready = [&]() {  // this thread's smem / tmem writes become visible to the next MMA
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
    };
    auto stage_wait = [&](int st) -> bool {
        const bool ok = ptx::mbar_wait_bounded(&lbar[st], lph[st], WAIT_LIMIT);
        lph[st] ^= 1u;
        pending[st] = false;
        return __syncthreads_and(ok);
    };

    const Header hd(ws, p.B);
    const int n_items = hd.w[1] * p.Hv;
    const int32_t *cbase = hd.cbase;
    const TIO *vg = static_cast<const TIO *>(p.v);
    // PAD: head sizes 32 / 64 on the zero-padded tiles (otherwise 128, known at compile time)
    const int dk_ = PAD ? p.dk : DH, dv_ = PAD ? p.dv : DH;
    const long long ubase = (long long)p.Hv + (long long)p.Hk * dk_;
    // this thread's state row and 32-column block hold data (the rest is zero padding)
    const bool row_in = !PAD || row < dv_, cols_in = !PAD || c32 < dk_;

    while (!failed) {
        if (tid == 0) item_s = atomicAdd(&hd.w[0], 1);
        __syncthreads();
        const int item = item_s;
        __syncthreads();
        if (item >= n_items) break;
        const int e = hd.list[item / p.Hv], h = item % p.Hv, kh = h / p.r;
        const int b = e >> 2, kind = SPLIT ? (e & 3) : K_WHOLE;
        const int bos = seq_start(p.cu, p.dense_S, b), eos = seq_start(p.cu, p.dense_S, b + 1);
        const int nc = (eos - bos + CH - 1) / CH;
        // the chunks of this chain: a whole sequence, or one segment of a split one
        const int c1 = (nc + 1) / 2;
        const int c_lo = kind >= K_ZERO ? c1 : 0, c_hi = kind == K_FIRST ? c1 : nc;
        const long long gbase = cbase[b];
        const int slot = p.slots ? p.slots[b] : b;
        if (slot < 0 || slot >= p.num_slots) {
            if (tid == 0 && h == 0 && kind <= K_FIRST) flag_error(p.status, GDN_DEVERR_STATE_SLOT);
            continue;
        }
        const size_t head_off = ((size_t)slot * p.Hv + h) * (size_t)dv_ * dk_;
        // where the outputs and the final state go: a split sequence's first segment
        // leaves its state S1 in the workspace, the second segment's zero run writes
        // the outputs (corrected later) and B, the identity run its outputs to the
        // workspace rows of this sequence and A
        float *sstate = nullptr;
        if (kind != K_WHOLE) sstate = split_states + ((size_t)(hd.sidx[b] * 3 + kind - 1) * p.Hv + h) * (DH * DH);
        TIO *const og = kind == K_IDENT ? oid : static_cast<TIO *>(p.out);
        const long long orow = kind == K_IDENT ? (long long)hd.obase[hd.sidx[b]] - (bos + CH * c1) : 0;
        const CUtensorMap *const mo = kind == K_IDENT ? &map_oi : &map_o;
        float *const fdst = kind == K_FIRST ? sstate
                                            : (p.final_state ? (kind == K_WHOLE ? p.final_state + head_off : sstate)
                                                             : nullptr);
        // capsule deltas come from chains that run from the true state (a split
        // sequence's captured tokens all lie in its first segment)
        const bool caps_here = p.caps != nullptr && kind <= K_FIRST;

        // chunk c's records (and fp16 v rows) into stage st
        auto stage_load = [&](int c, int st) {
            if (tid == 0) {
                uint8_t *stage = sm + st * STAGE_BYTES;
                ptx::mbar_arrive_expect_tx(&lbar[st], (uint32_t)(KREC_BYTES + VREC_BYTES + (STAGED ? CH * DH * 2 : 0)));
                ptx::bulk_g2s(stage + S_KREC, krec + ((gbase + c) * p.Hk + kh) * KREC_BYTES, KREC_BYTES, &lbar[st]);
                ptx::bulk_g2s(stage + S_VREC, vrec + ((gbase + c) * p.Hv + h) * VREC_BYTES, VREC_BYTES, &lbar[st]);
                if (STAGED) ptx::tma_load_2d(stage + S_V, &map_v, h * dv_, bos + CH * c, &lbar[st]);
            }
            pending[st] = true;
        };
        // S0 -> fp16 operand tile; the tensor-memory state becomes gamma_last S0
        bool state_live = kind == K_IDENT || (kind != K_ZERO && p.init != nullptr);
        auto build_s16 = [&](const float *F, int n) {
            const float gl = F[F_GAMMA + n - 1];
            float v[CS];
            if (state_live) {
                ptx::tmem_ld<CS>(tm + lane_sel + TM_S + c32, v);
            } else {
#pragma unroll
                for (int j = 0; j < CS; ++j) v[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < CS; j += 8) st_h8(sm + OFF_S16, sw(row, c32 + j, 128), v + j);
            if (state_live) {
#pragma unroll
                for (int j = 0; j < CS; ++j) v[j] *= gl;
                ptx::tmem_st<CS>(tm + lane_sel + TM_S + c32, v);
                ptx::tmem_st_wait();
            }
        };
        // outputs of the chunk starting at tp (n tokens): o = scale (gamma O' + Y).  With
        // `tile` (fp16, a full chunk) they go to the output tile for one tensor store.
        auto write_outputs = [&](int tp, int n, uint32_t ox, bool tile) {
            float o1[CW], y[CW], gm[CW];
            ptx::tmem_ld<CW>(tm + lane_sel + ox + c16, o1);
            ptx::tmem_ld<CW>(tm + lane_sel + TM_Y + c16, y);
            ld_fn<CW>(gam_prev + c16, gm);
            if (tile) {
                __half *ot = reinterpret_cast<__half *>(sm + OFF_OT);
#pragma unroll
                for (int j = 0; j < CW; ++j)
                    if (row_in) ot[(c16 + j) * dv_ + row] = __float2half_rn(p.scale * fmaf(gm[j], o1[j], y[j]));
                ptx::fence_proxy_async_smem();  // visible to the tensor store after the next barrier
                return;
            }
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                const int s = c16 + j;
                if (s < n && row_in)
                    og[((long long)(tp + s) + orow) * p.Hv * dv_ + (long long)h * dv_ + row] =
                        from_f32<TIO>(p.scale * fmaf(gm[j], o1[j], y[j]));
            }
        };
        const bool out_tile = STAGED && out_tma;

        // ---- chain start: the initial state into tensor memory, the first chunk's inputs
        if (kind == K_IDENT) {
            float v[CS];
#pragma unroll
            for (int j = 0; j < CS; ++j) v[j] = c32 + j == row ? 1.f : 0.f;
            ptx::tmem_st<CS>(tm + lane_sel + TM_S + c32, v);
            ptx::tmem_st_wait();
        } else if (state_live) {
            const float *src = p.init + head_off + (size_t)row * dk_ + c32;
            float v[CS];
#pragma unroll
            for (int j = 0; j < CS; j += 4) {
                const float4 x = row_in && cols_in ? *reinterpret_cast<const float4 *>(src + j)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                v[j] = x.x; v[j + 1] = x.y; v[j + 2] = x.z; v[j + 3] = x.w;
            }
            ptx::tmem_st<CS>(tm + lane_sel + TM_S + c32, v);
            ptx::tmem_st_wait();
        }
        if (c_hi > c_lo) {
            stage_load(c_lo, 0);
            if (c_hi > c_lo + 1) stage_load(c_lo + 1, 1);
            if (!stage_wait(0)) { failed = true; break; }
            build_s16(reinterpret_cast<const float *>(sm + S_VREC + VREC_F), min(CH, eos - bos - CH * c_lo));
        }
        mma_ready();

        for (int c = c_lo; c < c_hi && !failed; ++c) {
            const int st = (c - c_lo) & 1;
            uint8_t *stage = sm + st * STAGE_BYTES;
            const float *F = reinterpret_cast<const float *>(stage + S_VREC + VREC_F);
            const int t0 = bos + CH * c, n = min(CH, eos - t0);
            const uint32_t a_st = ptx::smem_u32(stage);
            const uint32_t ox = TM_OX + 128u * (uint32_t)st;
            // ---- MMA2: [O' | X] = S0 [Q;K]^T
            if (tid == 0) {
                ptx::tc_fence_after();
                const uint64_t bd = ptx::sdesc_k_sw128(a_st + S_KREC);
                for (int ks = 0; ks < dk_ / 16; ++ks) {  // state columns past dk are zero
                    const uint32_t ko = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                    ptx::mma_f16(tm + ox, d_S16 + ko, bd + ko, I128, ks > 0);
                }
                ptx::mma_commit(&bar);
            }
            // ---- while MMA2 runs: the outputs of chunk c - 1
            if (c > c_lo) write_outputs(t0 - CH, CH, TM_OX + 128u * (uint32_t)(st ^ 1), out_tile);
            if (!mma_wait()) { failed = true; break; }
            if (c > c_lo && out_tile && tid == 0) {  // chunk c - 1's outputs, one tensor store
                ptx::tma_store_2d(mo, sm + OFF_OT, h * dv_, (int)(t0 - CH + orow));
                ptx::bulk_commit();
            }
            // ---- R^T = diag(beta) V - diag(beta gamma) X^T, transposed; this chunk's gamma for its outputs
            {
                float x[CW];
                ptx::tmem_ld<CW>(tm + lane_sel + ox + 64 + c16, x);
                float be[CW], bg[CW];
                ld_fn<CW>(F + F_BETA + c16, be);
                ld_fn<CW>(F + F_BG + c16, bg);
                if (kind == K_IDENT) {  // the identity run has no v term
#pragma unroll
                    for (int j = 0; j < CW; ++j) be[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < CW; j += 8) {
                    float w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = c16 + j + e;
                        float vv;
                        if (!row_in)
                            vv = 0.f;  // the tile's rows past dv hold the next head's features
                        else if (STAGED)
                            vv = to_f32(reinterpret_cast<const TIO *>(stage + S_V)[s * DH + row]);
                        else
                            vv = s < n ? to_f32(vg[(long long)(t0 + s) * p.v_stride + (long long)h * dv_ + row]) : 0.f;
                        w[e] = fmaf(be[j + e], vv, -bg[j + e] * x[j + e]);
                    }
                    st_h8(sm + OFF_RT, sw(row, c16 + j, 128), w);
                }
                if (tid < CH) gam_prev[tid] = F[F_GAMMA + tid];
            }
            mma_ready();
            // ---- MMA3: U^T = R^T T^T
            if (tid == 0) {
                ptx::tc_fence_after();
                const uint64_t bd = ptx::sdesc_k_sw128(a_st + S_VREC + VREC_T);
                for (int ks = 0; ks < CH / 16; ++ks) ptx::mma_f16(tm + TM_U, d_RT + 2 * ks, bd + 2 * ks, I64, ks > 0);
                ptx::mma_commit(&bar);
            }
            if (!mma_wait()) { failed = true; break; }
            // ---- U^T -> fp16 operands (plain, and decayed to the chunk end in the
            //      v tile, which is free now)
            float u[CW], dc[CW];
            ptx::tmem_ld<CW>(tm + lane_sel + TM_U + c16, u);
            ld_fn<CW>(F + F_DECAY + c16, dc);
#pragma unroll
            for (int j = 0; j < CW; j += 8) {
                float w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = dc[j + e] * u[j + e];
                st_h8(sm + OFF_RT, sw(row, c16 + j, 128), u + j);
                st_h8(stage + S_V, sw(row, c16 + j, 128), w);
            }
            mma_ready();
            // ---- MMA4 (Y = U^T (P o D)^T) and MMA5 (state)
            if (tid == 0) {
                ptx::tc_fence_after();
                const uint64_t ud = ptx::sdesc_k_sw128(a_st + S_V), pd = ptx::sdesc_k_sw128(a_st + S_VREC + VREC_PD);
                // K as MN-major B: 16 tokens per step = 16 rows of 128 B = 2048 B
                const uint64_t kt = ptx::sdesc_mn_sw128(a_st + S_KREC + 64 * 128, 16384);
                for (int ks = 0; ks < CH / 16; ++ks) {
                    ptx::mma_f16(tm + TM_Y, d_RT + 2 * ks, pd + 2 * ks, I64, ks > 0);
                    ptx::mma_f16(tm + TM_S, ud + 2 * ks, kt + 128 * ks, I128_BMN, (state_live || ks > 0) ? 1u : 0u);
                }
                ptx::mma_commit(&bar);
            }
            // the capsule deltas while MMA4/5 run
            if (caps_here) {
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    const int s = c16 + j, tl = t0 + s - bos;
                    if (s < n && tl < p.cap && row_in)
                        p.caps[((long long)b * p.cap + tl) * p.W + ubase + (long long)h * dv_ + row] = u[j];
                }
            }
            if (!mma_wait()) { failed = true; break; }
            state_live = true;
            // this stage is free now (its gamma was copied to gam_prev): chunk c + 2 goes there
            if (c + 2 < c_hi) stage_load(c + 2, st);
            // ---- the next chunk's fp16 state copy (its inputs first)
            if (c + 1 < c_hi) {
                if (!stage_wait(st ^ 1)) { failed = true; break; }
                build_s16(reinterpret_cast<const float *>(sm + (st ^ 1) * STAGE_BYTES + S_VREC + VREC_F),
                          min(CH, eos - t0 - CH));
            } else {
                write_outputs(t0, n, ox, false);  // the last chunk's outputs: no MMA left to overlap
            }
            if (out_tile && tid == 0) ptx::bulk_wait_read_all();  // the output tile is free again
            mma_ready();
        }
        if (failed) break;
        // ---- chain end: the final state (unless the caller asked for none)
        if (fdst) {
            ptx::tc_fence_after();
            float *dst = fdst + (size_t)row * (kind == K_WHOLE ? dk_ : DH) + c32;
            float v[CS];
            if (state_live) {
                ptx::tmem_ld<CS>(tm + lane_sel + TM_S + c32, v);
            } else {
#pragma unroll
                for (int j = 0; j < CS; ++j) v[j] = 0.f;
            }
            if (row_in && cols_in) {
#pragma unroll
                for (int j = 0; j < CS; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
    }

    if (failed && tid == 0) {
        flag_error(p.status, GDN_DEVERR_TIMEOUT);
        ptx::mbar_wait_bounded(&bar, phase ^ 1u, WAIT_LIMIT);  // let in-flight MMAs drain
        ptx::mbar_wait_bounded(&bar, phase, WAIT_LIMIT);
        for (int st = 0; st < 2; ++st)  // and the staged copies
            if (pending[st]) ptx::mbar_wait_bounded(&lbar[st], lph[st], WAIT_LIMIT);
    }
    if (tid == 0) ptx::bulk_wait_all();  // the output tensor stores are complete
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tm, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- split plan: combining the segments

// Outputs of each split sequence's second segment: o_t += S1 o_t(identity),
// over tiles of OC_ROWS tokens of one (split sequence, value head).  Per tile
// one tcgen05 product [OC_ROWS tokens x dk] x [dk x dv] (the identity-run
// rows and the fp16 copy of S1, both K-major in the 128-byte swizzled
// layout) accumulates in tensor memory; the epilogue thread of token t adds
// its row to the output already there (the zero run's) and rounds once.
// Persistent over contiguous ranges of tiles, so consecutive tiles share
// (sequence, head) and S1 is converted once per range piece.
//
// HBM-bound (per token and head, fp16: 256 B of identity-run rows and 256 B
// of output read, 256 B written).  With fp16 I/O every copy is a tensor copy
// that overlaps other work: the next tile's identity-run rows load as soon as
// the product has read the current ones, the tile's output rows load (into a
// third swizzled tile) while S1 is converted and the product runs, and a full
// tile's updated rows leave by tensor stores that complete during the next
// tile.  A tile that ends past its sequence is written row by row by its
// threads instead, so rows of the next sequence are never stored.
constexpr int OC_NT = 128;
constexpr int OC_TILE = OC_ROWS * DH * 2;  // one fp16 [OC_ROWS][128] tile, two K-blocks
constexpr int OC_SMEM = 3 * OC_TILE + 1024;

// dst[0 .. 32) += c (FP32 I/O; 16-byte accesses).
__device__ __forceinline__ void add_row32(float *dst, const float (&c)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float4 v = reinterpret_cast<float4 *>(dst)[q];
        v.x += c[4 * q];
        v.y += c[4 * q + 1];
        v.z += c[4 * q + 2];
        v.w += c[4 * q + 3];
        reinterpret_cast<float4 *>(dst)[q] = v;
    }
}

// Eight fp16 values (one 16-byte piece of a row) plus c[0 .. 8), rounded once.
__device__ __forceinline__ uint4 add_h8(uint4 v, const float *c) {
    __half2 *hv = reinterpret_cast<__half2 *>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(hv[e]);
        hv[e] = __floats2half2_rn(f.x + c[2 * e], f.y + c[2 * e + 1]);
    }
    return v;
}

struct OcTile {
    int j, h, b, eos, t0, slot;
    long long r0;  // first identity-run row of the tile
};

template <typename TIO>
__global__ void __launch_bounds__(OC_NT, 1)
    wy_out_correction_kernel(const ForwardParams p, int32_t *ws, const float *split_states, const TIO *oid,
                             const __grid_constant__ CUtensorMap map_oa, const __grid_constant__ CUtensorMap map_out,
                             int tma) {
    dependent_prologue();
    constexpr bool F16 = sizeof(TIO) == 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *a_t = sm;                // identity-run outputs: [OC_ROWS][dk] fp16
    uint8_t *b_t = sm + OC_TILE;      // S1 (dv rows) as fp16
    uint8_t *o_t = sm + 2 * OC_TILE;  // the tile's output rows (fp16 I/O with tensor copies)
    __shared__ __align__(8) uint64_t bar, lbar, obar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5;
    const Header hd(ws, p.B);
    const int ns = hd.w[2];
    const long long ntiles = (long long)hd.tbase[ns] * p.Hv;
    const long long u0 = (long long)blockIdx.x * ntiles / gridDim.x;
    const long long u1 = (long long)(blockIdx.x + 1) * ntiles / gridDim.x;
    if (u0 >= u1) return;
    const bool use_tma = F16 && tma;
    // tile u -> split index j (tiles of j: [Hv tbase[j], Hv tbase[j + 1]), head-major), head, position
    auto resolve = [&](long long u) {
        int lo = 0, hi = ns;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((long long)hd.tbase[mid] * p.Hv <= u) lo = mid;
            else hi = mid;
        }
        OcTile x;
        x.j = lo;
        const long long nt = hd.tbase[lo + 1] - hd.tbase[lo];
        const long long rel = u - (long long)hd.tbase[lo] * p.Hv;
        x.h = (int)(rel / nt);
        const int k = (int)(rel % nt);
        x.b = hd.sseq[lo];
        const int bos = seq_start(p.cu, p.dense_S, x.b);
        x.eos = seq_start(p.cu, p.dense_S, x.b + 1);
        const int c1 = ((x.eos - bos + CH - 1) / CH + 1) / 2;
        x.t0 = bos + CH * c1 + OC_ROWS * k;
        x.r0 = hd.obase[lo] + (long long)OC_ROWS * k;
        x.slot = p.slots ? p.slots[x.b] : x.b;
        return x;
    };
    // thread 0: a tile's rows as two swizzled boxes of 64 columns
    auto load_tile = [&](uint8_t *dst, const CUtensorMap *map, int x0, int y0, uint64_t *mb) {
        ptx::mbar_arrive_expect_tx(mb, OC_TILE);
        ptx::tma_load_2d(dst, map, x0, y0, mb);
        ptx::tma_load_2d(dst + OC_ROWS * 128, map, x0 + 64, y0, mb);
    };
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base, 128);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::mbar_init(&lbar, 1);
        ptx::mbar_init(&obar, 1);
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tm = tmem_base;
    const uint32_t lane_sel = (uint32_t)(warp * 32) << 16;
    constexpr uint32_t I128 = ptx::idesc_f16_f32(128, 128);
    uint32_t ph = 0, lph = 0, oph = 0;
    bool ok = true, mma_out = false, a_out = false, o_out = false;
    int cur = -1;  // (split index, head) whose S1 is in b_t
    TIO *og = static_cast<TIO *>(p.out);
    OcTile x = resolve(u0);
    if (use_tma && tid == 0) {
        load_tile(a_t, &map_oa, x.h * DH, (int)x.r0, &lbar);
        a_out = true;
    }
    // a bounded wait on one of this CTA's barriers (false: flagged by the caller)
    auto wait_on = [&](uint64_t *mb, uint32_t &par, bool &outstanding) -> bool {
        const bool got = ptx::mbar_wait_bounded(mb, par, WAIT_LIMIT);
        if (got) {
            par ^= 1u;
            outstanding = false;
        }
        return __syncthreads_and(got);
    };
    for (long long u = u0; u < u1 && ok; ++u) {
        // Tiles of a sequence whose slot is out of range run like the others but
        // write nothing (the scan flagged the slot and computed nothing for it).
        const bool live_seq = x.slot >= 0 && x.slot < p.num_slots;
        const int t = x.t0 + tid;
        const bool live = live_seq && t < x.eos;
        const bool full = live_seq && x.t0 + OC_ROWS <= x.eos;  // every row of the tile is this sequence's
        TIO *dst = og + ((long long)t * p.Hv + x.h) * DH;
        if (use_tma && tid == 0) {  // the output rows; the buffer's previous tensor store has read it
            ptx::bulk_wait_read_all();
            load_tile(o_t, &map_out, x.h * DH, x.t0, &obar);
            o_out = true;
        }
        if (!use_tma) {  // rows converted here, zero past the segment
            const TIO *src = oid + ((x.r0 + tid) * p.Hv + x.h) * DH;
#pragma unroll 4
            for (int col = 0; col < DH; col += 8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = live ? to_f32(src[col + e]) : 0.f;
                st_h8(a_t, sw(tid, col, OC_ROWS), v);
            }
        }
        if (x.j * p.Hv + x.h != cur) {  // S1 of this (sequence, head) -> fp16 operand
            cur = x.j * p.Hv + x.h;
            const float *s1 = split_states + ((size_t)x.j * 3 * p.Hv + x.h) * (DH * DH) + (size_t)tid * DH;
#pragma unroll 4
            for (int col = 0; col < DH; col += 8) {
                const float4 x0 = *reinterpret_cast<const float4 *>(s1 + col);
                const float4 x1 = *reinterpret_cast<const float4 *>(s1 + col + 4);
                const float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                st_h8(b_t, sw(tid, col, DH), v);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (use_tma && !(ok = wait_on(&lbar, lph, a_out))) break;
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint64_t ad = ptx::sdesc_k_sw128(ptx::smem_u32(a_t)), bd = ptx::sdesc_k_sw128(ptx::smem_u32(b_t));
            for (int ks = 0; ks < DH / 16; ++ks) {
                const uint32_t ko = ((ks >> 2) * (OC_ROWS * 128) + (ks & 3) * 32) >> 4;
                ptx::mma_f16(tm, ad + ko, bd + ko, I128, ks > 0);
            }
            ptx::mma_commit(&bar);
        }
        mma_out = true;
        if (!(ok = wait_on(&bar, ph, mma_out))) break;
        ptx::tc_fence_after();
        // the operand tile is free: the next tile's rows are on their way during this epilogue
        const OcTile cx = x;
        if (u + 1 < u1) {
            x = resolve(u + 1);
            if (use_tma && tid == 0) {
                load_tile(a_t, &map_oa, x.h * DH, (int)x.r0, &lbar);
                a_out = true;
            }
        }
        if (use_tma) {
            if (!(ok = wait_on(&obar, oph, o_out))) break;
            // token t's row: TMEM columns 32q .. 32q + 31 onto the swizzled output tile
#pragma unroll
            for (int q = 0; q < DH / 32; ++q) {
                float c[32];
                ptx::tmem_ld32(tm + lane_sel + 32 * q, c);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint4 *pv = reinterpret_cast<uint4 *>(o_t + sw(tid, 32 * q + 8 * m, OC_ROWS));
                    const uint4 r = add_h8(*pv, c + 8 * m);
                    if (full) *pv = r;
                    else if (live) reinterpret_cast<uint4 *>(dst)[4 * q + m] = r;
                }
            }
            ptx::fence_proxy_async_smem();
            __syncthreads();
            if (full && tid == 0) {
                ptx::tma_store_2d(&map_out, o_t, cx.h * DH, cx.t0);
                ptx::tma_store_2d(&map_out, o_t + OC_ROWS * 128, cx.h * DH + 64, cx.t0);
                ptx::bulk_commit();
            }
        } else {
#pragma unroll
            for (int q = 0; q < DH / 32; ++q) {
                float c[32];
                ptx::tmem_ld32(tm + lane_sel + 32 * q, c);
                if (!live) continue;
                if constexpr (F16) {
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        reinterpret_cast<uint4 *>(dst)[4 * q + m] =
                            add_h8(reinterpret_cast<const uint4 *>(dst)[4 * q + m], c + 8 * m);
                } else {
                    add_row32(reinterpret_cast<float *>(dst) + 32 * q, c);
                }
            }
        }
        ptx::tc_fence_before();
        __syncthreads();
    }
    if (tid == 0) {
        if (!ok) flag_error(p.status, GDN_DEVERR_TIMEOUT);
        if (mma_out) ptx::mbar_wait_bounded(&bar, ph, WAIT_LIMIT);  // let the MMA drain before tensor memory is freed
        if (a_out) ptx::mbar_wait_bounded(&lbar, lph, WAIT_LIMIT);  // and the copies in flight
        if (o_out) ptx::mbar_wait_bounded(&obar, oph, WAIT_LIMIT);
        ptx::bulk_wait_all();  // the tensor stores are complete
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tm, 128);
    }
}

// Final state of each split sequence: S1 A + B (FP32, CUDA cores), one CTA
// per (split sequence, value head); 8 x 8 outputs per thread.
constexpr int FS_NT = 256;
constexpr int FS_LD = DH + 1;  // row stride of S1 in shared memory (column reads conflict-free)
constexpr int FS_SMEM = (DH * FS_LD + DH * DH) * 4;

__global__ void __launch_bounds__(FS_NT, 1)
    wy_split_final_kernel(const ForwardParams p, const int32_t *ws, const float *split_states) {
    dependent_prologue();
    extern __shared__ float fs_smem[];
    float *s1 = fs_smem;           // [dv][FS_LD]
    float *am = fs_smem + DH * FS_LD;  // [dk][dk]
    const Header hd(const_cast<int32_t *>(ws), p.B);
    const int j = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv;
    if (j >= hd.w[2]) return;
    const int b = hd.sseq[j];
    const int slot = p.slots ? p.slots[b] : b;
    if (slot < 0 || slot >= p.num_slots) return;
    const int tid = threadIdx.x;
    const float *S1 = split_states + ((size_t)(j * 3 + 0) * p.Hv + h) * (DH * DH);
    const float *Bm = split_states + ((size_t)(j * 3 + 1) * p.Hv + h) * (DH * DH);
    const float *Am = split_states + ((size_t)(j * 3 + 2) * p.Hv + h) * (DH * DH);
    for (int i = tid; i < DH * DH / 4; i += FS_NT) {
        const float4 x = reinterpret_cast<const float4 *>(S1)[i];
        const int r = (4 * i) / DH, c = (4 * i) % DH;
        s1[r * FS_LD + c] = x.x;
        s1[r * FS_LD + c + 1] = x.y;
        s1[r * FS_LD + c + 2] = x.z;
        s1[r * FS_LD + c + 3] = x.w;
        reinterpret_cast<float4 *>(am)[i] = reinterpret_cast<const float4 *>(Am)[i];
    }
    __syncthreads();
    const int i0 = (tid >> 4) * 8, m0 = (tid & 15) * 4;  // rows i0 .. i0+7; columns m0 .. m0+3 and 64 + m0 ..
    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < DH; ++kk) {
        const float4 a0 = *reinterpret_cast<const float4 *>(am + kk * DH + m0);
        const float4 a1 = *reinterpret_cast<const float4 *>(am + kk * DH + 64 + m0);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float sv = s1[(i0 + r) * FS_LD + kk];
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(sv, av[c], acc[r][c]);
        }
    }
    float *dst = p.final_state + ((size_t)slot * p.Hv + h) * (DH * DH);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const size_t row = (size_t)(i0 + r) * DH;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int m = m0 + 64 * half;
            const float4 bb = *reinterpret_cast<const float4 *>(Bm + row + m);
            *reinterpret_cast<float4 *>(dst + row + m) =
                make_float4(acc[r][4 * half] + bb.x, acc[r][4 * half + 1] + bb.y, acc[r][4 * half + 2] + bb.z,
                            acc[r][4 * half + 3] + bb.w);
        }
    }
}

int num_sms() { return current_device_sms(); }

template <typename TIO>
cudaError_t launch_io(const ForwardParams &p, int min_len, bool split, uint8_t *ws, cudaStream_t stream) {
    CUtensorMap mq{}, mk{}, mv{};
    if (sizeof(TIO) == 2 && p.T > 0) {  // (no tokens: no chunk reads q, k or v)
        // q, k: 64-token x 64-feature boxes in the 128-byte swizzle of the MMA operand tiles;
        // v: 64-token x 128-feature rows as they are
        if (!encode_rows_f16(&mq, p.q, (long long)p.Hk * p.dk, p.q_stride, p.T, 64, CH, true) ||
            !encode_rows_f16(&mk, p.k, (long long)p.Hk * p.dk, p.k_stride, p.T, 64, CH, true) ||
            !encode_rows_f16(&mv, p.v, (long long)p.Hv * p.dv, p.v_stride, p.T, DH, CH, false))
            return cudaErrorInvalidValue;
    }
    int32_t *hdr = reinterpret_cast<int32_t *>(ws);
    const long long maxch = max_chunks(p.B, p.T);
    uint8_t *krec = ws + header_bytes(p.B);
    uint8_t *vrec = krec + (size_t)maxch * p.Hk * KREC_BYTES;
    float *split_states = reinterpret_cast<float *>(vrec + (size_t)maxch * p.Hv * VREC_BYTES);
    // the split plan's identity run needs dk = dv; it is built for 128
    const long long nsplit = split && p.dk == DH && p.dv == DH ? max_split(p.B, p.T) : 0;
    TIO *oid = reinterpret_cast<TIO *>(reinterpret_cast<uint8_t *>(split_states) +
                                       (size_t)nsplit * 3 * p.Hv * STATE_BYTES);
    const long long oid_rows = max_split_rows(p.T);
    cudaError_t e = launch_dependent(wy_plan_kernel, dim3(1), dim3(PLAN_NT), 0, stream, p.cu, p.dense_S, p.B, p.T,
                                     min_len, nsplit > 0, p.cap, hdr, p.status);
    if (e != cudaSuccess) return e;
    const long long prep_ctas = maxch * p.Hk;
    if (prep_ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const bool pad = p.dk != DH || p.dv != DH;
    auto prep = pad ? wy_prep_kernel<TIO, true> : wy_prep_kernel<TIO, false>;
    e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
    if (e != cudaSuccess) return e;
    if (prep_ctas > 0) e = launch_dependent(prep, dim3((unsigned)prep_ctas), dim3(PT), PREP_SMEM, stream, p, hdr, krec, vrec, mq, mk);
    if (e != cudaSuccess) return e;
    auto scan = pad ? wy_scan_kernel<TIO, false, true>
                    : (nsplit > 0 ? wy_scan_kernel<TIO, true, false> : wy_scan_kernel<TIO, false, false>);
    e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, SCAN_SMEM);
    if (e != cudaSuccess) return e;
    const long long chains = (long long)p.B * p.Hv * (nsplit > 0 ? 3 : 1);
    const int grid = (int)(chains < num_sms() ? chains : num_sms());
    // outputs: fp16 chunks go out as 64-token x 128-feature tensor stores when the maps encode
    // (the identity runs of split sequences write their rows of the workspace buffer)
    CUtensorMap mo{}, moi{};
    const int out_tma =
        sizeof(TIO) == 2 &&
        encode_rows_f16(&mo, p.out, (long long)p.Hv * p.dv, (long long)p.Hv * p.dv, p.T, p.dv, CH, false) &&
        (nsplit == 0 || encode_rows_f16(&moi, oid, (long long)p.Hv * DH, (long long)p.Hv * DH, (int)oid_rows, DH,
                                        CH, false));
    e = launch_dependent(scan, dim3(grid), dim3(NT), SCAN_SMEM, stream, p, hdr, krec, vrec, split_states, oid, mv, mo,
                         moi, out_tma);
    if (e != cudaSuccess || nsplit == 0) return e;
    // split sequences: outputs of the second segments, then their final states
    CUtensorMap moa{}, mout{};
    const int oc_tma =
        sizeof(TIO) == 2 &&
        encode_rows_f16(&moa, oid, (long long)p.Hv * DH, (long long)p.Hv * DH, (int)oid_rows, 64, OC_ROWS, true) &&
        encode_rows_f16(&mout, p.out, (long long)p.Hv * DH, (long long)p.Hv * DH, p.T, 64, OC_ROWS, true);
    auto corr = wy_out_correction_kernel<TIO>;
    e = cudaFuncSetAttribute(corr, cudaFuncAttributeMaxDynamicSharedMemorySize, OC_SMEM);
    if (e != cudaSuccess) return e;
    e = launch_dependent(corr, dim3(2 * num_sms()), dim3(OC_NT), OC_SMEM, stream, p, hdr, split_states, oid, moa, mout,
                         oc_tma);
    if (e != cudaSuccess || !p.final_state) return e;
    e = cudaFuncSetAttribute(wy_split_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FS_SMEM);
    if (e != cudaSuccess) return e;
    return launch_dependent(wy_split_final_kernel, dim3((unsigned)(nsplit * p.Hv)), dim3(FS_NT), FS_SMEM, stream, p,
                            hdr, split_states);
}

}  // namespace

bool chunked_wy_supported(int dk, int dv) {
    auto ok = [](int d) { return d == 32 || d == 64 || d == DH; };
    return ok(dk) && ok(dv);
}
bool chunked_wy_splits(int dk, int dv) { return dk == DH && dv == DH; }

size_t chunked_wy_workspace_bytes(int B, int T, int Hk, int Hv, bool split, int io_bytes) {
    const long long maxch = max_chunks(B, T);
    size_t n = header_bytes(B) + (size_t)maxch * ((size_t)Hk * KREC_BYTES + (size_t)Hv * VREC_BYTES);
    if (split && max_split(B, T) > 0)
        n += (size_t)max_split(B, T) * 3 * Hv * STATE_BYTES + (size_t)max_split_rows(T) * Hv * DH * io_bytes;
    return n;
}

cudaError_t launch_chunked_wy(const ForwardParams &p, int min_len, bool split, void *workspace,
                              cudaStream_t stream) {
    if (p.B == 0) return cudaSuccess;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    return p.io_f16 ? launch_io<__half>(p, min_len, split, ws, stream)
                    : launch_io<float>(p, min_len, split, ws, stream);
}

}  // namespace gdn
