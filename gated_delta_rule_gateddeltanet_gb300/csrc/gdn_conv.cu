// Packed depthwise causal convolution with carried state (and SiLU), its
// compact value capture, and replay of an accepted prefix of captured values.
//
// Source: "[CUDA] Add compact GatedDeltaNet operator", embedded commit "Add
// compact VarlenCausalConv state updates" (Description, Motivation): packed
// token-major inputs [num_tokens, channels], a per-request state of the
// kernel_size - 1 preceding inputs per channel, three outputs [output,
// final_state, state_update] where state_update holds only the appended
// values [batch, state_update_capacity, channels], bounded by an optional
// per-request capture_count; "Add GatedDeltaNet evaluation export for Qwen
// hybrid models" (Copilot overview): fused depthwise conv1d + SiLU + carried
// state.
//
//   y[t, c] = silu(bias[c] + sum_{j<K} w[c, j] x_ext[t - (K-1) + j, c])
// where x_ext is the sequence's state (oldest first) followed by its tokens.
//
// The path is HBM-bound (K multiply-adds per element moved), so the kernels
// are laid out for bandwidth: a thread owns 4 channels (an 8- or 16-byte
// vector) and a CTA a block of consecutive packed tokens, so every load and
// store of x, y and the capture is coalesced across the warp.  Each thread
// issues the loads of GROUP tokens before computing any of them, so several
// loads per thread are in flight (registers stay low enough for 8 CTAs per
// SM).  Token blocks
// are independent: the K-1 inputs before a block come from x itself or, at a
// sequence start, from the state.  The state is therefore only read by the
// conv kernel; a second small kernel rolls each sequence's state forward
// afterwards (same thread reads then writes), so updating the state in place
// is race-free.  Short sequences (a max_seqlen hint of at most SHORT_MAX) run
// conv_short_kernel instead, in which a thread carries whole sequences.
#include <type_traits>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;

// tokens whose loads are issued together
template <typename T>
__host__ __device__ constexpr int group_of() { return 4; }

// A thread's 4 channels: one 8-byte (fp16) or 16-byte (fp32) vector.
template <typename T>
struct Vec {
    static constexpr int N = 4;
    using Raw = typename std::conditional<sizeof(T) == 2, uint2, uint4>::type;
};

template <typename T>
__device__ __forceinline__ typename Vec<T>::Raw load_raw(const T *p) {
    return __ldg(reinterpret_cast<const typename Vec<T>::Raw *>(p));  // read-only path: x is never written here
}

template <typename T>
__device__ __forceinline__ void unpack(const typename Vec<T>::Raw &raw, float (&v)[4]) {
    if constexpr (sizeof(T) == 2) {  // two conversions of two halves each
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
        const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = to_f32(e[i]);
    }
}

template <typename T>
__device__ __forceinline__ void load_vec(const T *p, float (&v)[4]) {
    unpack<T>(load_raw<T>(p), v);
}

template <typename T>
__device__ __forceinline__ void store_vec(T *p, const float (&v)[4]) {
    typename Vec<T>::Raw raw;
    if constexpr (sizeof(T) == 2) {  // two round-to-nearest conversions of two floats each
        const __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
        raw.x = *reinterpret_cast<const uint32_t *>(&a);
        raw.y = *reinterpret_cast<const uint32_t *>(&b);
    } else {
        T *e = reinterpret_cast<T *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) e[i] = from_f32<T>(v[i]);
    }
    *reinterpret_cast<typename Vec<T>::Raw *>(p) = raw;
}

// x * sigmoid(x) with the fast exponential and divide intrinsics: the conv
// is bound by instruction issue, and the IEEE forms cost ~5x more per element.
// For very negative x the denominator overflows and the quotient is 0.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// The same through sigmoid(x) = (1 + tanh(x / 2)) / 2 with the hardware tanh
// (one special-function operation instead of two).  Its relative error (about
// 2^-11) is below the fp16 output rounding's, so only fp16 I/O uses it.
__device__ __forceinline__ float silu_tanh(float x) {
    float t;
    const float h = 0.5f * x;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

// One token's outputs for a thread's 4 channels: bias + the K taps over the
// window (oldest first) and the token itself, then SiLU.  Every kernel that
// produces outputs calls this, so the launch shape chosen for a batch never
// changes a bit of the results.
template <typename T, int K>
__device__ __forceinline__ void conv_point(const float (&w)[4][K], const float (&bias)[4], const float (&win)[K - 1][4],
                                           const float (&xt)[4], int silu_on, float (&yv)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float acc = bias[i];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) acc = fmaf(w[i][j], win[j][i], acc);
        acc = fmaf(w[i][K - 1], xt[i], acc);
        yv[i] = silu_on ? (sizeof(T) == 2 ? silu_tanh(acc) : silu(acc)) : acc;
    }
}

// The window after token xt: entries move one place older, xt becomes the newest.
template <int K>
__device__ __forceinline__ void window_push(float (&win)[K - 1][4], const float (&xt)[4]) {
#pragma unroll
    for (int j = 0; j + 1 < K - 1; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) win[j][i] = win[j + 1][i];
#pragma unroll
    for (int i = 0; i < 4; ++i) win[K - 2][i] = xt[i];
}

// A thread's block of the state: 4 channels x (K-1) entries, contiguous, moved
// as 8-byte (fp16) or 16-byte (fp32) words.
template <typename T, int K>
struct StateBlock {
    using Word = typename Vec<T>::Raw;
    static constexpr int WORDS = (K - 1) * 4 * (int)sizeof(T) / (int)sizeof(Word);
    union {
        Word w[WORDS];
        T e[(K - 1) * 4];
    };
    __device__ __forceinline__ void load(const T *p) {
#pragma unroll
        for (int i = 0; i < WORDS; ++i) w[i] = reinterpret_cast<const Word *>(p)[i];
    }
    __device__ __forceinline__ void store(T *p) const {
#pragma unroll
        for (int i = 0; i < WORDS; ++i) reinterpret_cast<Word *>(p)[i] = w[i];
    }
    __device__ __forceinline__ T &at(int channel, int j) { return e[channel * (K - 1) + j]; }
};

constexpr int CU_SMEM = 4096;  // cu_seqlens entries staged in shared memory for the search

// Sequence holding packed token t: the largest b with cu[b] <= t.
__device__ __forceinline__ int seq_of(const int32_t *cu, int B, int t) {
    int lo = 0, hi = B;  // cu[lo] <= t < cu[hi] for a valid packing
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

template <typename T, int K>
__global__ void __launch_bounds__(NT, sizeof(T) == 2 ? 4 : 3) conv_kernel(const ConvParams p) {
    dependent_prologue();
    constexpr int V = Vec<T>::N;
    constexpr int GROUP = group_of<T>();
    const int cgroups = p.C / V;
    const int cg = blockIdx.y * NT + threadIdx.x;  // channel group of this thread
    const int t_begin = blockIdx.x * p.tokens_per_cta;
    const int t_end = min(t_begin + p.tokens_per_cta, p.T);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && (p.cu[0] != 0 || p.cu[p.B] != p.T))
        flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
    // the first tokens' loads go out before anything else, so they overlap the search
    const T *xg0 = static_cast<const T *>(p.x);
    const int c0_early = (blockIdx.y * NT + threadIdx.x) * Vec<T>::N;
    typename Vec<T>::Raw raw[GROUP];
    if (c0_early < p.C) {
#pragma unroll
        for (int g = 0; g < GROUP; ++g)
            if (t_begin + g < t_end) raw[g] = load_raw<T>(xg0 + (long long)(t_begin + g) * p.x_stride + c0_early);
    }
    __shared__ int32_t cu_s[CU_SMEM];
    const bool cu_staged = p.B + 1 <= CU_SMEM;
    if (cu_staged)
        for (int i = threadIdx.x; i <= p.B; i += NT) cu_s[i] = p.cu[i];
    __syncthreads();
    if (cg >= cgroups || t_begin >= t_end) return;
    const int c0 = cg * V;
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.out);
    T *vals = static_cast<T *>(p.values);
    const T *st_in = static_cast<const T *>(p.state_in);
    T *st_out = static_cast<T *>(p.state_out);

    float w[V][K], bias[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
#pragma unroll
        for (int j = 0; j < K; ++j) w[i][j] = p.w[(long long)(c0 + i) * K + j];
        bias[i] = p.bias ? p.bias[c0 + i] : 0.f;
    }

    int b = seq_of(cu_staged ? cu_s : p.cu, p.B, t_begin);
    int bos = 0, eos = 0, slot = 0, ncap = 0;
    bool ok = false;
    float win[K - 1][V];  // inputs at t-(K-1) .. t-1 (oldest first)
    const int32_t *cu = cu_staged ? cu_s : p.cu;
    auto enter = [&](int t) {  // (re)build the window for token t of sequence b
        bos = cu[b];
        eos = cu[b + 1];
        slot = p.slots ? p.slots[b] : b;
        ok = bos >= 0 && eos >= bos && eos <= p.T && slot >= 0 && slot < p.num_slots;
        ncap = p.cap;
        if (p.capture_count) {
            const int cc = p.capture_count[b];
            if (cc < 0 || cc > p.cap) {
                if (threadIdx.x == 0 && t == bos) flag_error(p.status, GDN_DEVERR_CAPTURE_COUNT);
                ncap = 0;
            } else {
                ncap = cc;
            }
        }
        if (!ok) {
            if (threadIdx.x == 0 && t == bos) {
                if (slot < 0 || slot >= p.num_slots) flag_error(p.status, GDN_DEVERR_STATE_SLOT);
                else flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
            }
            return;
        }
        StateBlock<T, K> sb;
        const bool need_state = t - (K - 1) < bos && st_in;
        if (need_state) sb.load(st_in + ((long long)slot * p.C + c0) * (K - 1));
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            const int pos = t - (K - 1) + j;  // packed position of window entry j
            float v[V];
            if (pos >= bos) {
                load_vec<T>(x + (long long)pos * p.x_stride + c0, v);
            } else if (need_state) {
                const int sj = (K - 1) - (bos - pos);  // state index, oldest first
#pragma unroll
                for (int i = 0; i < V; ++i) {  // select with constant indices: keeps sb in registers
                    float e = 0.f;
#pragma unroll
                    for (int q = 0; q < K - 1; ++q)
                        if (q == sj) e = to_f32(sb.at(i, q));
                    v[i] = e;
                }
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < V; ++i) win[j][i] = v[i];
        }
    };
    while (b < p.B && cu[b + 1] <= t_begin) ++b;  // skip empty sequences
    if (b >= p.B) return;
    enter(t_begin);
    for (int tg = t_begin; tg < t_end; tg += GROUP) {
        if (tg != t_begin) {
#pragma unroll
            for (int g = 0; g < GROUP; ++g)
                if (tg + g < t_end) raw[g] = load_raw<T>(x + (long long)(tg + g) * p.x_stride + c0);
        }
        // Interior group: every token inside the current sequence, none its last
        // one, none captured -- straight-line code without the per-token checks.
        // (The condition is the same for every thread of the CTA.)
        if (ok && tg >= bos && tg + GROUP < eos && tg + GROUP <= t_end && (!vals || tg - bos >= ncap)) {
            T *yp = y + (long long)tg * p.C + c0;
#pragma unroll
            for (int g = 0; g < GROUP; ++g) {
                float xt[V], yv[V];
                unpack<T>(raw[g], xt);
                conv_point<T, K>(w, bias, win, xt, p.silu, yv);
                store_vec<T>(yp, yv);
                yp += p.C;
                window_push<K>(win, xt);
            }
            continue;
        }
#pragma unroll
        for (int g = 0; g < GROUP; ++g) {
            const int t = tg + g;
            if (t >= t_end) break;
            while (t >= eos && b + 1 < p.B) {  // next sequence starts here
                ++b;
                enter(t);
            }
            if (!ok || t >= eos) continue;
            float xt[V];
            unpack<T>(raw[g], xt);
            float yv[V];
            conv_point<T, K>(w, bias, win, xt, p.silu, yv);
            store_vec<T>(y + (long long)t * p.C + c0, yv);
            const int tl = t - bos;
            if (vals && tl < ncap) store_vec<T>(vals + ((long long)b * p.cap + tl) * p.C + c0, xt);
            window_push<K>(win, xt);
            // A sequence that lies wholly inside this token block is read and
            // written by this thread only: its new state is the window now.
            if (t == eos - 1 && bos >= t_begin) {
                StateBlock<T, K> sb;
#pragma unroll
                for (int i = 0; i < V; ++i)
#pragma unroll
                    for (int j = 0; j < K - 1; ++j) sb.at(i, j) = from_f32<T>(win[j][i]);
                sb.store(st_out + ((long long)slot * p.C + c0) * (K - 1));
            }
        }
    }
}

// new state = the last K-1 entries of (old state, the sequence's tokens)
template <typename T, int K>
__global__ void __launch_bounds__(NT) conv_state_kernel(const ConvParams p) {
    dependent_prologue();
    constexpr int V = Vec<T>::N;
    const int cg = blockIdx.x * NT + threadIdx.x;
    const int b = blockIdx.y;
    if (cg >= p.C / V) return;
    const int bos = p.cu[b], eos = p.cu[b + 1];
    const int slot = p.slots ? p.slots[b] : b;
    if (bos < 0 || eos < bos || eos > p.T || slot < 0 || slot >= p.num_slots) {
        // flagged here as well: conv_kernel only sees sequences that own tokens
        if (blockIdx.x == 0 && threadIdx.x == 0)
            flag_error(p.status, slot < 0 || slot >= p.num_slots ? GDN_DEVERR_STATE_SLOT : GDN_DEVERR_CU_SEQLENS);
        return;
    }
    if (eos > bos && bos / p.tokens_per_cta == (eos - 1) / p.tokens_per_cta) return;  // written by conv_kernel
    const int c0 = cg * V;
    const T *x = static_cast<const T *>(p.x);
    const T *st_in = static_cast<const T *>(p.state_in);
    T *st_out = static_cast<T *>(p.state_out);
    const int len = eos - bos;
    T nw[V][K - 1];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int from_end = (K - 1) - j;  // entry j of the new state is the from_end-th last input
        if (from_end <= len) {
            const T *xp = x + (long long)(eos - from_end) * p.x_stride + c0;
            const typename Vec<T>::Raw raw = load_raw<T>(xp);
            const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
            for (int i = 0; i < V; ++i) nw[i][j] = e[i];
        } else {
            const int sj = j + len;  // shifted left by len within the old state
#pragma unroll
            for (int i = 0; i < V; ++i)
                nw[i][j] = st_in ? st_in[((long long)slot * p.C + c0 + i) * (K - 1) + sj] : from_f32<T>(0.f);
        }
    }
#pragma unroll
    for (int i = 0; i < V; ++i)
#pragma unroll
        for (int j = 0; j < K - 1; ++j) st_out[((long long)slot * p.C + c0 + i) * (K - 1) + j] = nw[i][j];
}

// Short sequences (decode steps, speculative drafts): a max_seqlen hint of
// 1 .. SHORT_MAX.  A thread owns 4 channels of SHORT_SEQS consecutive
// sequences and runs each sequence's tokens itself, so its work is two
// dependent rounds of loads: the sequence bounds, slots, capture counts and
// weights, then the states and the first SHORT_PREFETCH input rows of its
// sequences together.  The token-block kernel instead resolves each token's
// sequence through a search and loads the slot and then the state per
// sequence, one after the other (five dependent rounds for two 1-token
// sequences per CTA).  Each thread writes its sequences' new states itself,
// so there is no state-rolling launch.  A sequence longer than the hint
// (a caller error) still gets exact results: its remaining rows are loaded
// SHORT_PREFETCH at a time.
constexpr int SHORT_MAX = 8;       // longest hint served by conv_short_kernel
constexpr int SHORT_NT = 128;      // threads per CTA
constexpr int SHORT_SEQS = 2;      // sequences per thread (keeps a 64 x 10240 decode step in one wave)
constexpr int SHORT_PREFETCH = 4;  // input rows per sequence loaded with the state

template <typename T, int K>
__global__ void __launch_bounds__(SHORT_NT) conv_short_kernel(const ConvParams p) {
    dependent_prologue();
    constexpr int V = Vec<T>::N;
    using Raw = typename Vec<T>::Raw;
    const int cg = blockIdx.x * SHORT_NT + threadIdx.x;
    const int b0 = blockIdx.y * SHORT_SEQS;
    const bool leader = blockIdx.x == 0 && threadIdx.x == 0;  // raises the flags of its sequences
    if (leader && blockIdx.y == 0 && (p.cu[0] != 0 || p.cu[p.B] != p.T)) flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
    if (cg >= p.C / V) return;
    const int c0 = cg * V;
    const T *x = static_cast<const T *>(p.x);
    T *y = static_cast<T *>(p.out);
    T *vals = static_cast<T *>(p.values);
    const T *st_in = static_cast<const T *>(p.state_in);
    T *st_out = static_cast<T *>(p.state_out);

    // ---- first round: what each sequence is, and the weights
    int bos[SHORT_SEQS], eos[SHORT_SEQS], slot[SHORT_SEQS], cc[SHORT_SEQS];
#pragma unroll
    for (int u = 0; u < SHORT_SEQS; ++u) {
        const int b = b0 + u;
        bos[u] = eos[u] = slot[u] = 0;
        cc[u] = p.cap;
        if (b < p.B) {
            bos[u] = p.cu[b];
            eos[u] = p.cu[b + 1];
            slot[u] = p.slots ? p.slots[b] : b;
            if (p.capture_count) cc[u] = p.capture_count[b];
        }
    }
    float w[V][K], bias[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
#pragma unroll
        for (int j = 0; j < K; ++j) w[i][j] = p.w[(long long)(c0 + i) * K + j];
        bias[i] = p.bias ? p.bias[c0 + i] : 0.f;
    }
    bool ok[SHORT_SEQS];
    int len[SHORT_SEQS], ncap[SHORT_SEQS];
#pragma unroll
    for (int u = 0; u < SHORT_SEQS; ++u) {
        const int b = b0 + u;
        const bool slot_ok = slot[u] >= 0 && slot[u] < p.num_slots;
        ok[u] = b < p.B && bos[u] >= 0 && eos[u] >= bos[u] && eos[u] <= p.T && slot_ok;
        if (b < p.B && !ok[u] && leader)
            flag_error(p.status, slot_ok ? GDN_DEVERR_CU_SEQLENS : GDN_DEVERR_STATE_SLOT);
        ncap[u] = cc[u];
        if (p.capture_count && (cc[u] < 0 || cc[u] > p.cap)) {
            if (ok[u] && leader) flag_error(p.status, GDN_DEVERR_CAPTURE_COUNT);
            ncap[u] = 0;
        }
        len[u] = ok[u] ? eos[u] - bos[u] : 0;
    }

    // ---- second round: the states and the first input rows of every sequence
    StateBlock<T, K> sb[SHORT_SEQS];
    Raw raw[SHORT_SEQS][SHORT_PREFETCH];
#pragma unroll
    for (int u = 0; u < SHORT_SEQS; ++u) {
        if (ok[u] && st_in) sb[u].load(st_in + ((long long)slot[u] * p.C + c0) * (K - 1));
#pragma unroll
        for (int g = 0; g < SHORT_PREFETCH; ++g)
            if (g < len[u]) raw[u][g] = load_raw<T>(x + (long long)(bos[u] + g) * p.x_stride + c0);
    }

#pragma unroll
    for (int u = 0; u < SHORT_SEQS; ++u) {
        if (!ok[u]) continue;
        const int b = b0 + u;
        float win[K - 1][V];
#pragma unroll
        for (int j = 0; j < K - 1; ++j)
#pragma unroll
            for (int i = 0; i < V; ++i) win[j][i] = st_in ? to_f32(sb[u].at(i, j)) : 0.f;
        for (int t0 = 0; t0 < len[u]; t0 += SHORT_PREFETCH) {
            if (t0 > 0) {  // only past the prefetched rows (a sequence longer than the hint)
#pragma unroll
                for (int g = 0; g < SHORT_PREFETCH; ++g)
                    if (t0 + g < len[u]) raw[u][g] = load_raw<T>(x + (long long)(bos[u] + t0 + g) * p.x_stride + c0);
            }
#pragma unroll
            for (int g = 0; g < SHORT_PREFETCH; ++g) {
                const int tl = t0 + g;
                if (tl >= len[u]) break;
                float xt[V], yv[V];
                unpack<T>(raw[u][g], xt);
                conv_point<T, K>(w, bias, win, xt, p.silu, yv);
                store_vec<T>(y + (long long)(bos[u] + tl) * p.C + c0, yv);
                if (vals && tl < ncap[u]) store_vec<T>(vals + ((long long)b * p.cap + tl) * p.C + c0, xt);
                window_push<K>(win, xt);
            }
        }
        // the new state is the window; an empty sequence keeps its state (copied when
        // the state is not updated in place, zero when there is no initial state)
        if (len[u] > 0 || st_out != st_in) {
            StateBlock<T, K> nb;
#pragma unroll
            for (int i = 0; i < V; ++i)
#pragma unroll
                for (int j = 0; j < K - 1; ++j) nb.at(i, j) = from_f32<T>(win[j][i]);
            nb.store(st_out + ((long long)slot[u] * p.C + c0) * (K - 1));
        }
    }
}

// Replay: state[dst] = the last K-1 entries of (state[src], values[j, 0..n))
template <typename T, int K>
__global__ void __launch_bounds__(NT) conv_replay_kernel(const ConvReplayParams p) {
    dependent_prologue();
    constexpr int V = Vec<T>::N;
    const int cg = blockIdx.x * NT + threadIdx.x;
    const int j = blockIdx.y;
    const int src = p.src[j], dst = p.dst[j], n = p.n[j];
    const bool leader = blockIdx.x == 0 && threadIdx.x == 0;
    if (src < 0 || src >= p.num_slots || dst < 0 || dst >= p.num_slots) {
        if (leader) flag_error(p.status, GDN_DEVERR_REPLAY_SLOT);
        return;
    }
    if (n < 0 || n > p.cap) {
        if (leader) flag_error(p.status, GDN_DEVERR_ACCEPT_LEN);
        return;
    }
    if (cg >= p.C / V || (src == dst && n == 0)) return;
    const int c0 = cg * V;
    T *states = static_cast<T *>(p.states);
    const T *vals = static_cast<const T *>(p.values);
    T nw[V][K - 1];
#pragma unroll
    for (int e = 0; e < K - 1; ++e) {
        const int from_end = (K - 1) - e;
        if (from_end <= n) {
            const typename Vec<T>::Raw raw = load_raw<T>(vals + ((long long)j * p.cap + n - from_end) * p.C + c0);
            const T *el = reinterpret_cast<const T *>(&raw);
#pragma unroll
            for (int i = 0; i < V; ++i) nw[i][e] = el[i];
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) nw[i][e] = states[((long long)src * p.C + c0 + i) * (K - 1) + e + n];
        }
    }
#pragma unroll
    for (int i = 0; i < V; ++i)
#pragma unroll
        for (int e = 0; e < K - 1; ++e) states[((long long)dst * p.C + c0 + i) * (K - 1) + e] = nw[i][e];
}

template <typename T, int K>
cudaError_t launch_conv_k(const ConvParams &p, cudaStream_t stream) {
    constexpr int V = Vec<T>::N;
    const int cgroups = p.C / V;
    const long long seq_blocks = ((long long)p.B + SHORT_SEQS - 1) / SHORT_SEQS;
    if (p.max_len_hint >= 1 && p.max_len_hint <= SHORT_MAX && seq_blocks <= 65535) {
        dim3 grid((unsigned)((cgroups + SHORT_NT - 1) / SHORT_NT), (unsigned)seq_blocks);
        // a dependent launch (5.39 vs 5.57 us for the 64 x 10240 decode step); the
        // token-block kernels below measured the other way
        return launch_dependent(conv_short_kernel<T, K>, grid, dim3(SHORT_NT), 0, stream, p);
    }
    const int cblocks = (cgroups + NT - 1) / NT;
    if (p.T > 0) {
        dim3 grid((unsigned)((p.T + p.tokens_per_cta - 1) / p.tokens_per_cta), (unsigned)cblocks);
        // plain launches: as a dependent launch this kernel's one-wave decode step measured
        // slower (8.8 vs 7.4 us)
        conv_kernel<T, K><<<grid, NT, 0, stream>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.skip_state_kernel) return cudaSuccess;  // every sequence is whole inside one token block, state in place
    dim3 g2((unsigned)cblocks, (unsigned)p.B);
    conv_state_kernel<T, K><<<g2, NT, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename T, int K>
cudaError_t launch_replay_k(const ConvReplayParams &p, cudaStream_t stream) {
    constexpr int V = Vec<T>::N;
    dim3 grid((unsigned)((p.C / V + NT - 1) / NT), (unsigned)p.R);
    conv_replay_kernel<T, K><<<grid, NT, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_conv_t(const ConvParams &p, cudaStream_t s) {
    switch (p.K) {
        case 2: return launch_conv_k<T, 2>(p, s);
        case 3: return launch_conv_k<T, 3>(p, s);
        default: return launch_conv_k<T, 4>(p, s);
    }
}

template <typename T>
cudaError_t launch_replay_t(const ConvReplayParams &p, cudaStream_t s) {
    switch (p.K) {
        case 2: return launch_replay_k<T, 2>(p, s);
        case 3: return launch_replay_k<T, 3>(p, s);
        default: return launch_replay_k<T, 4>(p, s);
    }
}

}  // namespace

cudaError_t launch_conv(const ConvParams &p, cudaStream_t stream) {
    if (p.B == 0) return cudaSuccess;
    return p.io_f16 ? launch_conv_t<__half>(p, stream) : launch_conv_t<float>(p, stream);
}

cudaError_t launch_conv_replay(const ConvReplayParams &p, cudaStream_t stream) {
    if (p.R == 0) return cudaSuccess;
    return p.io_f16 ? launch_replay_t<__half>(p, stream) : launch_replay_t<float>(p, stream);
}

}  // namespace gdn
