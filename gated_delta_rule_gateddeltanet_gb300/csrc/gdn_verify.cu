// Short spans at dk = dv = 128 when some span of the batch has several tokens
// (speculative verification of draft tokens, short prefill pieces), on the
// 5th-generation tensor cores.
//
// Operator: "[CUDA] Add compact GatedDeltaNet operator" (Description) -- the
// recurrent path for short spans with the compact state_update capsule; the
// speculative step of "Replay compact fixed state for hybrid decoding"
// (Summary / Key Changes) verifies a few draft tokens per request with it
// every decoding step.
//
// Work item: one (sequence, value head), i.e. its whole 128 x 128 FP32 state
// (64 KiB), held in shared memory in the 128-byte swizzled layout the tensor
// copies give.  Two CTAs of 8 warps per SM, each persistent over a
// contiguous range of items (consecutive value heads of one key head reuse
// the key-side staging); while one CTA waits for its next item's copies the
// other computes.  CTAs with fewer items than the fullest ones start a few
// microseconds later, so that the first copies do not all land in one burst,
// and without a final state an item's successor is copied in as soon as its
// last products have read the rows.  For the row-local work thread (warp w, lane l) owns state
// row r = 32 (w % 4) + l -- the tensor-memory lane its warp can reach -- and
// half w / 4 of the row's columns, as 16 float4 chunks at columns
// 32 j + 16 (w / 4) + 4 m (j, m < 4).
//
// Tokens go four at a time through the closed form of a 4-token group (the
// token-by-token recurrence unrolled; G_t = g_0 .. g_t, r(t, s) = g_{s+1} .. g_t
// formed as products, n the group's last token):
//     P_t = S0 k_t,  Q_t = S0 q_t
//     u_t = beta_t v_t - beta_t G_t P_t - sum_{s<t} beta_t r(t,s) (k_s.k_t) u_s
//     o_t = scale (G_t Q_t + sum_{s<=t} r(t,s) (k_s.q_t) u_s)
//     S   = G_n S0 + sum_t r(n,t) u_t k_t^T
// The dense part, the eight dot products per row, is one tcgen05 product with
// an FP32 accumulator in tensor memory:
//   D1 [128 x 16] = S0 [128 x 128] . [k_hi k_lo q_hi q_lo]^T   (kind::tf32)
// issued twice into the same accumulator: with A = the rows in shared memory,
// which the tensor core reads as TF32 (the low 13 mantissa bits dropped), and
// with A = their exact remainders, written by the threads into tensor memory
// (the A operand of a tcgen05 product may sit there).  k_hi is k rounded to
// TF32 and k_lo = k - k_hi, so P_t = D1[t] + D1[4 + t] carries all four
// partial products of the split (about 2^-21 relative error, FP32-level).
// The rest runs on the CUDA cores: u_t and o_t on the thread that owns the
// row (both threads of a row form u), then the rank-4 update
// S = G_n S0 + sum_t r(n,t) u_t k_t^T in FP32 with warp w over rows
// 16 w .. 16 w + 15 and lane l over columns 4 l .. 4 l + 3, so that a row of
// final state leaves as one 512-byte store; the rows of a later group of the
// same span go back in place instead.
//
// One-token and empty spans in the same batch run the decode kernel's
// CUDA-core arithmetic in the same order, so a decode request gives the same
// bits in any batch: the decode kernel's eight lanes per row become four
// "virtual lanes" in each of the row's two threads, whose partial dot
// products meet through the accumulator's columns before the same butterfly
// sum; their rows go back by tensor stores.
//
// Every wait is bounded; on time-out the CTA flags GDN_DEVERR_TIMEOUT,
// drains its copies and products, frees its tensor memory and stops.
#include <algorithm>
#include <cstring>

#include "chunk_tiles.cuh"
#include "gdn_internal.cuh"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int D = 128;     // dk = dv
constexpr int TB = 4;      // tokens per group
constexpr int NTV = 256;   // threads per CTA (two CTAs per SM)
constexpr int ISSUER_HI = 128;  // the threads that issue the tensor-core products: rows (warp 4, lane 0)
constexpr int ISSUER_LO = 160;  // and remainders (warp 5, lane 0)
constexpr int STAGER = 32;      // the thread that issues the q, k, v copies (warp 1, lane 0)
constexpr float EPS = 1e-6f;
constexpr long long WAIT_LIMIT = 4000000000LL;  // SM cycles (~2 s)

// Tensor-memory columns (one allocation of 256 per CTA): the TF32 remainders of
// the rows and the two accumulators of the dot products (rows, remainders).
constexpr uint32_t TM_LO = 0, TM_D1 = 128, TM_D1L = 144, TM_COLS = 256;

constexpr uint32_t TILE = D * D * 4;  // one state: 4 boxes of 128 rows x 128 bytes (128-byte swizzle)

// Dynamic shared memory, offsets from a 1024-byte aligned base: the item's
// rows, the split keys and queries (16 rows x 128, tf32, 4 boxes of 2 KiB), and
// the first group's q, k, v rows (fp16 I/O only: FP32 inputs are read directly).
template <typename TIO>
struct Layout {
    static constexpr bool STAGE = sizeof(TIO) == 2;
    static constexpr uint32_t B1 = TILE;
    static constexpr uint32_t STG = B1 + 8192;
    static constexpr uint32_t DYN = STG + (STAGE ? 3u * TB * D * 2u : 0u) + 1024;  // + alignment slack
};

// Tensor maps of one launch.  Input boxes of the q, k, v rows are 128 fp16
// features wide and TB tokens high; output boxes TB tokens x 64 elements.
struct VMaps {
    CUtensorMap in, fin;      // the state pools, boxes of 128 rows x 32 floats (128-byte swizzle)
    CUtensorMap in3;          // the initial pool, one box of 128 rows x 128 floats as four such tiles
    CUtensorMap out, caps;    // outputs and capsules of full groups
    CUtensorMap q, k, v;      // the first group's q, k, v rows of an item
    int out_ok, stg_ok, in3_ok;
};

struct VItem {
    int b, h, kh, bos, eos;
    int row0;  // first state row of the item in the [slots Hv D, D] view
    bool ok;
};

// Position of an item, advanced one item at a time (no divisions).
struct VCursor {
    int b, h, kh, hr;  // hr = h % r
};

__device__ __forceinline__ void advance(const ForwardParams &p, VCursor &c) {
    if (++c.h == p.Hv) {
        c.h = c.kh = c.hr = 0;
        ++c.b;
    } else if (++c.hr == p.r) {
        c.hr = 0;
        ++c.kh;
    }
}

// The descriptor loads of an item, issued ahead of their use.
struct VRaw {
    int cu0, cu1, slot;
};

__device__ __forceinline__ VRaw load_raw(const ForwardParams &p, int b) {
    VRaw r;
    r.cu0 = seq_start(p.cu, p.dense_S, b);
    r.cu1 = seq_start(p.cu, p.dense_S, b + 1);
    r.slot = p.slots ? p.slots[b] : b;
    return r;
}

// Work item from its descriptor loads; not ok when there is nothing to do (a
// bad descriptor, flagged once, or a span longer than max_len, which the
// chunked kernel owns).
__device__ __forceinline__ VItem make_item(const ForwardParams &p, const VCursor &c, const VRaw &r) {
    VItem it;
    it.b = c.b;
    it.h = c.h;
    it.kh = c.kh;
    it.bos = r.cu0;
    it.eos = r.cu1;
    it.row0 = 0;
    it.ok = false;
    const bool leader = it.h == 0 && threadIdx.x == 0;
    if (p.cu && it.b == 0 && leader && (r.cu0 != 0 || p.cu[p.B] != p.T)) flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
    if (it.bos < 0 || it.eos < it.bos || it.eos > p.T) {
        if (leader) flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
        return it;
    }
    if (it.eos - it.bos > p.max_len || it.eos - it.bos < p.min_len) return it;  // another kernel's
    if (r.slot < 0 || r.slot >= p.num_slots) {
        if (leader) flag_error(p.status, GDN_DEVERR_STATE_SLOT);
        return it;
    }
    it.row0 = (r.slot * p.Hv + it.h) * D;
    it.ok = true;
    return it;
}

__device__ __forceinline__ VItem no_item() {
    VItem it;
    it.b = it.h = it.kh = it.bos = it.eos = it.row0 = 0;
    it.ok = false;
    return it;
}

// Byte offset of 16-byte chunk q (0..7) of row `row` in box j of a state
// buffer (128-byte swizzle: chunk q of row r sits at q ^ (r % 8)).
__device__ __forceinline__ uint32_t chunk_at(int row, int j, int q) {
    return (uint32_t)(j * (D * 128) + row * 128 + ((q ^ (row & 7)) << 4));
}

// TF32 high part of x as the tensor core reads an FP32 operand (the low 13
// mantissa bits dropped), so that x - hi is the exact remainder.
__device__ __forceinline__ float tf32_trunc(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }
// TF32 value nearest to x (for the split keys and queries, whose both parts
// are written explicitly).
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(ct::to_tf32(x)); }

// D1 [128 x 16] = S [128 x 128] . B1^T, B1 rows k_hi(t), k_lo(t), q_hi(t),
// q_lo(t) (t < 4), K-major, 16 K steps of 8, in two parts issued by two threads
// into two accumulators: the rows themselves (shared memory, read as TF32) and
// their remainders (tensor memory).
__device__ __forceinline__ void issue_mma_rows(uint32_t tm, uint32_t rows_base, uint32_t b1_base) {
    constexpr uint32_t idesc = ptx::idesc_tf32_f32(128, 16);
#pragma unroll 4
    for (int s = 0; s < D / 8; ++s) {
        // K step s: 32 bytes into box s / 4 of the rows and of B1
        const uint64_t ad = ptx::sdesc_k_sw128(rows_base + (uint32_t)(s >> 2) * (D * 128u)) + (uint64_t)(2 * (s & 3));
        const uint64_t bd = ptx::sdesc_k_sw128(b1_base + (uint32_t)(s >> 2) * 2048u) + (uint64_t)(2 * (s & 3));
        ptx::mma_tf32_ss(tm + TM_D1, ad, bd, idesc, s != 0);
    }
}

__device__ __forceinline__ void issue_mma_rem(uint32_t tm, uint32_t b1_base) {
    constexpr uint32_t idesc = ptx::idesc_tf32_f32(128, 16);
#pragma unroll 4
    for (int s = 0; s < D / 8; ++s) {
        const uint64_t bd = ptx::sdesc_k_sw128(b1_base + (uint32_t)(s >> 2) * 2048u) + (uint64_t)(2 * (s & 3));
        ptx::mma_tf32_ts(tm + TM_D1L, tm + TM_LO + 8u * s, bd, idesc, s != 0);
    }
}

// Sum over the warp of eight values at once (a halving butterfly: 9 shuffles
// instead of 40); lane l ends with the sum of value (l >> 2) & 7.
__device__ __forceinline__ float warp_sum8(const float (&v)[8]) {
    const int lane = threadIdx.x & 31;
    float a4[4], a2[2];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float send = up ? v[j] : v[j + 4], keep = up ? v[j + 4] : v[j];
            a4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    {
        const bool up = lane & 8;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float send = up ? a4[j] : a4[j + 2], keep = up ? a4[j + 2] : a4[j];
            a2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    const bool up = lane & 4;
    float a1 = (up ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, up ? a2[0] : a2[1], 4);
    a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
    a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
    return a1;
}

// Gate inputs of the first group of an item (lanes 0..3 of warps 0..3:
// token = lane), loaded one item ahead of their use.
struct GateIn {
    float a, b, A, d;
};

__device__ __forceinline__ GateIn load_gates(const ForwardParams &p, const VItem &it) {
    GateIn g = {0.f, 0.f, 0.f, 0.f};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < TB && lane < TB && it.ok && it.bos + lane < it.eos) {
        const long long t = it.bos + lane;
        g.a = p.a[t * p.Hv + it.h];
        g.b = p.b[t * p.Hv + it.h];
        if (p.gate_raw) {
            g.A = p.A_log[it.h];
            g.d = p.dt_bias[it.h];
        }
    }
    return g;
}

template <typename TIO>
__global__ void __launch_bounds__(NTV, 2)
    verify_kernel(const ForwardParams p, int items, const __grid_constant__ VMaps mp) {
    using L = Layout<TIO>;
    dependent_prologue();
    extern __shared__ uint8_t dyn_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    // the group's unit keys and queries (FP32) and their products
    __shared__ __align__(16) float kn_s[TB][D];
    __shared__ __align__(16) float qn_s[TB][D];
    __shared__ float dkk_s[TB][TB], dkq_s[TB][TB];
    __shared__ float g1_s, beta1_s, kq1_s;  // one-token spans: gate, beta, k.q
    // group factors
    __shared__ float bt_s[TB], bG_s[TB], sG_s[TB], eG_s[TB], Gn_s;
    __shared__ float mkk_s[TB][TB], mq_s[TB][TB];
    __shared__ __align__(16) float w_s[D][TB];  // the decayed deltas r(n, t) u_t of every row
    // outputs and deltas of an item's last full group (one tensor-store box per 64 rows)
    __shared__ __align__(128) TIO o_s[2][TB][64];
    __shared__ __align__(128) float u_s[2][TB][64];
    __shared__ __align__(8) uint64_t full_bar;
    __shared__ __align__(8) uint64_t mma_bar;
    __shared__ uint32_t tmem_base;
    // the next item as thread 0 resolved it early (no final state: its copies start
    // once the current item's products have read the rows)
    __shared__ VCursor nx_cur_s;
    __shared__ VRaw nx_seq_s;
    __shared__ VItem nx_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;

    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base, TM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        ptx::mbar_init(&full_bar, 1);
        ptx::mbar_init(&mma_bar, 2);  // one commit per issuing thread
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tm = tmem_base;
    uint8_t *const rows = sm;  // the item's rows, updated in place
    const uint32_t rows_base = ptx::smem_u32(rows), b1_base = ptx::smem_u32(sm + L::B1);
    const TIO *const stq = reinterpret_cast<const TIO *>(sm + L::STG);  // first group's q, k, v rows
    const TIO *const stk = stq + TB * D, *const stv = stq + 2 * TB * D;

    const TIO *qg = static_cast<const TIO *>(p.q);
    const TIO *kg = static_cast<const TIO *>(p.k);
    const TIO *vg = static_cast<const TIO *>(p.v);
    TIO *og = static_cast<TIO *>(p.out);
    const long long ubase = (long long)p.Hv + (long long)p.Hk * D;

    const int first = (int)((long long)blockIdx.x * items / gridDim.x);
    const int stop = (int)((long long)(blockIdx.x + 1) * items / gridDim.x);

    // ---- copies (thread 0): the item's rows and its first group's q, k, v rows
    auto load_bytes = [&](const VItem &it) -> uint32_t {
        if (!it.ok) return 0u;
        return (p.init ? TILE : 0u) + (mp.stg_ok && it.eos > it.bos ? 3u * TB * D * (uint32_t)sizeof(TIO) : 0u);
    };
    // thread 0 arms the barrier and copies the rows, thread STAGER copies the q, k, v rows
    // (a copy may complete before the barrier is armed: its bytes are counted all the same)
    // (with `one`, the caller is thread 0 alone and copies everything)
    auto issue_load = [&](const VItem &it, bool one = false) {
        const uint32_t bytes = load_bytes(it);
        if (!bytes) return;
        if (tid == 0) {
            ptx::mbar_arrive_expect_tx(&full_bar, bytes);
            if (p.init) {
                if (mp.in3_ok) {
                    ptx::tma_load_3d(rows, &mp.in3, 0, it.row0, 0, &full_bar);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) ptx::tma_load_2d(rows + j * (D * 128), &mp.in, 32 * j, it.row0, &full_bar);
                }
            }
        }
        if ((one ? tid == 0 : tid == STAGER) && L::STAGE && mp.stg_ok && it.eos > it.bos) {
            TIO *st = reinterpret_cast<TIO *>(sm + L::STG);
            ptx::tma_load_2d(st, &mp.q, it.kh * D, it.bos, &full_bar);
            ptx::tma_load_2d(st + TB * D, &mp.k, it.kh * D, it.bos, &full_bar);
            ptx::tma_load_2d(st + 2 * TB * D, &mp.v, it.h * D, it.bos, &full_bar);
        }
    };

    // the current item's position and its sequence's descriptor (loaded again only when
    // the position moves to another sequence)
    VCursor cur_c;
    cur_c.b = first / p.Hv;
    cur_c.h = first - cur_c.b * p.Hv;
    cur_c.kh = cur_c.h / p.r;
    cur_c.hr = cur_c.h - cur_c.kh * p.r;
    VRaw seq = load_raw(p, cur_c.b);
    VItem it = first < stop ? make_item(p, cur_c, seq) : no_item();
    bool loaded = load_bytes(it) != 0;
    // CTAs with fewer items than the fullest ones (one item of slack) start their
    // copies about 3 us later: the fullest CTAs then have the memory system to
    // themselves while their first rows arrive, instead of every CTA's first copy
    // landing in one burst (16 x 4 verify: 27.5 vs 29.3 us, 18.4 vs 19.9 writing no
    // final state).  Costs nothing when every CTA has the same number of items, and
    // a CTA whose first item has no work (another kernel's span, or a bad one) does
    // not wait.
    if (it.ok && stop - first < (int)(((long long)items + gridDim.x - 1) / gridDim.x)) __nanosleep(3000);
    issue_load(it);
    GateIn gc = load_gates(p, it);  // this item's first-group gate inputs

    uint32_t full_phase = 0u, mma_phase = 0u;
    bool mma_out = false;  // a committed product not yet waited for
    bool failed = false;
    int staged_key = -1;   // b Hk + kh whose first-group keys sit in B1, kn_s and the products

    // Warps 0..3, warp = token: q and k of tokens t0 .. t0 + 3 (zeros past nt),
    // normalised into kn_s / qn_s and split into B1.
    auto stage_keys = [&](const VItem &cur, int t0, int nt, bool staged) {
        const int tw = warp;
        float qv[4], kv[4];
        if (tw >= nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) qv[e] = kv[e] = 0.f;
        } else if (staged) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qv[e] = to_f32(stq[tw * D + lane * 4 + e]);
                kv[e] = to_f32(stk[tw * D + lane * 4 + e]);
            }
        } else {
            const long long t = t0 + tw;
            const TIO *qp = qg + t * p.q_stride + (long long)cur.kh * D + lane * 4;
            const TIO *kp = kg + t * p.k_stride + (long long)cur.kh * D + lane * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qv[e] = to_f32(qp[e]);
                kv[e] = to_f32(kp[e]);
            }
        }
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            sq = fmaf(qv[e], qv[e], sq);
            sk = fmaf(kv[e], kv[e], sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float iq = 1.f / fmaxf(sqrtf(sq), EPS), ik = 1.f / fmaxf(sqrtf(sk), EPS);
        float4 kh4, kl4, qh4, ql4;
        float *khp = &kh4.x, *klp = &kl4.x, *qhp = &qh4.x, *qlp = &ql4.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qv[e] *= iq;
            kv[e] *= ik;
            khp[e] = tf32_hi(kv[e]);
            klp[e] = kv[e] - khp[e];
            qhp[e] = tf32_hi(qv[e]);
            qlp[e] = qv[e] - qhp[e];
        }
        *reinterpret_cast<float4 *>(&kn_s[tw][lane * 4]) = make_float4(kv[0], kv[1], kv[2], kv[3]);
        *reinterpret_cast<float4 *>(&qn_s[tw][lane * 4]) = make_float4(qv[0], qv[1], qv[2], qv[3]);
        // B1 rows tw (k hi), 4 + tw (k lo), 8 + tw (q hi), 12 + tw (q lo); this lane's
        // features are chunk lane % 8 of box lane / 8
        uint8_t *bx = sm + L::B1 + (lane >> 3) * 2048;
        const int qc = lane & 7;
        *reinterpret_cast<float4 *>(bx + tw * 128 + ((qc ^ tw) << 4)) = kh4;
        *reinterpret_cast<float4 *>(bx + (4 + tw) * 128 + ((qc ^ (4 + tw)) << 4)) = kl4;
        *reinterpret_cast<float4 *>(bx + (8 + tw) * 128 + ((qc ^ tw) << 4)) = qh4;
        *reinterpret_cast<float4 *>(bx + (12 + tw) * 128 + ((qc ^ (4 + tw)) << 4)) = ql4;
    };

    // Warps 0..3 (warp = token): k_s.k_t and k_s.q_t (s <= t) unless kept, the
    // gates, and the group factors.
    auto group_factors = [&](const VItem &cur, int t0, int nt, bool first_group, bool rebuild) {
        const int tw = warp;
        if (rebuild) {
            const float4 kt = *reinterpret_cast<const float4 *>(&kn_s[tw][lane * 4]);
            const float4 qt = *reinterpret_cast<const float4 *>(&qn_s[tw][lane * 4]);
            float v8[8];
#pragma unroll
            for (int s = 0; s < TB; ++s) {
                float xk = 0.f, xq = 0.f;
                if (s <= tw) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&kn_s[s][lane * 4]);
                    xk = fmaf(k4.x, kt.x, xk);
                    xq = fmaf(k4.x, qt.x, xq);
                    xk = fmaf(k4.y, kt.y, xk);
                    xq = fmaf(k4.y, qt.y, xq);
                    xk = fmaf(k4.z, kt.z, xk);
                    xq = fmaf(k4.z, qt.z, xq);
                    xk = fmaf(k4.w, kt.w, xk);
                    xq = fmaf(k4.w, qt.w, xq);
                }
                v8[s] = xk;
                v8[TB + s] = xq;
            }
            const float sum = warp_sum8(v8);
            const int vid = (lane >> 2) & 7;
            if ((lane & 3) == 0) {
                if (vid < TB) dkk_s[tw][vid] = sum;
                else dkq_s[tw][vid - TB] = sum;
            }
            __syncwarp();
        }
        // lane s < 4: the gates of token s (tokens past the span: g = 1, beta = 0)
        GateIn g = gc;
        const bool glive = lane < nt;
        if (!first_group && lane < TB && glive) {
            const long long t = t0 + lane;
            g.a = p.a[t * p.Hv + cur.h];
            g.b = p.b[t * p.Hv + cur.h];
            if (p.gate_raw) {
                g.A = p.A_log[cur.h];
                g.d = p.dt_bias[cur.h];
            }
        }
        float gl = 1.f, bl = 0.f;
        if (lane < TB && glive) gates_from(p.gate_raw, g.a, g.b, g.A, g.d, gl, bl);
        float gt[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j) gt[j] = __shfl_sync(0xffffffffu, gl, j);
        const float bt = __shfl_sync(0xffffffffu, bl, tw);
        if (tw == 0 && lane < nt && p.caps && t0 + lane - cur.bos < p.cap)
            p.caps[((long long)cur.b * p.cap + (t0 + lane - cur.bos)) * p.W + cur.h] = gl;  // capsule decay
        if (lane < TB) {
            const int s = lane;
            const bool live = tw < nt;
            float rts = 1.f;  // r(t, s) for s <= t
#pragma unroll
            for (int j = 1; j < TB; ++j)
                if (j > s && j <= tw) rts *= gt[j];
            const float kk = dkk_s[tw][s], kq = dkq_s[tw][s];
            mkk_s[tw][s] = (s < tw) ? bt * rts * kk : 0.f;
            mq_s[tw][s] = (s <= tw && live) ? p.scale * rts * kq : 0.f;
            if (s == 0) {
                const float Gt = rts * gt[0];
                bt_s[tw] = bt;
                bG_s[tw] = bt * Gt;
                sG_s[tw] = live ? p.scale * Gt : 0.f;
                if (tw == nt - 1) Gn_s = Gt;
            }
            if (s == 1) {
                float e = 1.f;
#pragma unroll
                for (int j = 1; j < TB; ++j)
                    if (j > tw && j < nt) e *= gt[j];
                eG_s[tw] = live ? e : 0.f;
            }
        }
    };

    for (int i = first; i < stop; ++i) {
        // warm the next sequence's descriptor in L2 (read when the position gets there)
        if (tid == 0 && p.cu && cur_c.b + 2 <= p.B) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.cu + cur_c.b + 1));
        if (tid == 0 && p.slots && cur_c.b + 1 < p.B) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.slots + cur_c.b + 1));

        // ---- this item's copies have landed (no copies: zeros without an initial state)
        bool bad = false;
        if (loaded) {
            bad = !ptx::mbar_wait_bounded(&full_bar, full_phase, WAIT_LIMIT);
            full_phase ^= 1u;
            loaded = false;  // (true again once the next item's copies are issued)
        }
        const int n = it.ok ? it.eos - it.bos : -1;
        if (it.ok && !p.init) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    *reinterpret_cast<float4 *>(rows + chunk_at(row, j, 4 * half + m)) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        bool tma_group = false;
        bool early = false;  // the next item's copies are already on their way

        if (n >= 2) {
            // ================= tensor-core groups
            const int key = it.b * p.Hk + it.kh;
            const bool single = n <= TB;
            for (int t0 = it.bos; t0 < it.eos; t0 += TB) {
                const int nt = min(TB, it.eos - t0);
                const bool first_group = t0 == it.bos;
                const bool staged = first_group && L::STAGE && mp.stg_ok;
                const bool keep = first_group && single && staged_key == key;
                const bool last = t0 + TB >= it.eos;
                // ---- stage 1: warp t normalises token t's q and k (unless kept); every
                //      thread writes the TF32 remainders of its columns into tensor memory
                if (!keep && warp < TB) stage_keys(it, t0, nt, staged);
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    float lo[16];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float4 x4 = *reinterpret_cast<const float4 *>(rows + chunk_at(row, j, 4 * half + m));
                        lo[4 * m + 0] = x4.x - tf32_trunc(x4.x);
                        lo[4 * m + 1] = x4.y - tf32_trunc(x4.y);
                        lo[4 * m + 2] = x4.z - tf32_trunc(x4.z);
                        lo[4 * m + 3] = x4.w - tf32_trunc(x4.w);
                    }
                    ptx::tmem_st16(tm + lane_sel + TM_LO + 32 * j + 16 * half, lo);
                }
                ptx::tmem_st_wait();
                ptx::fence_proxy_async_smem();  // rows (zeros) and B1 before the tensor core reads them
                ptx::tc_fence_before();
                __syncthreads();
                staged_key = single ? key : -1;

                // ---- the dot products: one thread of warp 4 issues them while warps 0-3 form
                //      the gates, k_s.k_t and k_s.q_t (s <= t, unless kept) and the group
                //      factors, and warps 5-7 write the capsule keys
                if (tid == ISSUER_HI) {
                    ptx::tc_fence_after();
                    issue_mma_rows(tm, rows_base, b1_base);
                    ptx::mma_commit(&mma_bar);
                } else if (tid == ISSUER_LO) {
                    ptx::tc_fence_after();
                    issue_mma_rem(tm, b1_base);
                    ptx::mma_commit(&mma_bar);
                }
                mma_out = true;
                if (tid == 0) ptx::bulk_wait_read_all();  // the previous output boxes have been read
                if (warp < TB) {
                    group_factors(it, t0, nt, first_group, !keep);
                } else if (warp > TB + 1 && p.caps && it.h % p.r == 0) {
                    for (int x = tid - (TB + 2) * 32; x < nt * D; x += (NTV / 32 - TB - 2) * 32) {
                        const int tt = x >> 7, e = x & (D - 1);
                        const int tl = t0 + tt - it.bos;
                        if (tl < p.cap)
                            p.caps[((long long)it.b * p.cap + tl) * p.W + p.Hv + (long long)it.kh * D + e] =
                                kn_s[tt][e];
                    }
                }
                // v of this row (both threads of the row form its deltas), read before the
                // barrier so that the staged rows are free once the products are done
                float vr[TB];
#pragma unroll
                for (int t = 0; t < TB; ++t)
                    vr[t] = t >= nt ? 0.f
                            : staged ? to_f32(stv[t * D + row])
                                     : to_f32(vg[(long long)(t0 + t) * p.v_stride + (long long)it.h * D + row]);
                __syncthreads();

                // ---- every thread: its row's deltas from P and Q, outputs (half 0), then the
                //      rank-4 update of its columns in place
                bad |= !ptx::mbar_wait_bounded(&mma_bar, mma_phase, WAIT_LIMIT);
                mma_phase ^= 1u;
                mma_out = false;
                ptx::tc_fence_after();
                const bool tg = mp.out_ok && last && nt == TB && (!p.caps || t0 - it.bos + TB <= p.cap);
                tma_group = tg;
                // Writing no final state, nothing reads this item's rows or staged q, k,
                // v once its last group's products are done (every thread holds its v
                // since the barrier above): thread 0 resolves the next item and starts
                // its copies, which then overlap the deltas, the outputs and the item's
                // end.  The other threads take the next item from shared memory after
                // the item's last barrier; the next item's own barriers come before
                // thread 0 writes the descriptor again.
                early = last && !p.final_state;
                if (early) {
                    if (tid == 0 && !bad) {
                        VCursor nc = cur_c;
                        advance(p, nc);
                        VRaw ns = seq;
                        VItem nxe = no_item();
                        if (i + 1 < stop) {
                            if (nc.h == 0) ns = load_raw(p, nc.b);
                            nxe = make_item(p, nc, ns);
                        }
                        nx_cur_s = nc;
                        nx_seq_s = ns;
                        nx_s = nxe;
                        issue_load(nxe, true);
                        loaded = load_bytes(nxe) != 0;  // in flight until the next item waits
                    }
                }
                float d1[16], d1l[16];
                ptx::tmem_ld16(tm + lane_sel + TM_D1, d1);
                ptx::tmem_ld16(tm + lane_sel + TM_D1L, d1l);
#pragma unroll
                for (int c = 0; c < 16; ++c) d1[c] += d1l[c];
                float u[TB];
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    float x = fmaf(bt_s[t], vr[t], -bG_s[t] * (d1[t] + d1[4 + t]));
#pragma unroll
                    for (int s = 0; s < t; ++s) x = fmaf(-mkk_s[t][s], u[s], x);
                    u[t] = x;
                }
                if (half == 0) {
#pragma unroll
                    for (int c = 0; c < TB; ++c) {
                        if (c < nt) {
                            float o = sG_s[c] * (d1[8 + c] + d1[12 + c]);
#pragma unroll
                            for (int s = 0; s < TB; ++s) o = fmaf(mq_s[c][s], u[s], o);
                            const TIO ot = from_f32<TIO>(o);
                            if (tg) {
                                o_s[row >> 6][c][row & 63] = ot;
                                u_s[row >> 6][c][row & 63] = u[c];
                            } else {
                                const long long t = t0 + c;
                                og[(t * p.Hv + it.h) * D + row] = ot;
                                const int tl = (int)(t - it.bos);
                                if (p.caps && tl < p.cap)
                                    p.caps[((long long)it.b * p.cap + tl) * p.W + ubase + (long long)it.h * D + row] =
                                        u[c];
                            }
                        }
                    }
                }
                if (!last || p.final_state) {
                    if (half == 0)
                        *reinterpret_cast<float4 *>(&w_s[row][0]) =
                            make_float4(eG_s[0] * u[0], eG_s[1] * u[1], eG_s[2] * u[2], eG_s[3] * u[3]);
                    __syncthreads();
                    // the rank-4 update, warp w over rows 16 w .. 16 w + 15, lane l over columns
                    // 4 l .. 4 l + 3 (a whole row per instruction): the final rows go straight to
                    // global memory (512-byte stores), the rows of a later group back in place
                    const float2 Gn2 = make_float2(Gn_s, Gn_s);
                    float2 k2[TB][2];
#pragma unroll
                    for (int t = 0; t < TB; ++t) {
                        const float4 k4 = *reinterpret_cast<const float4 *>(&kn_s[t][4 * lane]);
                        k2[t][0] = make_float2(k4.x, k4.y);
                        k2[t][1] = make_float2(k4.z, k4.w);
                    }
                    float *fin = p.final_state + (size_t)it.row0 * D + 4 * lane;
#pragma unroll 8
                    for (int rr = 0; rr < 16; ++rr) {
                        const int r = 16 * warp + rr;
                        float4 *sp = reinterpret_cast<float4 *>(rows + chunk_at(r, lane >> 3, lane & 7));
                        const float4 x4 = *sp;
                        const float4 w4 = *reinterpret_cast<const float4 *>(&w_s[r][0]);
                        // pairs of columns: two FP32 FMAs per instruction
                        float2 x0 = __fmul2_rn(make_float2(x4.x, x4.y), Gn2);
                        float2 x1 = __fmul2_rn(make_float2(x4.z, x4.w), Gn2);
                        const float wt[TB] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int t = 0; t < TB; ++t) {
                            const float2 w2 = make_float2(wt[t], wt[t]);
                            x0 = __ffma2_rn(w2, k2[t][0], x0);
                            x1 = __ffma2_rn(w2, k2[t][1], x1);
                        }
                        const float4 y = make_float4(x0.x, x0.y, x1.x, x1.y);
                        if (last)
                            *reinterpret_cast<float4 *>(fin + (size_t)r * D) = y;
                        else
                            *sp = y;
                    }
                }
                ptx::fence_proxy_async_smem();  // rows and output boxes before the tensor copies read them
                ptx::tc_fence_before();
                if (__syncthreads_or(bad)) {
                    failed = true;
                    break;
                }
                bad = false;
            }
            if (failed) break;
        } else if (n >= 0) {
            // ================= one token (the decode kernel's arithmetic) or none.  Partial
            //      dot products of virtual lanes l = 4 half + m (the decode kernel's lane l
            //      holds float4 chunks 8 j + l of the row) meet through the accumulator
            //      columns: half h writes its pk, pq partials to columns 8 h .. 8 h + 7.
            if (n == 1) {
                staged_key = -1;
                const long long t = it.bos;
                const float v0 = (L::STAGE && mp.stg_ok) ? to_f32(stv[row])
                                                         : to_f32(vg[t * p.v_stride + (long long)it.h * D + row]);
                if (warp == 0) {
                    float qv[4], kv[4];
                    if (L::STAGE && mp.stg_ok) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            qv[e] = to_f32(stq[lane * 4 + e]);
                            kv[e] = to_f32(stk[lane * 4 + e]);
                        }
                    } else {
                        const TIO *qp = qg + t * p.q_stride + (long long)it.kh * D + lane * 4;
                        const TIO *kp = kg + t * p.k_stride + (long long)it.kh * D + lane * 4;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            qv[e] = to_f32(qp[e]);
                            kv[e] = to_f32(kp[e]);
                        }
                    }
                    float sq = 0.f, sk = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        sq = fmaf(qv[e], qv[e], sq);
                        sk = fmaf(kv[e], kv[e], sk);
                    }
                    sq = warp_sum(sq);
                    sk = warp_sum(sk);
                    const float iq = 1.f / fmaxf(sqrtf(sq), EPS), ik = 1.f / fmaxf(sqrtf(sk), EPS);
                    float kq = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        qv[e] *= iq;
                        kv[e] *= ik;
                        qn_s[0][lane * 4 + e] = qv[e];
                        kn_s[0][lane * 4 + e] = kv[e];
                        kq = fmaf(qv[e], kv[e], kq);
                    }
                    kq = warp_sum(kq);
                    if (lane == 0) {
                        float g, beta;
                        gates_from(p.gate_raw, gc.a, gc.b, gc.A, gc.d, g, beta);
                        g1_s = g;
                        beta1_s = beta;
                        kq1_s = kq;
                    }
                }
                __syncthreads();
                const float4 *kk = reinterpret_cast<const float4 *>(kn_s[0]);
                const float4 *qq = reinterpret_cast<const float4 *>(qn_s[0]);
                {
                    float part[8];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int l = 4 * half + m;
                        float pk0 = 0.f, pk1 = 0.f, pq0 = 0.f, pq1 = 0.f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 s4 = *reinterpret_cast<const float4 *>(rows + chunk_at(row, j, l));
                            const float4 k4 = kk[j * 8 + l], q4 = qq[j * 8 + l];
                            pk0 = fmaf(s4.x, k4.x, pk0);
                            pk1 = fmaf(s4.y, k4.y, pk1);
                            pk0 = fmaf(s4.z, k4.z, pk0);
                            pk1 = fmaf(s4.w, k4.w, pk1);
                            pq0 = fmaf(s4.x, q4.x, pq0);
                            pq1 = fmaf(s4.y, q4.y, pq1);
                            pq0 = fmaf(s4.z, q4.z, pq0);
                            pq1 = fmaf(s4.w, q4.w, pq1);
                        }
                        part[m] = pk0 + pk1;
                        part[4 + m] = pq0 + pq1;
                    }
                    ptx::tmem_st8(tm + lane_sel + TM_D1 + 8u * half, part);
                    ptx::tmem_st_wait();
                }
                ptx::tc_fence_before();
                __syncthreads();
                ptx::tc_fence_after();
                float xr[16];  // pk of lanes 0..3, pq of lanes 0..3, pk of lanes 4..7, pq of lanes 4..7
                ptx::tmem_ld16(tm + lane_sel + TM_D1, xr);
                // lane l of the decode kernel ends with ((p0 + p4) + (p2 + p6)) + ((p1 + p5) + (p3 + p7))
                const float pk = ((xr[0] + xr[8]) + (xr[2] + xr[10])) + ((xr[1] + xr[9]) + (xr[3] + xr[11]));
                const float pq = ((xr[4] + xr[12]) + (xr[6] + xr[14])) + ((xr[5] + xr[13]) + (xr[7] + xr[15]));
                const float g = g1_s, beta = beta1_s, kq = kq1_s;
                const float u = beta * (v0 - g * pk);
                if (p.final_state) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            float4 *sp = reinterpret_cast<float4 *>(rows + chunk_at(row, j, 4 * half + m));
                            float4 s4 = *sp;
                            const float4 k4 = kk[j * 8 + 4 * half + m];
                            s4.x = fmaf(u, k4.x, g * s4.x);
                            s4.y = fmaf(u, k4.y, g * s4.y);
                            s4.z = fmaf(u, k4.z, g * s4.z);
                            s4.w = fmaf(u, k4.w, g * s4.w);
                            *sp = s4;
                        }
                }
                if (half == 0) {
                    og[((long long)it.bos * p.Hv + it.h) * D + row] = from_f32<TIO>(p.scale * fmaf(u, kq, g * pq));
                    if (p.caps && p.cap > 0)
                        p.caps[(long long)it.b * p.cap * p.W + ubase + (long long)it.h * D + row] = u;
                } else if (p.caps && p.cap > 0) {
                    float *crow = p.caps + (long long)it.b * p.cap * p.W;
                    for (int e = tid - 128; e <= D; e += 128) {
                        if (e == D)
                            crow[it.h] = g;
                        else if (it.h % p.r == 0)
                            crow[p.Hv + (long long)it.kh * D + e] = kn_s[0][e];
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            if (__syncthreads_or(bad)) {
                failed = true;
                break;
            }
        } else {
            if (__syncthreads_or(bad)) {
                failed = true;
                break;
            }
        }

        // ---- the next item (resolved by thread 0 already when `early`; the barrier
        //      at the end of the item orders its shared-memory copy before these reads)
        VItem nx = no_item();
        if (early) {
            cur_c = nx_cur_s;
            seq = nx_seq_s;
            nx = nx_s;
        } else {
            advance(p, cur_c);
            if (i + 1 < stop) {
                if (cur_c.h == 0) seq = load_raw(p, cur_c.b);
                nx = make_item(p, cur_c, seq);
            }
        }
        // ---- the item's output boxes and rows go back; then the buffer takes the next item
        if (tid == 0) {
            if (tma_group) {
                const int t0 = it.eos - TB;
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    ptx::tma_store_2d(&mp.out, &o_s[hb][0][0], it.h * D + 64 * hb, t0);
                    if (p.caps)
                        ptx::tma_store_2d(&mp.caps, &u_s[hb][0][0], (int)ubase + it.h * D + 64 * hb,
                                          it.b * p.cap + (t0 - it.bos));
                }
            }
            const bool rows_out = it.ok && n < 2 && p.final_state;  // one-token and empty spans
            if (rows_out) {                                         // (the others are written directly)
#pragma unroll
                for (int j = 0; j < 4; ++j) ptx::tma_store_2d(&mp.fin, rows + j * (D * 128), 32 * j, it.row0);
            }
            ptx::bulk_commit();
            if (rows_out) ptx::bulk_wait_read_all();  // the stores have read the buffer
        }
        if (!early) issue_load(nx);
        loaded = load_bytes(nx) != 0;
        it = nx;
        gc = load_gates(p, it);  // used once its copies have landed
    }

    if (tid == 0) {
        if (failed) {
            flag_error(p.status, GDN_DEVERR_TIMEOUT);
            if (mma_out) ptx::mbar_wait_bounded(&mma_bar, mma_phase, WAIT_LIMIT);  // let the products drain
            if (loaded) ptx::mbar_wait_bounded(&full_bar, full_phase, WAIT_LIMIT);  // and the copies land
        }
        ptx::bulk_wait_all();  // every tensor store is complete
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tm, TM_COLS);
    }
}

template <typename TIO>
cudaError_t launch_io(const ForwardParams &p, cudaStream_t stream) {
    using L = Layout<TIO>;
    const long long rows = (long long)p.num_slots * p.Hv * D;
    if (rows > 0x7fffffffLL || (long long)p.B * p.Hv > 0x7fffffffLL) return cudaErrorInvalidValue;
    VMaps mp;
    memset(&mp, 0, sizeof(mp));
    if (p.init && !encode_rows_f32(&mp.in, p.init, D, rows, 32, D, true)) return cudaErrorInvalidValue;
    mp.in3_ok = p.init && encode_state_tiles(&mp.in3, p.init, D, rows, D) ? 1 : 0;
    if (p.final_state && !encode_rows_f32(&mp.fin, p.final_state, D, rows, 32, D, true)) return cudaErrorInvalidValue;
    const bool f16 = sizeof(TIO) == 2;
    // outputs and capsule deltas of full groups as tensor stores: box coordinates must be
    // 16-byte aligned (capsule deltas start at float Hv + Hk dk of a row)
    {
        const long long ubase = (long long)p.Hv + (long long)p.Hk * D;
        bool ok = !p.caps || (ubase % 4 == 0 && p.W % 4 == 0);
        if (ok)
            ok = f16 ? encode_rows_f16(&mp.out, p.out, (long long)p.Hv * D, (long long)p.Hv * D, p.T, 64, TB, false)
                     : encode_rows_f32(&mp.out, static_cast<const float *>(p.out), (long long)p.Hv * D, p.T, 64, TB,
                                       false);
        if (ok && p.caps) ok = encode_rows_f32(&mp.caps, p.caps, p.W, (long long)p.B * p.cap, 64, TB, false);
        mp.out_ok = ok ? 1 : 0;
    }
    // the first group's q, k, v rows by tensor copies when their strides allow (else plain loads)
    if (L::STAGE) {
        auto enc = [&](CUtensorMap *m, const void *base, long long row_elems, long long stride) {
            if ((reinterpret_cast<uintptr_t>(base) & 15) || (stride * 2) % 16) return false;
            return encode_rows_f16(m, base, row_elems, stride, p.T, D, TB, false);
        };
        const bool ok = p.T > 0 && enc(&mp.q, p.q, (long long)p.Hk * D, p.q_stride) &&
                        enc(&mp.k, p.k, (long long)p.Hk * D, p.k_stride) &&
                        enc(&mp.v, p.v, (long long)p.Hv * D, p.v_stride);
        mp.stg_ok = ok ? 1 : 0;
    }
    auto kern = verify_kernel<TIO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::DYN);
    if (e != cudaSuccess) return e;
    const int items = p.B * p.Hv;
    const int grid = std::min(items, 2 * current_device_sms());
    return launch_dependent(kern, dim3(grid), dim3(NTV), (size_t)L::DYN, stream, p, items, mp);
}

}  // namespace

bool verify_kernel_supported(const ForwardParams &p) { return p.dk == D && p.dv == D; }

cudaError_t launch_verify(const ForwardParams &p, cudaStream_t stream) {
    if (p.B == 0) return cudaSuccess;
    return p.io_f16 ? launch_io<__half>(p, stream) : launch_io<float>(p, stream);
}

}  // namespace gdn
