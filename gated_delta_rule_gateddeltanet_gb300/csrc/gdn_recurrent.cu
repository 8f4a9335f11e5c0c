// Token-by-token (decode / short-span) gated delta rule kernels.
//
// Operator: "[CUDA] Add compact GatedDeltaNet operator" (Description) -- the
// recurrent path for decode and short spans, with the native gate arithmetic
// and the compact state_update capsule fused in.
//
// 1. Decode kernel (every span has at most one token) -- CUDA cores.
//
// With a V-major state, row i of S (dk floats, value channel i) evolves on its
// own: for a token with unit key kn, unit query qn, decay g and beta,
//     p   = S_i . kn,   s = S_i . qn            (one read of the old row)
//     u_i = beta (v_i - g p)
//     S_i <- g S_i + u_i kn
//     o_i = scale (g s + u_i (kn . qn))          (= scale S_i(new) . qn)
// so both dot products come from one read of the row, and the state is read
// once and written once per call however many tokens the span has.
//
// Data movement (the kernel is HBM-bound: 0.75 FLOP per state byte): a CTA
// owns a tile of ROWS = 64 consecutive rows of one (sequence, value head),
// which is one contiguous 64*dk*4-byte run of the state (32 KiB at dk = 128).
// One thread moves the whole tile with a single bulk (TMA) copy into shared
// memory, completion tracked by an mbarrier; the per-token vectors
// (normalised q and k, k.q, gates, v) are staged meanwhile, so their
// dependent loads overlap the tile's flight.  After the update the tile goes
// back with one bulk store (none when the caller passes no final-state
// buffer).  No state bytes live in registers while in flight, so registers
// stay low (48) and 5 CTAs fit per SM: up to 160 KiB of state in flight per
// SM, enough to cover HBM latency.
//
// Compute mapping: LPR = dk/16 lanes share a row, 16 floats each as four
// float4 (lane l reads float4 j*LPR + l, so the LPR lanes of a row cover one
// contiguous run and the shared-memory reads are conflict-free); both dot
// products are LPR-wide xor-shuffle reductions.  Tokens are staged TB at a
// time; rows stay in registers across the staged tokens.
//
// 2. Mixed kernel (some span has several tokens: speculative verification,
// short prefill) at head sizes 32 and 64 (at dk = dv = 128 such batches run
// the tcgen05 kernel of gdn_verify.cu) -- a persistent kernel of 4-warp CTAs
// (4 per SM at 128 registers), each over a contiguous range of work items
// (sequence, value head, 64-row block).  One-token spans run the code above (the same bits as
// the decode kernel); longer spans run the tensor-core evaluation below.  At
// four tokens per span the CUDA-core loop is bound by instruction issue
// (about 95 instructions per row group and token), not by HBM.
//
// Tokens are taken TB = 4 at a time.  Within such a group the token-by-token
// recurrence S_t = g_t S_{t-1} + u_t k_t^T, u_t = beta_t (v_t - g_t S_{t-1} k_t),
// o_t = scale S_t q_t (unit k_t, q_t) unrolls to a closed form in the state S0
// at the start of the group.  With G_t = g_0 ... g_t and
// r(t, s) = g_{s+1} ... g_t (= G_t / G_s, formed as a product, never divided):
//     P_t = S0 k_t,  Q_t = S0 q_t                 (eight dot products per row)
//     u_t = beta_t v_t - beta_t G_t P_t - sum_{s<t} beta_t r(t,s) (k_s.k_t) u_s
//     o_t = scale (G_t Q_t + sum_{s<=t} r(t,s) (k_s.q_t) u_s)
//     S   = G_n S0 + sum_s r(n,s) u_s k_s^T       (n: last token of the group)
// The per-row work is then two dense products, S0 [rows x dk] x
// [k_0 q_0 .. k_3 q_3] [dk x 8] and the rank-4 update [rows x 4] x [4 x dk],
// and both run as mma.sync TF32 products.  Every FP32 operand is split into a
// TF32 high part and the exact remainder and three products are summed
// (hi.hi + hi.lo + lo.hi), so a product carries about 2^-21 relative error
// (FP32-level, like the CUDA-core path) for about a quarter of its
// instructions.
//
// Layout: warp w of the CTA holds tile rows 16w .. 16w + 15; lane 4 g + c
// holds rows 16w + g and 16w + g + 8 at columns 8j + 2c and 8j + 2c + 1
// (j < dk / 8).  That is the accumulator layout of the m16n8 products, so
// the rows stay in registers for the whole span and the update product
// accumulates into them directly.  The dot products use the same registers
// as their A operand with the k index permuted inside each 8-column block
// (k = c <-> column 2c, k = c + 4 <-> column 2c + 1); the staged vectors are
// read with the same permutation.
//
// Data movement: while an item computes, the next item's 64 rows arrive in
// shared memory as dk/32 TMA tensor boxes of 64 rows x 32 floats in the
// 128-byte swizzled layout (one tensor copy per box; one bulk copy per row
// was issue-bound).  Fragment row g reads tile row 2g (g < 4) or 2(g - 4) + 1
// of its 8-row group, so the swizzled 8-byte reads are conflict-free.  The
// final rows go out from registers with 8-byte stores whose 32-byte sectors
// are fully written (four lanes cover one row's 8-column block).  Items of
// one (sequence, key head) are adjacent, so a CTA keeps the key-side staging
// (unit q and k, their TF32 parts, k.k and k.q) and redoes only the gates and
// v of each value head.
#include <algorithm>
#include <cstring>

#include "chunk_tiles.cuh"
#include "gdn_internal.cuh"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;    // threads per CTA of the decode kernel
constexpr int NTM = 128;   // threads per CTA of the mixed kernel (4 warps x 16 rows on the tensor-core path)
constexpr int TB = 4;      // tokens staged per round (one warp normalises one token)
constexpr int ROWS = 64;   // state rows per CTA tile
constexpr float EPS = 1e-6f;
// Bound on any mbarrier wait (SM cycles, ~2 s); past it the CTA reports
// GDN_DEVERR_TIMEOUT and leaves its tile unwritten.
constexpr long long WAIT_LIMIT = 4000000000LL;

// Per-group staging of both span evaluations (a CTA runs one at a time): the
// staged tokens' v entries for the tile's rows, their gates, and the outputs
// and deltas before they are stored.

// One CTA's unit of work: ROWS consecutive state rows of one (sequence, value head).
struct Span {
    int b, h, rb, bos, eos, kh, rows_here;
    size_t off;  // first float of the tile in the state arrays
};

// Tensor maps for the tensor path's output stores: outputs [T, Hv dv] and
// capsules [B cap, W], boxes of TB rows x ROWS elements; ok = 0 when a map
// could not be encoded or a box coordinate would not be 16-byte aligned.
struct OutMaps {
    CUtensorMap out, caps;
    int ok;
};

// Resolves and checks the work item (sequence b, value head h, row block
// rb): its span and state slot.  False when there is nothing to do (a bad
// descriptor, which is flagged, or a span longer than max_len, which the
// chunked kernel owns).
__device__ __forceinline__ bool resolve_span(const ForwardParams &p, int b, int h, int rb, Span &sp) {
    sp.rb = rb;
    sp.h = h;
    sp.b = b;
    const bool leader = (sp.rb == 0 && sp.h == 0 && threadIdx.x == 0);
    if (p.cu && sp.b == 0 && leader && (p.cu[0] != 0 || p.cu[p.B] != p.T)) flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
    sp.bos = seq_start(p.cu, p.dense_S, sp.b);
    sp.eos = seq_start(p.cu, p.dense_S, sp.b + 1);
    if (sp.bos < 0 || sp.eos < sp.bos || sp.eos > p.T) {
        if (leader) flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
        return false;
    }
    if (sp.eos - sp.bos > p.max_len || sp.eos - sp.bos < p.min_len) return false;  // another kernel's
    const int slot = p.slots ? p.slots[sp.b] : sp.b;
    if (slot < 0 || slot >= p.num_slots) {
        if (leader) flag_error(p.status, GDN_DEVERR_STATE_SLOT);
        return false;
    }
    sp.kh = sp.h / p.r;
    sp.rows_here = min(ROWS, p.dv - sp.rb * ROWS);
    sp.off = (((size_t)slot * p.Hv + sp.h) * (size_t)p.dv + (size_t)sp.rb * ROWS) * p.dk;
    return true;
}

// The CUDA-core evaluation of one span with NTH threads.  Every row's
// arithmetic is independent of NTH, so both kernels that use it give
// bit-identical results for the spans they share.
template <typename TIO, int DK, int NTH>
__device__ __forceinline__ void span_cuda_cores(const ForwardParams &p, const Span &sp) {
    constexpr int LPR = DK / 16;             // lanes per state row
    constexpr int GPW = 32 / LPR;            // rows per warp per pass
    constexpr int ROWS_PASS = (NTH / 32) * GPW;
    constexpr int NPASS = (ROWS + ROWS_PASS - 1) / ROWS_PASS;
    constexpr int EPL = DK / 32;             // q/k elements per lane when normalising
    static_assert(NTH / 32 >= TB, "one warp normalises one staged token");

    extern __shared__ __align__(128) float tile[];  // [ROWS][DK]
    __shared__ __align__(16) float kn_s[TB][DK];
    __shared__ __align__(16) float qn_s[TB][DK];
    __shared__ float g_s[TB], beta_s[TB], kq_s[TB];
    __shared__ float v_s[TB][ROWS], o_s[TB][ROWS], u_s[TB][ROWS];
    __shared__ __align__(8) uint64_t bar;

    const int rb = sp.rb, h = sp.h, b = sp.b, bos = sp.bos, eos = sp.eos, kh = sp.kh, rows_here = sp.rows_here;
    const size_t off = sp.off;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int l = lane % LPR, grp = lane / LPR;
    const uint32_t bytes = (uint32_t)rows_here * DK * 4;

    // ---- the state tile: one bulk copy in flight while the tokens are staged
    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (p.init) {
        if (tid == 0) {
            ptx::mbar_arrive_expect_tx(&bar, bytes);
            ptx::bulk_g2s(tile, p.init + off, bytes, &bar);
        }
    } else {
        float4 *t4 = reinterpret_cast<float4 *>(tile);
        for (int i = tid; i < rows_here * DK / 4; i += NTH) t4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    bool tile_pending = p.init != nullptr;

    const TIO *qg = static_cast<const TIO *>(p.q);
    const TIO *kg = static_cast<const TIO *>(p.k);
    const TIO *vg = static_cast<const TIO *>(p.v);
    TIO *og = static_cast<TIO *>(p.out);
    const long long ubase = (long long)p.Hv + (long long)p.Hk * DK;

    for (int t0 = bos; t0 < eos; t0 += TB) {
        const int nt = min(TB, eos - t0);
        // ---- stage: every global load of the round is issued first (v entries of
        //      the tile's rows, q and k rows, gate inputs), then the normalised q
        //      and k, k.q and the gates (one warp per token)
        constexpr int VPT = (TB * ROWS + NTH - 1) / NTH;
        float vreg[VPT];
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            const int i = tid + m * NTH, tt = i / ROWS, rr = i % ROWS;
            vreg[m] = (i < nt * ROWS && rr < rows_here)
                          ? to_f32(vg[(long long)(t0 + tt) * p.v_stride + (long long)h * p.dv + rb * ROWS + rr])
                          : 0.f;
        }
        const bool stager = warp < nt;
        float qv[EPL], kv[EPL];
        float ga = 0.f, gb = 0.f, gA = 0.f, gd = 0.f;
        if (stager) {
            const long long t = t0 + warp;
            const TIO *qp = qg + t * p.q_stride + (long long)kh * DK + lane * EPL;
            const TIO *kp = kg + t * p.k_stride + (long long)kh * DK + lane * EPL;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                qv[e] = to_f32(qp[e]);
                kv[e] = to_f32(kp[e]);
            }
            if (lane == 0) {
                ga = p.a[t * p.Hv + h];
                gb = p.b[t * p.Hv + h];
                if (p.gate_raw) {
                    gA = p.A_log[h];
                    gd = p.dt_bias[h];
                }
            }
        }
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            const int i = tid + m * NTH;
            if (i < nt * ROWS) v_s[i / ROWS][i % ROWS] = vreg[m];
        }
        if (stager) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                sq = fmaf(qv[e], qv[e], sq);
                sk = fmaf(kv[e], kv[e], sk);
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            const float iq = 1.f / fmaxf(sqrtf(sq), EPS), ik = 1.f / fmaxf(sqrtf(sk), EPS);
            float kq = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                qv[e] *= iq;
                kv[e] *= ik;
                qn_s[warp][lane * EPL + e] = qv[e];
                kn_s[warp][lane * EPL + e] = kv[e];
                kq = fmaf(qv[e], kv[e], kq);
            }
            kq = warp_sum(kq);
            if (lane == 0) {
                float g, beta;
                gates_from(p.gate_raw, ga, gb, gA, gd, g, beta);
                g_s[warp] = g;
                beta_s[warp] = beta;
                kq_s[warp] = kq;
            }
        }
        __syncthreads();
        if (tile_pending) {
            const bool ok = ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) {
                    flag_error(p.status, GDN_DEVERR_TIMEOUT);
                    ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);  // let the copy land before exit
                }
                return;
            }
            tile_pending = false;
        }

        // ---- the recurrence, token by token, on register-resident rows
#pragma unroll
        for (int pass = 0; pass < NPASS; ++pass) {
            const int lrow = pass * ROWS_PASS + warp * GPW + grp;
            const bool act = lrow < rows_here;
            const int srow = act ? lrow : 0;
            float4 s[4];
            const float4 *rowp = reinterpret_cast<const float4 *>(tile + (size_t)srow * DK);
#pragma unroll
            for (int j = 0; j < 4; ++j) s[j] = act ? rowp[j * LPR + l] : make_float4(0.f, 0.f, 0.f, 0.f);
            for (int tt = 0; tt < nt; ++tt) {
                const float g = g_s[tt], beta = beta_s[tt], kq = kq_s[tt];
                const float4 *kk = reinterpret_cast<const float4 *>(kn_s[tt]);
                const float4 *qq = reinterpret_cast<const float4 *>(qn_s[tt]);
                float pk0 = 0.f, pk1 = 0.f, pq0 = 0.f, pq1 = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 k4 = kk[j * LPR + l], q4 = qq[j * LPR + l];
                    pk0 = fmaf(s[j].x, k4.x, pk0);
                    pk1 = fmaf(s[j].y, k4.y, pk1);
                    pk0 = fmaf(s[j].z, k4.z, pk0);
                    pk1 = fmaf(s[j].w, k4.w, pk1);
                    pq0 = fmaf(s[j].x, q4.x, pq0);
                    pq1 = fmaf(s[j].y, q4.y, pq1);
                    pq0 = fmaf(s[j].z, q4.z, pq0);
                    pq1 = fmaf(s[j].w, q4.w, pq1);
                }
                float pk = pk0 + pk1, pq = pq0 + pq1;
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1) {
                    pk += __shfl_xor_sync(0xffffffffu, pk, o);
                    pq += __shfl_xor_sync(0xffffffffu, pq, o);
                }
                const float u = beta * (v_s[tt][srow] - g * pk);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 k4 = kk[j * LPR + l];
                    s[j].x = fmaf(u, k4.x, g * s[j].x);
                    s[j].y = fmaf(u, k4.y, g * s[j].y);
                    s[j].z = fmaf(u, k4.z, g * s[j].z);
                    s[j].w = fmaf(u, k4.w, g * s[j].w);
                }
                if (l == 0 && act) {
                    o_s[tt][lrow] = p.scale * fmaf(u, kq, g * pq);
                    u_s[tt][lrow] = u;
                }
            }
            if (act) {
                float4 *roww = reinterpret_cast<float4 *>(tile + (size_t)lrow * DK);
#pragma unroll
                for (int j = 0; j < 4; ++j) roww[j * LPR + l] = s[j];
            }
        }
        __syncthreads();

        // ---- outputs and capsules of the staged tokens
        for (int i = tid; i < nt * ROWS; i += NTH) {
            const int tt = i / ROWS, rr = i % ROWS;
            if (rr >= rows_here) continue;
            const int row = rb * ROWS + rr;
            const long long t = t0 + tt;
            og[(t * p.Hv + h) * p.dv + row] = from_f32<TIO>(o_s[tt][rr]);
            const int tl = (int)(t - bos);
            if (p.caps && tl < p.cap)
                p.caps[((long long)b * p.cap + tl) * p.W + ubase + (long long)h * p.dv + row] = u_s[tt][rr];
        }
        if (p.caps && rb == 0) {
            for (int i = tid; i < nt * (DK + 1); i += NTH) {
                const int tt = i / (DK + 1), e = i % (DK + 1);
                const int tl = t0 + tt - bos;
                if (tl >= p.cap) continue;
                float *row = p.caps + ((long long)b * p.cap + tl) * p.W;
                if (e == DK)
                    row[h] = g_s[tt];
                else if (h % p.r == 0)
                    row[p.Hv + (long long)kh * DK + e] = kn_s[tt][e];
            }
        }
        __syncthreads();
    }

    if (tile_pending) {  // empty sequence: the tile is stored unchanged
        const bool ok = ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                flag_error(p.status, GDN_DEVERR_TIMEOUT);
                ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);
            }
            return;
        }
    }
    // ---- the tile goes back with one bulk store (unless the caller asked for no final state)
    if (!p.final_state) return;
    ptx::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        ptx::bulk_s2g(p.final_state + off, tile, bytes);
        ptx::bulk_commit();
        ptx::bulk_wait_read_all();  // the shared-memory source must outlive the copy's reads
    }
}

template <typename TIO, int DK>
__global__ void __launch_bounds__(NT, 5) recurrent_kernel(const ForwardParams p) {
    dependent_prologue();
    Span sp;
    const int nrb = (p.dv + ROWS - 1) / ROWS;
    if (!resolve_span(p, blockIdx.y, blockIdx.x / nrb, blockIdx.x % nrb, sp)) return;
    span_cuda_cores<TIO, DK, NT>(p, sp);
}

using ct::mma_tf32;
using ct::to_tf32;

// D += A B, m16n8k4 TF32: A (rows g, g + 8; k = c), B (k = c; n = g).
__device__ __forceinline__ void mma_k4(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k4.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// x = hi + lo exactly: hi is x rounded to TF32, lo the remainder (the tensor
// core reads lo's top 19 bits).
__device__ __forceinline__ void split(float x, uint32_t &hi, uint32_t &lo) {
    hi = to_tf32(x);
    lo = __float_as_uint(x - __uint_as_float(hi));
}

// Thread 0: the item's ROWS rows into shared memory as DK/32 tensor copies
// of [ROWS rows x 32 floats] boxes, each in the 128-byte swizzled layout
// (box j holds columns 32j .. 32j + 31; rows past the array read as zeros,
// rows past the tile belong to the next head and are ignored).  Earlier
// generic writes to the buffer must have been fenced to the async proxy
// before the barrier that precedes this call.
template <int DK>
__device__ __forceinline__ void issue_rows(const Span &sp, const CUtensorMap *map, float *rows_s, uint64_t *bar) {
    ptx::mbar_arrive_expect_tx(bar, (uint32_t)ROWS * DK * 4);
    const int row0 = (int)(sp.off / DK);
#pragma unroll
    for (int j = 0; j < DK / 32; ++j) ptx::tma_load_2d(rows_s + j * 32 * ROWS, map, 32 * j, row0, bar);
}

// Float offset of element (r, col) in the swizzled boxes written by issue_rows.
__device__ __forceinline__ int rows_at(int r, int col) {
    const int cb = col & 31;
    return (col >> 5) * (32 * ROWS) + r * 32 + ((((cb >> 2) ^ (r & 7)) << 2) | (cb & 3));
}

// One multi-token span.  Its rows are in flight into rows_s (when the call
// has an initial state); once every lane holds its rows the buffer is
// refilled with those of `next` (if given).  With `reuse` the key-side
// staging of the first group (unit q and k, their TF32 parts and the k.k,
// k.q products) is still in shared memory from the previous item, which had
// the same sequence and key head.  False if the copy never landed (flagged;
// the caller stops).
template <typename TIO, int DK>
__device__ __forceinline__ bool span_tensor_cores(const ForwardParams &p, const Span &sp, const CUtensorMap *map,
                                                  float *rows_s, uint64_t *bar, uint32_t &parity, const Span *next,
                                                  bool reuse, const OutMaps &om) {
    constexpr int NJ = DK / 8;       // 8-column blocks per row
    constexpr int VS = DK + 8;       // row stride of the staged vectors (bank-conflict free reads)
    constexpr int EPL = DK / 32;     // q/k elements per lane when normalising

    // vector n < TB: k_n, n >= TB: q_{n - TB} (unit vectors), TF32 high parts and remainders
    __shared__ __align__(16) float vh_s[2 * TB][VS];
    __shared__ __align__(16) float vl_s[2 * TB][VS];
    // per token t: beta_t, beta_t G_t, scale G_t, r(n, t); and the pair coefficients
    __shared__ float bt_s[TB], bG_s[TB], sG_s[TB], eG_s[TB];
    __shared__ float v_s[TB][ROWS];
    __shared__ __align__(128) TIO o_s[TB][ROWS];   // the group's outputs (I/O type): one tensor-store box
    __shared__ __align__(128) float u_s[TB][ROWS]; // the group's deltas: one tensor-store box
    __shared__ float g_s[TB], beta_s[TB];
    __shared__ float mkk_s[TB][TB], mq_s[TB][TB];  // beta_t r(t,s) k_s.k_t (s < t); scale r(t,s) k_s.q_t (s <= t)
    __shared__ float dkk_s[TB][TB], dkq_s[TB][TB];  // k_s.k_t and k_s.q_t (s <= t), kept for reuse
    __shared__ float Gn_s;

    const int rb = sp.rb, h = sp.h, b = sp.b, bos = sp.bos, eos = sp.eos, kh = sp.kh, rows_here = sp.rows_here;
    const size_t off = sp.off;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    // tile-local rows of this lane: fragment row g is row 2g (g < 4) or 2(g - 4) + 1 of the
    // warp's first 8 (and the same + 8), so that the swizzled reads below are conflict-free
    const int r0 = warp * 16 + (g < 4 ? 2 * g : 2 * g - 7), r1 = r0 + 8;
    const bool a0 = r0 < rows_here, a1 = r1 < rows_here;

    // ---- the rows, from the swizzled copy in shared memory (conflict-free 8-byte reads)
    float2 sa[NJ], sb[NJ];
    if (p.init) {
        const bool ok = ptx::mbar_wait_bounded(bar, parity, WAIT_LIMIT);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                flag_error(p.status, GDN_DEVERR_TIMEOUT);
                ptx::mbar_wait_bounded(bar, parity, WAIT_LIMIT);  // let the copies land before exit
            }
            return false;
        }
        parity ^= 1u;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            sa[j] = a0 ? *reinterpret_cast<const float2 *>(rows_s + rows_at(r0, 8 * j + 2 * c)) : make_float2(0.f, 0.f);
            sb[j] = a1 ? *reinterpret_cast<const float2 *>(rows_s + rows_at(r1, 8 * j + 2 * c)) : make_float2(0.f, 0.f);
        }
    } else {
#pragma unroll
        for (int j = 0; j < NJ; ++j) sa[j] = sb[j] = make_float2(0.f, 0.f);
    }
    __syncthreads();  // every lane holds its rows: the buffer takes the next item's
    if (next && tid == 0) issue_rows<DK>(*next, map, rows_s, bar);

    const TIO *qg = static_cast<const TIO *>(p.q);
    const TIO *kg = static_cast<const TIO *>(p.k);
    const TIO *vg = static_cast<const TIO *>(p.v);
    TIO *og = static_cast<TIO *>(p.out);
    const long long ubase = (long long)p.Hv + (long long)p.Hk * DK;

    for (int t0 = bos; t0 < eos; t0 += TB) {
        const int nt = min(TB, eos - t0);
        // ---- stage 1: v entries of the tile's rows; warp t normalises token t's q and k
        //      and computes its gates (tokens past the span become zero vectors, g = 1, beta = 0)
        constexpr int VPT = TB * ROWS / NTM;
        float vreg[VPT];
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            const int i = tid + m * NTM, tt = i / ROWS, rr = i % ROWS;
            vreg[m] = (tt < nt && rr < rows_here)
                          ? to_f32(vg[(long long)(t0 + tt) * p.v_stride + (long long)h * p.dv + rb * ROWS + rr])
                          : 0.f;
        }
        const int tw = warp;  // this warp's token
        const bool live = tw < nt;
        const bool keep = reuse && t0 == bos;  // the key-side staging is already in place
        float kv[EPL], qv[EPL];
        float ga = 0.f, gb = 0.f, gA = 0.f, gd = 0.f;
        if (live) {
            const long long t = t0 + tw;
            if (!keep) {
                const TIO *qp = qg + t * p.q_stride + (long long)kh * DK + lane * EPL;
                const TIO *kp = kg + t * p.k_stride + (long long)kh * DK + lane * EPL;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    qv[e] = to_f32(qp[e]);
                    kv[e] = to_f32(kp[e]);
                }
            }
            if (lane == 0) {
                ga = p.a[t * p.Hv + h];
                gb = p.b[t * p.Hv + h];
                if (p.gate_raw) {
                    gA = p.A_log[h];
                    gd = p.dt_bias[h];
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) qv[e] = kv[e] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            const int i = tid + m * NTM;
            v_s[i / ROWS][i % ROWS] = vreg[m];
        }
        if (!keep) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                sq = fmaf(qv[e], qv[e], sq);
                sk = fmaf(kv[e], kv[e], sk);
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            const float iq = 1.f / fmaxf(sqrtf(sq), EPS), ik = 1.f / fmaxf(sqrtf(sk), EPS);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                qv[e] *= iq;
                kv[e] *= ik;
                const int col = lane * EPL + e;
                uint32_t kh_, kl_, qh_, ql_;
                split(kv[e], kh_, kl_);
                split(qv[e], qh_, ql_);
                vh_s[tw][col] = __uint_as_float(kh_);
                vl_s[tw][col] = __uint_as_float(kl_);
                vh_s[TB + tw][col] = __uint_as_float(qh_);
                vl_s[TB + tw][col] = __uint_as_float(ql_);
            }
        }
        if (lane == 0) {
            float gt = 1.f, bt = 0.f;
            if (live) gates_from(p.gate_raw, ga, gb, gA, gd, gt, bt);
            g_s[tw] = gt;
            beta_s[tw] = bt;
        }
        __syncthreads();

        if (om.ok && tid == 0) ptx::bulk_wait_read_all();  // the previous group's stores have read o_s, u_s
        // ---- stage 2: warp t forms row t of the pair coefficients (k_s.k_t, k_s.q_t
        //      for s <= t) and its per-token factors
        {
            if (!keep) {
                float dkk[TB], dkq[TB];
#pragma unroll
                for (int s = 0; s < TB; ++s) {
                    float xk = 0.f, xq = 0.f;
                    if (s <= tw) {
#pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            const int col = lane * EPL + e;
                            const float ks = vh_s[s][col] + vl_s[s][col];
                            xk = fmaf(ks, kv[e], xk);
                            xq = fmaf(ks, qv[e], xq);
                        }
                    }
                    dkk[s] = warp_sum(xk);
                    dkq[s] = warp_sum(xq);
                }
#pragma unroll
                for (int m = 0; m < TB; ++m)
                    if (lane == m) dkk_s[tw][m] = dkk[m], dkq_s[tw][m] = dkq[m];
                __syncwarp();
            }
            if (lane < TB) {
                // lane s: r(t, s) = g_{s+1} .. g_t for s <= t
                const int s = lane;
                float rts = 1.f;
                for (int j = s + 1; j <= tw; ++j) rts *= g_s[j];
                const float kk = dkk_s[tw][s], kq = dkq_s[tw][s];
                const float bt = beta_s[tw];
                mkk_s[tw][s] = (s < tw) ? bt * rts * kk : 0.f;
                mq_s[tw][s] = (s <= tw && live) ? p.scale * rts * kq : 0.f;
                if (s == 0) {
                    const float Gt = rts * g_s[0];  // G_t = g_0 r(t, 0)
                    bt_s[tw] = bt;
                    bG_s[tw] = bt * Gt;
                    sG_s[tw] = live ? p.scale * Gt : 0.f;
                    if (tw == nt - 1) Gn_s = Gt;
                }
                if (s == 1) {
                    // r(n, t) for this warp's token (zero past the span)
                    float e = 1.f;
                    for (int j = tw + 1; j < nt; ++j) e *= g_s[j];
                    eG_s[tw] = live ? e : 0.f;
                }
            }
        }
        __syncthreads();

        // ---- the eight dot products per row: D[row][n] = S0[row] . vec_n (split TF32)
        // three accumulators: hi.hi, hi.lo, lo.hi (independent chains)
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            uint32_t ah[4], al[4];
            split(sa[j].x, ah[0], al[0]);
            split(sb[j].x, ah[1], al[1]);
            split(sa[j].y, ah[2], al[2]);
            split(sb[j].y, ah[3], al[3]);
            const float2 bh = *reinterpret_cast<const float2 *>(&vh_s[g][8 * j + 2 * c]);
            const float2 bl = *reinterpret_cast<const float2 *>(&vl_s[g][8 * j + 2 * c]);
            const uint32_t bhh[2] = {__float_as_uint(bh.x), __float_as_uint(bh.y)};
            const uint32_t bll[2] = {__float_as_uint(bl.x), __float_as_uint(bl.y)};
            mma_tf32(d0, ah, bhh);
            mma_tf32(d1, ah, bll);
            mma_tf32(d2, al, bhh);
        }
        // lane c holds vectors 2c and 2c + 1 of rows r0 (x0, x1) and r1 (x2, x3):
        // P_0, P_1 in lane 0, P_2, P_3 in lane 1, Q_0, Q_1 in lane 2, Q_2, Q_3 in lane 3
        const float x0 = d0[0] + (d1[0] + d2[0]), x1 = d0[1] + (d1[1] + d2[1]);
        const float x2 = d0[2] + (d1[2] + d2[2]), x3 = d0[3] + (d1[3] + d2[3]);
        const int quad = lane & ~3;
        float Pa[TB], Pb[TB];
#pragma unroll
        for (int s2 = 0; s2 < TB / 2; ++s2) {
            Pa[2 * s2] = __shfl_sync(0xffffffffu, x0, quad | s2);
            Pa[2 * s2 + 1] = __shfl_sync(0xffffffffu, x1, quad | s2);
            Pb[2 * s2] = __shfl_sync(0xffffffffu, x2, quad | s2);
            Pb[2 * s2 + 1] = __shfl_sync(0xffffffffu, x3, quad | s2);
        }
        // Q_c of both rows for this lane's token c
        const int qsrc = quad | (2 + (c >> 1));
        const float qa0 = __shfl_sync(0xffffffffu, x0, qsrc), qa1 = __shfl_sync(0xffffffffu, x1, qsrc);
        const float qb0 = __shfl_sync(0xffffffffu, x2, qsrc), qb1 = __shfl_sync(0xffffffffu, x3, qsrc);
        const float Q0 = (c & 1) ? qa1 : qa0, Q1 = (c & 1) ? qb1 : qb0;

        // ---- the deltas u_t of both rows (every lane of the quad forms all of them)
        float ua[TB], ub[TB];
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            const float pa = Pa[t], pb = Pb[t];
            const float bt = bt_s[t], bG = bG_s[t];
            float xa = fmaf(bt, v_s[t][r0], -bG * pa);
            float xb = fmaf(bt, v_s[t][r1], -bG * pb);
#pragma unroll
            for (int s = 0; s < t; ++s) {
                const float m = mkk_s[t][s];
                xa = fmaf(-m, ua[s], xa);
                xb = fmaf(-m, ub[s], xb);
            }
            ua[t] = xa;
            ub[t] = xb;
        }
        // ---- token c's outputs and deltas of both rows
        if (c < nt) {
            float oa = sG_s[c] * Q0, ob = sG_s[c] * Q1, uc_a = 0.f, uc_b = 0.f;
#pragma unroll
            for (int s = 0; s < TB; ++s) {
                const float m = mq_s[c][s];
                oa = fmaf(m, ua[s], oa);
                ob = fmaf(m, ub[s], ob);
                if (s == c) uc_a = ua[s], uc_b = ub[s];
            }
            o_s[c][r0] = from_f32<TIO>(oa);
            o_s[c][r1] = from_f32<TIO>(ob);
            u_s[c][r0] = uc_a;
            u_s[c][r1] = uc_b;
        }
        // a full group whose outputs and deltas all land inside this span and block: two tensor stores
        const bool tma_group = om.ok && nt == TB && rows_here == ROWS && (!p.caps || t0 - bos + TB <= p.cap);
        if (tma_group) ptx::fence_proxy_async_smem();

        // ---- S = G_n S0 + [r(n, t) u_t] [k_t]: the rank-4 update accumulates into the rows
        {
            float xa = 0.f, xb = 0.f;
#pragma unroll
            for (int s = 0; s < TB; ++s)
                if (s == c) xa = ua[s], xb = ub[s];
            const float e = eG_s[c];
            uint32_t a0h, a0l, a1h, a1l;
            split(e * xa, a0h, a0l);
            split(e * xb, a1h, a1l);
            const float Gn = Gn_s;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                // B[k = c][n = g] = k_c[8j + g]
                const uint32_t kbh = __float_as_uint(vh_s[c][8 * j + g]), kbl = __float_as_uint(vl_s[c][8 * j + g]);
                float dd[4] = {Gn * sa[j].x, Gn * sa[j].y, Gn * sb[j].x, Gn * sb[j].y};
                mma_k4(dd, a0h, a1h, kbh);
                mma_k4(dd, a0h, a1h, kbl);
                mma_k4(dd, a0l, a1l, kbh);
                sa[j] = make_float2(dd[0], dd[1]);
                sb[j] = make_float2(dd[2], dd[3]);
            }
        }
        __syncthreads();

        // ---- outputs and capsules of the group
        if (tma_group) {
            if (tid == 0) {
                ptx::tma_store_2d(&om.out, &o_s[0][0], h * p.dv + rb * ROWS, t0);
                if (p.caps)
                    ptx::tma_store_2d(&om.caps, &u_s[0][0], (int)ubase + h * p.dv + rb * ROWS, b * p.cap + (t0 - bos));
                ptx::bulk_commit();
            }
        } else {
            for (int i = tid; i < nt * ROWS; i += NTM) {
                const int tt = i / ROWS, rr = i % ROWS;
                if (rr >= rows_here) continue;
                const int row = rb * ROWS + rr;
                const long long t = t0 + tt;
                og[(t * p.Hv + h) * p.dv + row] = o_s[tt][rr];
                const int tl = (int)(t - bos);
                if (p.caps && tl < p.cap)
                    p.caps[((long long)b * p.cap + tl) * p.W + ubase + (long long)h * p.dv + row] = u_s[tt][rr];
            }
        }
        if (p.caps && rb == 0) {
            for (int i = tid; i < nt * (DK + 1); i += NTM) {
                const int tt = i / (DK + 1), e = i % (DK + 1);
                const int tl = t0 + tt - bos;
                if (tl >= p.cap) continue;
                float *row = p.caps + ((long long)b * p.cap + tl) * p.W;
                if (e == DK)
                    row[h] = g_s[tt];
                else if (h % p.r == 0)
                    row[p.Hv + (long long)kh * DK + e] = vh_s[tt][e] + vl_s[tt][e];
            }
        }
        __syncthreads();
    }

    // ---- the rows go back (none when the caller asked for no final state)
    if (!p.final_state) return true;
    float *d0p = p.final_state + off + (size_t)r0 * DK + 2 * c;
    float *d1p = d0p + 8 * DK;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        if (a0) *reinterpret_cast<float2 *>(d0p + 8 * j) = sa[j];
        if (a1) *reinterpret_cast<float2 *>(d1p + 8 * j) = sb[j];
    }
    return true;
}

// Batches with multi-token spans: a persistent kernel, each CTA over a
// contiguous range of work items.  Spans of one token (and empty ones) take the
// CUDA-core path, so a decode request gets the same bits whichever batch it
// is packed in; longer spans take the tensor-core path, and the next item's
// rows are copied into shared memory while the current one computes (a wave
// of one-shot CTAs would instead pay the full load latency in every wave).
template <typename TIO, int DK>
__global__ void __launch_bounds__(NTM, 4)
    recurrent_mixed_kernel(const ForwardParams p, int items, const __grid_constant__ CUtensorMap rows_map,
                           const __grid_constant__ OutMaps out_maps) {
    dependent_prologue();
    extern __shared__ __align__(128) float dyn_s[];  // the CUDA-core path's tile, or (1024-aligned) the swizzled rows
    float *rows_s = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(dyn_s) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t rows_bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&rows_bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    uint32_t parity = 0;
    // a contiguous range of items per CTA: consecutive items share the sequence
    // and key head (item order b, h, rb), so their key-side staging is reused
    const int stop = (int)((long long)(blockIdx.x + 1) * items / gridDim.x);
    int it = (int)((long long)blockIdx.x * items / gridDim.x);
    int staged = -1;  // b Hk + kh whose single-group staging is in shared memory, or -1
    Span cur;
    const int nrb = (p.dv + ROWS - 1) / ROWS;
    // item = (b Hv + h) nrb + rb
    auto resolve_item = [&](int item, Span &sp) {
        return resolve_span(p, item / (nrb * p.Hv), (item / nrb) % p.Hv, item % nrb, sp);
    };
    bool cur_ok = it < stop && resolve_item(it, cur);
    if (cur_ok && cur.eos - cur.bos > 1 && p.init && threadIdx.x == 0) issue_rows<DK>(cur, &rows_map, rows_s, &rows_bar);
    while (it < stop) {
        const int nx = it + 1;
        Span nxt;
        const bool nxt_ok = nx < stop && resolve_item(nx, nxt);
        const bool nxt_rows = nxt_ok && nxt.eos - nxt.bos > 1 && p.init;  // the next item wants its rows copied
        bool issued = false;
        if (cur_ok) {
            if (cur.eos - cur.bos > 1) {
                const int key = cur.b * p.Hk + cur.kh;
                const bool single = cur.eos - cur.bos <= TB;
                if (!span_tensor_cores<TIO, DK>(p, cur, &rows_map, rows_s, &rows_bar, parity, nxt_rows ? &nxt : nullptr,
                                                single && staged == key, out_maps)) {
                    if (out_maps.ok && threadIdx.x == 0) ptx::bulk_wait_all();
                    return;
                }
                staged = single ? key : -1;
                issued = nxt_rows;
            } else {
                span_cuda_cores<TIO, DK, NTM>(p, cur);
            }
        }
        ptx::fence_proxy_async_smem();  // the CUDA-core path's tile writes, before copies overwrite them
        __syncthreads();
        if (nxt_rows && !issued && threadIdx.x == 0) issue_rows<DK>(nxt, &rows_map, rows_s, &rows_bar);
        cur = nxt;
        cur_ok = nxt_ok;
        it = nx;
    }
    if (out_maps.ok && threadIdx.x == 0) ptx::bulk_wait_all();  // the output tensor stores are complete
}

template <typename TIO, int DK>
cudaError_t launch_mixed(const ForwardParams &p, cudaStream_t stream);

template <typename TIO, int DK>
cudaError_t launch_dk(const ForwardParams &p, cudaStream_t stream) {
    const int nrb = (p.dv + ROWS - 1) / ROWS;
    const bool promised = p.max_len_hint == 1;  // the caller bounds every span to one token
    if (promised || p.T == p.B) {
        // the decode kernel; without the promise only for spans of at most one token
        // (T == B allows multi-token spans next to empty ones), the rest below
        ForwardParams pd = p;
        if (!promised) pd.max_len = std::min(p.max_len, 1);
        const int smem = ROWS * DK * 4;
        auto kern = recurrent_kernel<TIO, DK>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = launch_dependent(kern, dim3((unsigned)(nrb * p.Hv), (unsigned)p.B), dim3(NT), smem, stream, pd);
        if (e != cudaSuccess || promised || p.max_len < 2) return e;
        ForwardParams pm = p;
        pm.min_len = 2;
        return verify_kernel_supported(pm) ? launch_verify(pm, stream) : launch_mixed<TIO, DK>(pm, stream);
    }
    if (verify_kernel_supported(p)) return launch_verify(p, stream);
    return launch_mixed<TIO, DK>(p, stream);
}

// Some span has several tokens: the persistent mixed kernel, as many CTAs as fit at once.
template <typename TIO, int DK>
cudaError_t launch_mixed(const ForwardParams &p, cudaStream_t stream) {
    const int nrb = (p.dv + ROWS - 1) / ROWS;
    const int smem = ROWS * DK * 4 + 1024;
    CUtensorMap rows_map;
    memset(&rows_map, 0, sizeof(rows_map));
    if (p.init && !encode_rows_f32(&rows_map, p.init, DK, (long long)p.num_slots * p.Hv * p.dv, 32, ROWS, true))
        return cudaErrorInvalidValue;
    // outputs and capsule deltas of full groups as tensor stores: box coordinates must be
    // 16-byte aligned (capsule deltas start at float Hv + Hk dk of a row)
    OutMaps out_maps;
    memset(&out_maps, 0, sizeof(out_maps));
    {
        const long long ubase = (long long)p.Hv + (long long)p.Hk * DK;
        bool ok = !p.caps || (ubase % 4 == 0 && p.W % 4 == 0);
        if (ok)
            ok = p.io_f16 ? encode_rows_f16(&out_maps.out, p.out, (long long)p.Hv * p.dv, (long long)p.Hv * p.dv, p.T,
                                            ROWS, TB, false)
                          : encode_rows_f32(&out_maps.out, static_cast<const float *>(p.out), (long long)p.Hv * p.dv, p.T,
                                            ROWS, TB, false);
        if (ok && p.caps) ok = encode_rows_f32(&out_maps.caps, p.caps, p.W, (long long)p.B * p.cap, ROWS, TB, false);
        out_maps.ok = ok ? 1 : 0;
    }
    auto kern = recurrent_mixed_kernel<TIO, DK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // CTAs per SM depend on the kernel only: asked once (0 if the query fails: one per SM)
    static const int per_sm = [&] {
        int n = 0;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NTM, smem) == cudaSuccess ? n : 0;
    }();
    const long long items = (long long)p.B * p.Hv * nrb;
    if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int grid = (int)std::min<long long>(items, (long long)std::max(per_sm, 1) * sms);
    return launch_dependent(kern, dim3(grid), dim3(NTM), smem, stream, p, (int)items, rows_map, out_maps);
}

template <typename TIO>
cudaError_t launch_io(const ForwardParams &p, cudaStream_t stream) {
    switch (p.dk) {
        case 32: return launch_dk<TIO, 32>(p, stream);
        case 64: return launch_dk<TIO, 64>(p, stream);
        default: return launch_dk<TIO, 128>(p, stream);
    }
}

}  // namespace

cudaError_t launch_recurrent(const ForwardParams &p, cudaStream_t stream) {
    if (p.B == 0) return cudaSuccess;
    return p.io_f16 ? launch_io<__half>(p, stream) : launch_io<float>(p, stream);
}

}  // namespace gdn
