// Token-by-token (decode / short-span) gated delta rule kernel.
//
// Operator: "[CUDA] Add compact GatedDeltaNet operator" (Description) -- the
// recurrent decode path of the GatedDeltaNet operator, with the native gate
// arithmetic and the compact state_update capsule fused in.
//
// With a V-major state, row i of S (dk floats, value channel i) evolves on its
// own: for a token with unit key kn, unit query qn, decay g and beta,
//     p   = S_i . kn,   s = S_i . qn            (one read of the old row)
//     u_i = beta (v_i - g p)
//     S_i <- g S_i + u_i kn
//     o_i = scale (g s + u_i (kn . qn))          (= scale S_i(new) . qn)
// so both dot products come from the same registers and the state is read
// once and written once per call however many tokens the span has.
//
// Work split: a CTA of 256 threads owns ROWS_CTA rows of one (sequence,
// value head).  LPR = dk/16 lanes share a row, each holding 16 floats of it as
// four float4 (coalesced 128-bit loads: the LPR lanes of a row read one
// contiguous 64*LPR-byte run per instruction).  Reductions are LPR-wide xor
// shuffles.  The per-token vectors (normalised q and k, gates, v, k.q) are
// staged in shared memory TB tokens at a time; the state loads are issued
// before that staging so their latency overlaps it.  State traffic uses
// streaming (evict-first) loads and stores: it is touched once.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;  // threads per CTA
constexpr int TB = 8;    // tokens staged per round (one warp normalises one token)
constexpr float EPS = 1e-6f;

template <typename TIO, int DK, int RPT>
__global__ void __launch_bounds__(NT) recurrent_kernel(const ForwardParams p) {
    constexpr int LPR = DK / 16;             // lanes per state row
    constexpr int GPW = 32 / LPR;            // rows per warp per pass
    constexpr int ROWS_PASS = (NT / 32) * GPW;
    constexpr int ROWS_CTA = ROWS_PASS * RPT;
    constexpr int EPL = DK / 32;             // q/k elements per lane when normalising

    __shared__ __align__(16) float kn_s[TB][DK];
    __shared__ __align__(16) float qn_s[TB][DK];
    __shared__ float g_s[TB], beta_s[TB], kq_s[TB];
    __shared__ float v_s[TB][ROWS_CTA];
    __shared__ float o_s[TB][ROWS_CTA];
    __shared__ float u_s[TB][ROWS_CTA];

    const int nrb = (p.dv + ROWS_CTA - 1) / ROWS_CTA;
    const int rb = blockIdx.x % nrb;
    const int h = blockIdx.x / nrb;
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int l = lane % LPR, grp = lane / LPR;
    const bool leader = (rb == 0 && h == 0 && tid == 0);

    if (b == 0 && leader && (p.cu[0] != 0 || p.cu[p.B] != p.T)) flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
    const int bos = p.cu[b], eos = p.cu[b + 1];
    if (bos < 0 || eos < bos || eos > p.T) {
        if (leader) flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
        return;
    }
    if (eos - bos > p.max_len) return;  // long span: the chunked kernel owns it
    const int slot = p.slots ? p.slots[b] : b;
    if (slot < 0 || slot >= p.num_slots) {
        if (leader) flag_error(p.status, GDN_DEVERR_STATE_SLOT);
        return;
    }
    const int kh = h / p.r;

    // ---- state rows into registers (issued first)
    const size_t head_off = ((size_t)slot * p.Hv + h) * (size_t)p.dv * DK;
    float4 s[RPT][4];
    int lrow[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        lrow[k] = k * ROWS_PASS + warp * GPW + grp;
        const int row = rb * ROWS_CTA + lrow[k];
        if (p.init && row < p.dv) {
            const float4 *src = reinterpret_cast<const float4 *>(p.init + head_off + (size_t)row * DK);
#pragma unroll
            for (int j = 0; j < 4; ++j) s[k][j] = __ldcs(src + j * LPR + l);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) s[k][j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    const TIO *qg = static_cast<const TIO *>(p.q);
    const TIO *kg = static_cast<const TIO *>(p.k);
    const TIO *vg = static_cast<const TIO *>(p.v);
    TIO *og = static_cast<TIO *>(p.out);
    const long long ubase = (long long)p.Hv + (long long)p.Hk * DK;

    for (int t0 = bos; t0 < eos; t0 += TB) {
        const int nt = min(TB, eos - t0);
        // ---- stage: normalised q and k, k.q and gates; one warp per token
        if (warp < nt) {
            const long long t = t0 + warp;
            const TIO *qp = qg + t * p.q_stride + (long long)kh * DK + lane * EPL;
            const TIO *kp = kg + t * p.k_stride + (long long)kh * DK + lane * EPL;
            float qv[EPL], kv[EPL];
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                qv[e] = to_f32(qp[e]);
                kv[e] = to_f32(kp[e]);
                sq = fmaf(qv[e], qv[e], sq);
                sk = fmaf(kv[e], kv[e], sk);
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            const float nq = fmaxf(sqrtf(sq), EPS), nk = fmaxf(sqrtf(sk), EPS);
            float kq = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                qv[e] = qv[e] / nq;
                kv[e] = kv[e] / nk;
                qn_s[warp][lane * EPL + e] = qv[e];
                kn_s[warp][lane * EPL + e] = kv[e];
                kq = fmaf(qv[e], kv[e], kq);
            }
            kq = warp_sum(kq);
            if (lane == 0) {
                float g, beta;
                gates(p, t, h, g, beta);
                g_s[warp] = g;
                beta_s[warp] = beta;
                kq_s[warp] = kq;
            }
        }
        for (int i = tid; i < nt * ROWS_CTA; i += NT) {
            const int tt = i / ROWS_CTA, rr = i % ROWS_CTA;
            const int row = rb * ROWS_CTA + rr;
            v_s[tt][rr] = row < p.dv ? to_f32(vg[(long long)(t0 + tt) * p.v_stride + (long long)h * p.dv + row]) : 0.f;
        }
        __syncthreads();

        // ---- the recurrence, token by token, on register-resident rows
        for (int tt = 0; tt < nt; ++tt) {
            const float g = g_s[tt], beta = beta_s[tt], kq = kq_s[tt];
            float4 kk[4], qq[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                kk[j] = reinterpret_cast<const float4 *>(kn_s[tt])[j * LPR + l];
                qq[j] = reinterpret_cast<const float4 *>(qn_s[tt])[j * LPR + l];
            }
#pragma unroll
            for (int k = 0; k < RPT; ++k) {
                float pk0 = 0.f, pk1 = 0.f, pq0 = 0.f, pq1 = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    pk0 = fmaf(s[k][j].x, kk[j].x, pk0);
                    pk1 = fmaf(s[k][j].y, kk[j].y, pk1);
                    pk0 = fmaf(s[k][j].z, kk[j].z, pk0);
                    pk1 = fmaf(s[k][j].w, kk[j].w, pk1);
                    pq0 = fmaf(s[k][j].x, qq[j].x, pq0);
                    pq1 = fmaf(s[k][j].y, qq[j].y, pq1);
                    pq0 = fmaf(s[k][j].z, qq[j].z, pq0);
                    pq1 = fmaf(s[k][j].w, qq[j].w, pq1);
                }
                float pk = pk0 + pk1, pq = pq0 + pq1;
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1) {
                    pk += __shfl_xor_sync(0xffffffffu, pk, off);
                    pq += __shfl_xor_sync(0xffffffffu, pq, off);
                }
                const float u = beta * (v_s[tt][lrow[k]] - g * pk);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[k][j].x = fmaf(u, kk[j].x, g * s[k][j].x);
                    s[k][j].y = fmaf(u, kk[j].y, g * s[k][j].y);
                    s[k][j].z = fmaf(u, kk[j].z, g * s[k][j].z);
                    s[k][j].w = fmaf(u, kk[j].w, g * s[k][j].w);
                }
                if (l == 0) {
                    o_s[tt][lrow[k]] = p.scale * fmaf(u, kq, g * pq);
                    u_s[tt][lrow[k]] = u;
                }
            }
        }
        __syncthreads();

        // ---- outputs and capsules of the staged tokens
        for (int i = tid; i < nt * ROWS_CTA; i += NT) {
            const int tt = i / ROWS_CTA, rr = i % ROWS_CTA;
            const int row = rb * ROWS_CTA + rr;
            if (row >= p.dv) continue;
            const long long t = t0 + tt;
            og[(t * p.Hv + h) * p.dv + row] = from_f32<TIO>(o_s[tt][rr]);
            const int tl = (int)(t - bos);
            if (p.caps && tl < p.cap)
                p.caps[((long long)b * p.cap + tl) * p.W + ubase + (long long)h * p.dv + row] = u_s[tt][rr];
        }
        if (p.caps && rb == 0) {
            for (int i = tid; i < nt * (DK + 1); i += NT) {
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

    // ---- state rows out
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int row = rb * ROWS_CTA + lrow[k];
        if (row >= p.dv) continue;
        float4 *dst = reinterpret_cast<float4 *>(p.final_state + head_off + (size_t)row * DK);
#pragma unroll
        for (int j = 0; j < 4; ++j) __stcs(dst + j * LPR + l, s[k][j]);
    }
}

template <typename TIO, int DK>
cudaError_t launch_dk(const ForwardParams &p, cudaStream_t stream) {
    constexpr int RPT = 2;
    constexpr int ROWS_CTA = (NT / 32) * (32 / (DK / 16)) * RPT;
    const int nrb = (p.dv + ROWS_CTA - 1) / ROWS_CTA;
    dim3 grid((unsigned)(nrb * p.Hv), (unsigned)p.B);
    recurrent_kernel<TIO, DK, RPT><<<grid, NT, 0, stream>>>(p);
    return cudaGetLastError();
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
