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
#include "gdn_internal.cuh"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;    // threads per CTA
constexpr int TB = 4;      // tokens staged per round (one warp normalises one token)
constexpr int ROWS = 64;   // state rows per CTA tile
constexpr float EPS = 1e-6f;
// Bound on any mbarrier wait (SM cycles, ~2 s); past it the CTA reports
// GDN_DEVERR_TIMEOUT and leaves its tile unwritten.
constexpr long long WAIT_LIMIT = 4000000000LL;

template <typename TIO, int DK>
__global__ void __launch_bounds__(NT, 5) recurrent_kernel(const ForwardParams p) {
    constexpr int LPR = DK / 16;             // lanes per state row
    constexpr int GPW = 32 / LPR;            // rows per warp per pass
    constexpr int ROWS_PASS = (NT / 32) * GPW;
    constexpr int NPASS = (ROWS + ROWS_PASS - 1) / ROWS_PASS;
    constexpr int EPL = DK / 32;             // q/k elements per lane when normalising

    extern __shared__ __align__(128) float tile[];  // [ROWS][DK]
    __shared__ __align__(16) float kn_s[TB][DK];
    __shared__ __align__(16) float qn_s[TB][DK];
    __shared__ float g_s[TB], beta_s[TB], kq_s[TB];
    __shared__ float v_s[TB][ROWS], o_s[TB][ROWS], u_s[TB][ROWS];
    __shared__ __align__(8) uint64_t bar;

    const int nrb = (p.dv + ROWS - 1) / ROWS;
    const int rb = blockIdx.x % nrb;
    const int h = blockIdx.x / nrb;
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int l = lane % LPR, grp = lane / LPR;
    const bool leader = (rb == 0 && h == 0 && tid == 0);

    if (p.cu && b == 0 && leader && (p.cu[0] != 0 || p.cu[p.B] != p.T)) flag_error(p.status, GDN_DEVERR_CU_SEQLENS);
    const int bos = seq_start(p.cu, p.dense_S, b), eos = seq_start(p.cu, p.dense_S, b + 1);
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
    const int rows_here = min(ROWS, p.dv - rb * ROWS);
    const uint32_t bytes = (uint32_t)rows_here * DK * 4;
    const size_t off = (((size_t)slot * p.Hv + h) * (size_t)p.dv + (size_t)rb * ROWS) * DK;

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
        for (int i = tid; i < rows_here * DK / 4; i += NT) t4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
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
        constexpr int VPT = (TB * ROWS + NT - 1) / NT;
        float vreg[VPT];
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            const int i = tid + m * NT, tt = i / ROWS, rr = i % ROWS;
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
            const int i = tid + m * NT;
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
        for (int i = tid; i < nt * ROWS; i += NT) {
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
cudaError_t launch_dk(const ForwardParams &p, cudaStream_t stream) {
    const int nrb = (p.dv + ROWS - 1) / ROWS;
    dim3 grid((unsigned)(nrb * p.Hv), (unsigned)p.B);
    const int smem = ROWS * DK * 4;
    auto kern = recurrent_kernel<TIO, DK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, NT, smem, stream>>>(p);
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
