// Prefix replay of compact state-update capsules into an inactive bank.
//
// Source: "Replay compact fixed state for hybrid decoding" (Summary, Key
// changes): only the accepted prefix of the captured per-token updates is
// replayed into the inactive state bank, which is then published.  Each
// capsule row carries the decay g, the shared unit key kn and the delta u of
// one token ("[CUDA] Add compact GatedDeltaNet operator", Description), so the
// replay of token i is the rank-1 transition  S <- g_i S + u_i kn_i^T.
//
// Like the recurrent kernel, rows of the V-major state are independent: a CTA
// of 256 threads streams ROWS_CTA rows of one (request, value head) from the
// source bank into registers (LPR = dk/16 lanes per row, 16 floats per lane),
// applies the accepted transitions, and streams them to the destination bank.
// No reductions are needed.  A replay of zero tokens is a copy, and nothing is
// done when the destination is the source and nothing was accepted.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;
constexpr int TB = 8;  // capsules staged per round

template <int DK, int RPT>
__global__ void __launch_bounds__(NT) replay_kernel(const ReplayParams p) {
    constexpr int LPR = DK / 16;
    constexpr int GPW = 32 / LPR;
    constexpr int ROWS_PASS = (NT / 32) * GPW;
    constexpr int ROWS_CTA = ROWS_PASS * RPT;

    __shared__ __align__(16) float kn_s[TB][DK];
    __shared__ float g_s[TB];
    __shared__ float u_s[TB][ROWS_CTA];

    const int nrb = (p.dv + ROWS_CTA - 1) / ROWS_CTA;
    const int rb = blockIdx.x % nrb;
    const int h = blockIdx.x / nrb;
    const int j = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int l = lane % LPR, grp = lane / LPR;
    const bool leader = (rb == 0 && h == 0 && tid == 0);

    const int src = p.src[j], dst = p.dst[j], n = p.n[j];
    if (src < 0 || src >= p.num_slots || dst < 0 || dst >= p.num_slots) {
        if (leader) flag_error(p.status, GDN_DEVERR_REPLAY_SLOT);
        return;
    }
    if (n < 0 || n > p.cap) {
        if (leader) flag_error(p.status, GDN_DEVERR_ACCEPT_LEN);
        return;
    }
    if (src == dst && n == 0) return;
    const int kh = h / p.r;

    const size_t src_off = ((size_t)src * p.Hv + h) * (size_t)p.dv * DK;
    const size_t dst_off = ((size_t)dst * p.Hv + h) * (size_t)p.dv * DK;
    float4 s[RPT][4];
    int lrow[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        lrow[k] = k * ROWS_PASS + warp * GPW + grp;
        const int row = rb * ROWS_CTA + lrow[k];
        if (row < p.dv) {
            const float4 *sp = reinterpret_cast<const float4 *>(p.banks + src_off + (size_t)row * DK);
#pragma unroll
            for (int q = 0; q < 4; ++q) s[k][q] = __ldcs(sp + q * LPR + l);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) s[k][q] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    const long long ubase = (long long)p.Hv + (long long)p.Hk * DK + (long long)h * p.dv;
    for (int i0 = 0; i0 < n; i0 += TB) {
        const int nt = min(TB, n - i0);
        for (int i = tid; i < nt * DK; i += NT) {
            const int tt = i / DK, e = i % DK;
            kn_s[tt][e] = p.caps[((long long)j * p.cap + i0 + tt) * p.W + p.Hv + (long long)kh * DK + e];
        }
        for (int i = tid; i < nt * ROWS_CTA; i += NT) {
            const int tt = i / ROWS_CTA, rr = i % ROWS_CTA;
            const int row = rb * ROWS_CTA + rr;
            u_s[tt][rr] = row < p.dv ? p.caps[((long long)j * p.cap + i0 + tt) * p.W + ubase + row] : 0.f;
        }
        if (tid < nt) g_s[tid] = p.caps[((long long)j * p.cap + i0 + tid) * p.W + h];
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            const float g = g_s[tt];
#pragma unroll
            for (int k = 0; k < RPT; ++k) {
                const float u = u_s[tt][lrow[k]];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 kk = reinterpret_cast<const float4 *>(kn_s[tt])[q * LPR + l];
                    s[k][q].x = fmaf(u, kk.x, g * s[k][q].x);
                    s[k][q].y = fmaf(u, kk.y, g * s[k][q].y);
                    s[k][q].z = fmaf(u, kk.z, g * s[k][q].z);
                    s[k][q].w = fmaf(u, kk.w, g * s[k][q].w);
                }
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int row = rb * ROWS_CTA + lrow[k];
        if (row >= p.dv) continue;
        float4 *dp = reinterpret_cast<float4 *>(p.banks + dst_off + (size_t)row * DK);
#pragma unroll
        for (int q = 0; q < 4; ++q) __stcs(dp + q * LPR + l, s[k][q]);
    }
}

template <int DK>
cudaError_t launch_dk(const ReplayParams &p, cudaStream_t stream) {
    constexpr int RPT = 2;
    constexpr int ROWS_CTA = (NT / 32) * (32 / (DK / 16)) * RPT;
    const int nrb = (p.dv + ROWS_CTA - 1) / ROWS_CTA;
    dim3 grid((unsigned)(nrb * p.Hv), (unsigned)p.R);
    replay_kernel<DK, RPT><<<grid, NT, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_replay(const ReplayParams &p, cudaStream_t stream) {
    if (p.R == 0) return cudaSuccess;
    switch (p.dk) {
        case 32: return launch_dk<32>(p, stream);
        case 64: return launch_dk<64>(p, stream);
        default: return launch_dk<128>(p, stream);
    }
}

}  // namespace gdn
