// Prefix replay of compact state-update capsules into an inactive bank.
//
// Source: "Replay compact fixed state for hybrid decoding" (Summary, Key
// changes): only the accepted prefix of the captured per-token updates is
// replayed into the inactive state bank, which is then published.  Each
// capsule row carries the decay g, the shared unit key kn and the delta u of
// one token ("[CUDA] Add compact GatedDeltaNet operator", Description), so the
// replay of token i is the rank-1 transition  S <- g_i S + u_i kn_i^T.
//
// Like the recurrent kernel, rows of the V-major state are independent and the
// kernel is HBM-bound: a CTA moves a 64-row tile of one (request, value head)
// from the source bank into shared memory with one bulk (TMA) copy, stages the
// accepted capsules meanwhile, applies the transitions on register-resident
// rows (LPR = dk/16 lanes per row, 16 floats per lane; no reductions needed)
// and sends the tile to the destination bank with one bulk store.  A replay of
// zero tokens is a copy; nothing is done when the destination is the source
// and nothing was accepted.
#include "gdn_internal.cuh"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;
constexpr int TB = 8;     // capsules staged per round
constexpr int ROWS = 64;  // state rows per CTA tile
constexpr long long WAIT_LIMIT = 4000000000LL;

template <int DK>
__global__ void __launch_bounds__(NT, 5) replay_kernel(const ReplayParams p) {
    constexpr int LPR = DK / 16;
    constexpr int GPW = 32 / LPR;
    constexpr int ROWS_PASS = (NT / 32) * GPW;
    constexpr int NPASS = (ROWS + ROWS_PASS - 1) / ROWS_PASS;

    extern __shared__ __align__(128) float tile[];  // [ROWS][DK]
    __shared__ __align__(16) float kn_s[TB][DK];
    __shared__ float g_s[TB];
    __shared__ float u_s[TB][ROWS];
    __shared__ __align__(8) uint64_t bar;

    const int nrb = (p.dv + ROWS - 1) / ROWS;
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
    const int rows_here = min(ROWS, p.dv - rb * ROWS);
    const uint32_t bytes = (uint32_t)rows_here * DK * 4;
    const size_t row0 = ((size_t)h * p.dv + (size_t)rb * ROWS) * DK;
    const size_t src_off = (size_t)src * p.Hv * p.dv * DK + row0;
    const size_t dst_off = (size_t)dst * p.Hv * p.dv * DK + row0;

    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
        ptx::mbar_arrive_expect_tx(&bar, bytes);
        ptx::bulk_g2s(tile, p.banks + src_off, bytes, &bar);
    }
    bool tile_pending = true;

    const long long ubase = (long long)p.Hv + (long long)p.Hk * DK + (long long)h * p.dv + rb * ROWS;
    for (int i0 = 0; i0 < n || tile_pending; i0 += TB) {
        const int nt = max(0, min(TB, n - i0));
        for (int i = tid; i < nt * DK; i += NT) {
            const int tt = i / DK, e = i % DK;
            kn_s[tt][e] = p.caps[((long long)j * p.cap + i0 + tt) * p.W + p.Hv + (long long)kh * DK + e];
        }
        for (int i = tid; i < nt * ROWS; i += NT) {
            const int tt = i / ROWS, rr = i % ROWS;
            u_s[tt][rr] = rr < rows_here ? p.caps[((long long)j * p.cap + i0 + tt) * p.W + ubase + rr] : 0.f;
        }
        if (tid < nt) g_s[tid] = p.caps[((long long)j * p.cap + i0 + tid) * p.W + h];
        __syncthreads();  // also orders the mbarrier init before other threads wait on it
        if (tile_pending) {
            const bool ok = ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) {
                    flag_error(p.status, GDN_DEVERR_TIMEOUT);
                    ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);
                }
                return;
            }
            tile_pending = false;
        }
#pragma unroll
        for (int pass = 0; pass < NPASS; ++pass) {
            const int lrow = pass * ROWS_PASS + warp * GPW + grp;
            if (lrow >= rows_here || nt == 0) continue;
            float4 *rowp = reinterpret_cast<float4 *>(tile + (size_t)lrow * DK);
            float4 s[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) s[q] = rowp[q * LPR + l];
            for (int tt = 0; tt < nt; ++tt) {
                const float g = g_s[tt], u = u_s[tt][lrow];
                const float4 *kk = reinterpret_cast<const float4 *>(kn_s[tt]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 k4 = kk[q * LPR + l];
                    s[q].x = fmaf(u, k4.x, g * s[q].x);
                    s[q].y = fmaf(u, k4.y, g * s[q].y);
                    s[q].z = fmaf(u, k4.z, g * s[q].z);
                    s[q].w = fmaf(u, k4.w, g * s[q].w);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) rowp[q * LPR + l] = s[q];
        }
        __syncthreads();
    }

    ptx::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        ptx::bulk_s2g(p.banks + dst_off, tile, bytes);
        ptx::bulk_commit();
        ptx::bulk_wait_read_all();
    }
}

template <int DK>
cudaError_t launch_dk(const ReplayParams &p, cudaStream_t stream) {
    const int nrb = (p.dv + ROWS - 1) / ROWS;
    dim3 grid((unsigned)(nrb * p.Hv), (unsigned)p.R);
    const int smem = ROWS * DK * 4;
    auto kern = replay_kernel<DK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, NT, smem, stream>>>(p);
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
