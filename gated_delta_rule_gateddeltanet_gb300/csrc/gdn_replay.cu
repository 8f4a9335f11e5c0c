// Prefix replay of compact state-update capsules into an inactive bank.
//
// Source: "Replay compact fixed state for hybrid decoding" (Summary, Key
// changes): only the accepted prefix of the captured per-token updates is
// replayed into the inactive state bank, which is then published.  Each
// capsule row carries the decay g, the shared unit key kn and the delta u of
// one token ("[CUDA] Add compact GatedDeltaNet operator", Description), so the
// replay of token i is the rank-1 transition  S <- g_i S + u_i kn_i^T.
//
// Rows of the V-major state are independent, so the kernel is a stream: read
// each state row once, apply the accepted transitions in registers, write it
// once.  It is HBM-bound, and with only a few state tiles per SM (16 requests
// x 48 heads x 64 KiB = 48 MiB is two to three tiles per SM at 64 rows) the
// time goes into filling the memory pipe, not into arithmetic.  So the unit of
// work is small: a CTA of two warps owns an 8-row slice (4 KiB at dk = 128) of
// one (request, value head), and up to 30 CTAs share an SM, which keeps ~120
// KiB of state reads in flight per SM and leaves no long wave tail.
//
// Per CTA: one bulk (TMA) copy brings the 8 rows into shared memory while the
// first TBC accepted capsules (kn of the key head, the 8 u entries, a 16-byte
// group of decays holding g_h) arrive by bulk copies on the same mbarrier
// (plain loads where the capsule rows are not 16-byte aligned).  A lane owns
// one float4 column group of RPT rows; the transitions need no reductions.
// The rows go back to the destination bank as coalesced 16-byte stores.  A
// replay of zero tokens is a copy (the tile is sent back by one bulk store);
// nothing is done when the destination is the source and nothing was accepted.
#include "gdn_internal.cuh"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int NT = 64;    // two warps
constexpr int ROWS = 8;   // state rows per CTA
constexpr int TBC = 4;    // capsules staged per round
constexpr int MIN_CTAS = 30;
constexpr long long WAIT_LIMIT = 4000000000LL;

template <int DK>
__global__ void __launch_bounds__(NT, MIN_CTAS) replay_kernel(const ReplayParams p, int bulk_caps) {
    dependent_prologue();
    constexpr int LPR4 = DK / 4;                   // lanes covering one row, a float4 each
    constexpr int RPI = 32 / LPR4;                 // rows per warp instruction
    constexpr int RPT = ROWS / ((NT / 32) * RPI);  // rows per thread
    static_assert(RPT >= 1 && RPT * RPI * (NT / 32) == ROWS, "row split");

    __shared__ __align__(128) float tile[ROWS * DK];
    __shared__ __align__(16) float kn_s[TBC][DK];
    __shared__ __align__(16) float u_s[TBC][ROWS];
    __shared__ __align__(16) float gq_s[TBC][4];  // the 16-byte group of decays holding g_h
    __shared__ __align__(8) uint64_t bar;

    const int nrb = (p.dv + ROWS - 1) / ROWS;
    const int rb = blockIdx.x % nrb, h = blockIdx.x / nrb, j = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane % LPR4, rsub = lane / LPR4;
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
    const long long kbase = (long long)p.Hv + (long long)kh * DK;
    const long long ubase = (long long)p.Hv + (long long)p.Hk * DK + (long long)h * p.dv + rb * ROWS;
    const float *caps_j = p.caps + (long long)j * p.cap * p.W;
    const int nt0 = min(TBC, n);

    // capsules i0 .. i0+nt-1 into the staging buffers with plain loads
    auto stage_plain = [&](int i0, int nt) {
        for (int i = tid; i < nt * DK; i += NT) {
            const int tt = i / DK, e = i % DK;
            kn_s[tt][e] = caps_j[(long long)(i0 + tt) * p.W + kbase + e];
        }
        for (int i = tid; i < nt * ROWS; i += NT) {
            const int tt = i / ROWS, rr = i % ROWS;
            u_s[tt][rr] = rr < rows_here ? caps_j[(long long)(i0 + tt) * p.W + ubase + rr] : 0.f;
        }
        if (tid < nt) gq_s[tid][h & 3] = caps_j[(long long)(i0 + tid) * p.W + h];
    };

    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const bool bulk = bulk_caps && rows_here == ROWS;
    if (tid == 0) {
        const uint32_t cap_bytes = bulk ? (uint32_t)nt0 * (DK * 4 + ROWS * 4 + 16) : 0u;
        ptx::mbar_arrive_expect_tx(&bar, bytes + cap_bytes);
        ptx::bulk_g2s(tile, p.banks + (size_t)src * p.Hv * p.dv * DK + row0, bytes, &bar);
    }
    if (bulk) {
        if (tid >= 32 && tid < 32 + 3 * nt0) {
            const int c = tid - 32, tt = c / 3, what = c % 3;
            const float *row = caps_j + (long long)tt * p.W;
            if (what == 0)
                ptx::bulk_g2s(kn_s[tt], row + kbase, DK * 4, &bar);
            else if (what == 1)
                ptx::bulk_g2s(u_s[tt], row + ubase, ROWS * 4, &bar);
            else
                ptx::bulk_g2s(gq_s[tt], row + (h & ~3), 16, &bar);
        }
    } else {
        stage_plain(0, nt0);
    }
    const bool ok = ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            flag_error(p.status, GDN_DEVERR_TIMEOUT);
            ptx::mbar_wait_bounded(&bar, 0, WAIT_LIMIT);  // let the copies in flight land
        }
        return;
    }

    float *dstp = p.banks + (size_t)dst * p.Hv * p.dv * DK + row0;
    if (n == 0) {  // a copy: the tile goes back unchanged
        if (tid == 0) {
            ptx::bulk_s2g(dstp, tile, bytes);
            ptx::bulk_commit();
            ptx::bulk_wait_read_all();
        }
        return;
    }

    float4 s[RPT];
    const float4 *tile4 = reinterpret_cast<const float4 *>(tile);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = (warp * RPT + i) * RPI + rsub;
        s[i] = r < rows_here ? tile4[r * LPR4 + cg] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i0 = 0; i0 < n; i0 += TBC) {
        const int nt = min(TBC, n - i0);
        if (i0 > 0) {  // capsules past the ones staged with the tile
            __syncthreads();
            stage_plain(i0, nt);
            __syncthreads();
        }
        for (int tt = 0; tt < nt; ++tt) {
            const float g = gq_s[tt][h & 3];
            const float4 k4 = reinterpret_cast<const float4 *>(kn_s[tt])[cg];
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float u = u_s[tt][(warp * RPT + i) * RPI + rsub];
                float4 &x = s[i];
                x.x = fmaf(u, k4.x, g * x.x);
                x.y = fmaf(u, k4.y, g * x.y);
                x.z = fmaf(u, k4.z, g * x.z);
                x.w = fmaf(u, k4.w, g * x.w);
            }
        }
    }
    float4 *dst4 = reinterpret_cast<float4 *>(dstp);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = (warp * RPT + i) * RPI + rsub;
        if (r < rows_here) dst4[r * LPR4 + cg] = s[i];
    }
}

template <int DK>
cudaError_t launch_dk(const ReplayParams &p, cudaStream_t stream) {
    const int nrb = (p.dv + ROWS - 1) / ROWS;
    dim3 grid((unsigned)(nrb * p.Hv), (unsigned)p.R);
    // Capsule rows are 16-byte aligned (bulk-copyable) when the row width and
    // the offsets of kn, u and the decay groups are multiples of four floats:
    // W = Hv + Hk dk + Hv dv is, whenever Hv is (dk, dv are multiples of 32).
    const int bulk_caps = (p.Hv % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.caps) & 15) == 0);
    return launch_dependent(replay_kernel<DK>, grid, dim3(NT), 0, stream, p, bulk_caps);
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
