// Chunked (WY / UT-transform) gated delta rule on the tcgen05 tensor cores.
//
// Operator: "[CUDA] Add compact GatedDeltaNet operator" (Description) -- the
// tensor-core chunked prefill path of the GatedDeltaNet operator.  Same
// results as the token-by-token recurrence, evaluated 64 tokens at a time.
//
// Algebra (per (sequence, value head) chain, chunk of n <= 64 tokens, S0 the
// dv x dk state entering the chunk, Gamma_r the within-chunk cumulative log
// decay, gamma_r = exp(Gamma_r)):
//   A[r,s] = beta_r exp(Gamma_r - Gamma_s) (k_r . k_s)  (s < r);  T = (I + A)^-1
//   R^T    = (V - diag(gamma) K S0^T)^T diag(beta)       (dv x n)
//   U^T    = R^T T^T                                      (the capsule deltas)
//   O^T    = scale (S0 (diag(gamma) Q)^T + U^T (P o D)^T),  P = Q K^T,
//            D[r,s] = exp(Gamma_r - Gamma_s) (s <= r)
//   S1     = gamma_last S0 + (U^T diag(exp(Gamma_last - Gamma))) K
// This follows from S_r = gamma_r S0 + sum_{s<=r} (gamma_r/gamma_s) u_s k_s^T
// and u_r = beta_r (v_r - g_r S_{r-1} k_r).  Only differences Gamma_r -
// Gamma_s with r >= s are exponentiated (never exp(-Gamma)).
//
// Every product is an M = 128 tcgen05.mma (kind::f16, fp16 operands, fp32
// accumulators in tensor memory) with the operands in the 128-byte swizzled
// layout, K-major except K in MMA5 (read from the tile's K rows as an MN-major
// operand), and the value dimension (dv = 128) as M:
//   MMA1  [Q;K] K^T            -> P = Q K^T, G = K K^T      (128 x 64, K = dk)
//   MMA2  S0 [K ; gamma Q]^T   -> X^T = S0 K^T, S0 (gamma Q)^T (128 x 128, K = dk)
// Q, K and gamma Q are the three 64-row bands of one 192-row tile, so MMA1
// reads rows 0-127 and MMA2 rows 64-191 (one N = 128 MMA instead of two
// N = 64 ones that would each re-read S0).
//   MMA3  R^T T^T              -> U^T                        (128 x 64, K = n)
//   MMA4  U^T (P o D)^T        accumulated onto S0 (gamma Q)^T -> O^T
//   MMA5  (U^T diag) K         accumulated onto gamma_last S0 -> S1 (128 x 128, K = n)
// The FP32 state lives in tensor memory for the whole chain (128 columns);
// its fp16 copy for MMA2 is rebuilt from it every chunk.  The triangular
// inverse is stored in FP32: 16 x 16 diagonal blocks by forward substitution
// on the CUDA cores, then two levels of block combination as warp-level TF32
// products.
//
// Staging: with fp16 I/O the q, k and v rows of the next chunk arrive by three
// 2-D TMA copies (tensor maps over the packed [T, heads * 128] arrays, one
// 64-token x 128-element box each) while the current chunk computes.
//
// Scheduling: a persistent grid of one CTA per SM (the shared-memory
// footprint forces one) pulls (sequence, value head) chains from a list that a
// one-CTA planning kernel sorts longest-first, through an atomic counter in
// the caller's workspace.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "chunk_tiles.cuh"
#include "gdn_internal.cuh"
#include "ptx.cuh"

namespace gdn {
namespace {

using namespace ct;

constexpr int NT = 512;  // 16 warps: four per tensor-memory lane quarter
constexpr int CH = 64;   // chunk length
constexpr int DH = 128;  // dk = dv on this path
constexpr float EPS = 1e-6f;
constexpr float LOG_DECAY_FLOOR = -200.f;  // exp(-200) is 0 in fp32; keeps Gamma well-conditioned
constexpr long long WAIT_LIMIT = 4000000000LL;
constexpr int TMEM_COLS = 512;

// Tensor-memory columns (128 lanes each).
constexpr uint32_t TM_S = 0;     // FP32 state S (dv lanes x dk columns)
constexpr uint32_t TM_D1 = 128;  // P (lanes 0-63) and G (lanes 64-127), 64 columns
constexpr uint32_t TM_D3 = 192;  // U^T, 64 columns
constexpr uint32_t TM_X = 256;   // X^T = S0 K^T, 64 columns
constexpr uint32_t TM_O = 320;   // S0 (gamma Q)^T + U^T (P o D)^T, 64 columns

// Shared-memory layout (bytes from a 1024-byte aligned base).  fp16 tiles are
// K-major with the 128-byte swizzle.
constexpr int OFF_QKG = 0;                 // [192][128]: rows 0-63 Q, 64-127 K, 128-191 gamma Q  48 KiB
constexpr int QKG_ROWS = 192;
constexpr int QKG_KB = QKG_ROWS * 128;     // bytes between its two 64-element K blocks
constexpr int OFF_KT = OFF_QKG + 49152;    // 16 KiB, unused (K is read from the K rows as an MN-major operand)
constexpr int OFF_S16 = OFF_KT + 16384;    // [128][128]: S0 in fp16                    32 KiB
constexpr int OFF_A32 = OFF_S16 + 32768;   //   (R^T/U^T tiles, idle until R^T is built): A in fp32 [64][65]
constexpr int OFF_RT = OFF_S16 + 32768;    // [128][64]: R^T, then U^T                  16 KiB
constexpr int OFF_UD = OFF_RT + 16384;     // [128][64]: U^T diag(exp(Gamma_last - Gamma)) 16 KiB
constexpr int OFF_T = OFF_UD + 16384;      // [64][64]: T                               8 KiB
constexpr int OFF_PD = OFF_T + 8192;       // [64][64]: P o D                           8 KiB
constexpr int OFF_V = OFF_PD + 8192;       // [64][128] fp32 v                          32 KiB
constexpr int OFF_T32 = OFF_V + 32768;     //   (staging, idle from A3 to the next prefetch): T in fp32 [64][68]
constexpr int OFF_M = OFF_T32 + 64 * 68 * 4; //   and the block-combination scratch [32][36]
constexpr int OFF_STG = OFF_V + 32768;     // fp16 I/O: raw q, k, v rows of the next chunk  48 KiB
constexpr int STG_BYTES = 3 * CH * DH * 2;
constexpr int SMEM_ALLOC = OFF_STG + STG_BYTES + 1024;  // + slack for the 1024-byte alignment
static_assert(SMEM_ALLOC + 2048 <= 227 * 1024, "shared memory budget (dynamic + static)");
static_assert(64 * 65 * 4 <= 32768, "fp32 A staging fits the R^T and U^T tiles");
static_assert(OFF_M + 32 * 36 * 4 <= OFF_STG + STG_BYTES, "fp32 T staging fits the staging area");

// Row strides (floats) of the fp32 A and T staging and of the block-product scratch.
constexpr int AS = 65, TS = 68, MS = 36;

// Unit lower-triangular inverse T = (I + A)^-1 of a 64 x 64 strictly lower A
// (fp32, row stride AS, shared) into T32 (row stride TS).  The four 16 x 16
// diagonal blocks come from forward substitution; the off-diagonal blocks from
// the block identity [[L11, 0], [L21, L22]]^-1 = [[T11, 0], [-T22 L21 T11, T22]],
// first for the two 32 x 32 diagonal blocks, then for the whole matrix.  Only
// the strictly lower half and the two upper 16 x 16 blocks inside the 32 x 32
// diagonal blocks are written (the latter as zeros: they are read as part of
// T11 and T22); the upper-right 32 x 32 quadrant is never read.
__device__ void tri_inverse(const float *A, float *T32, float *M, int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    // zeros above the diagonal blocks inside the two 32 x 32 diagonal blocks
    {
        const int e = tid;  // 512 threads, 2 blocks x 256 entries
        const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15, o = 32 * pr;
        T32[(o + r) * TS + o + 16 + c] = 0.f;
    }
    // level 0: the diagonal 16 x 16 blocks, one column per thread
    if (tid < 64) {
        const int blk = tid >> 4, c = tid & 15, o = blk * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc0 = 0.f, acc1 = 0.f;  // two partial sums shorten the dependency chain
#pragma unroll
            for (int s = 0; s < r; s += 2) {
                acc0 = fmaf(A[(o + r) * AS + o + s], x[s], acc0);
                if (s + 1 < r) acc1 = fmaf(A[(o + r) * AS + o + s + 1], x[s + 1], acc1);
            }
            x[r] = (r < c) ? 0.f : (r == c ? 1.f : -(acc0 + acc1));
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T32[(o + r) * TS + o + c] = x[r];
    }
    __syncthreads();
    // level 1, for both 32 x 32 diagonal blocks (o = 0, 32): M = A21 T11 then
    // T21 = -T22 M (16 x 16 each), one 16 x 8 tile per warp (warps 0-3)
    if (warp < 4) {
        const int pr = warp >> 1, n0 = (warp & 1) * 8, o = 32 * pr;
        float *Mp = M + pr * 16 * MS;
        warp_tile_16x8<16>(A + (o + 16) * AS + o, AS, T32 + o * TS + o + n0, TS, Mp + n0, MS, 1.f, lane);
    }
    __syncthreads();
    if (warp < 4) {
        const int pr = warp >> 1, n0 = (warp & 1) * 8, o = 32 * pr;
        const float *Mp = M + pr * 16 * MS;
        warp_tile_16x8<16>(T32 + (o + 16) * TS + o + 16, TS, Mp + n0, MS, T32 + (o + 16) * TS + o + n0, TS, -1.f,
                           lane);
    }
    __syncthreads();
    // level 2: the lower-left 32 x 32 block, one 16 x 8 tile per warp (warps 0-7)
    if (warp < 8) {
        const int m0 = (warp >> 2) * 16, n0 = (warp & 3) * 8;
        warp_tile_16x8<32>(A + (32 + m0) * AS, AS, T32 + n0, TS, M + m0 * MS + n0, MS, 1.f, lane);
    }
    __syncthreads();
    if (warp < 8) {
        const int m0 = (warp >> 2) * 16, n0 = (warp & 3) * 8;
        warp_tile_16x8<32>(T32 + (32 + m0) * TS + 32, TS, M + n0, MS, T32 + (32 + m0) * TS + n0, TS, -1.f, lane);
    }
    __syncthreads();
}

struct Shared {
    float Gam[CH], gam[CH], beta[CH], gate[CH];  // Gam: cumulative log decay in log2 units
    uint64_t bar;   // MMA completion
    uint64_t bar1;  // MMA1 completion (its own barrier: two commits on one barrier before a wait would alias phases)
    uint64_t lbar;  // staged rows of the next chunk
    uint32_t tmem;
    int item;
};

template <typename TIO>
__global__ void __launch_bounds__(NT, 1)
    chunked_kernel(const ForwardParams p, int32_t *ws, const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v) {
    dependent_prologue();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Shared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Tensor memory: a warp reaches only the 32 lanes of its quarter (warp % 4);
    // the four warps of a quarter split the columns.
    const int quarter = warp & 3, cq = warp >> 2;
    const int row = quarter * 32 + lane;  // the tensor-memory lane (matrix row) of this thread
    const uint32_t lane_sel = (uint32_t)(quarter * 32) << 16;
    const int c16 = cq * 16;  // this thread's 16 columns of a 64-column region
    const int c32 = cq * 32;  // this thread's 32 columns of a 128-column region

    float *V_s = reinterpret_cast<float *>(sm + OFF_V);
    float *A32 = reinterpret_cast<float *>(sm + OFF_A32);
    float *T32 = reinterpret_cast<float *>(sm + OFF_T32);
    float *Mws = reinterpret_cast<float *>(sm + OFF_M);
    const uint32_t a_QKG = ptx::smem_u32(sm + OFF_QKG);
    const uint32_t a_S16 = ptx::smem_u32(sm + OFF_S16);
    const uint32_t a_RT = ptx::smem_u32(sm + OFF_RT), a_UD = ptx::smem_u32(sm + OFF_UD);
    const uint32_t a_T = ptx::smem_u32(sm + OFF_T), a_PD = ptx::smem_u32(sm + OFF_PD);

    if (warp == 0) {
        ptx::tmem_alloc(&sh.tmem, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        ptx::mbar_init(&sh.bar, 1);
        ptx::mbar_init(&sh.bar1, 1);
        ptx::mbar_init(&sh.lbar, 1);
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tm = sh.tmem;
    uint32_t phase = 0, phase1 = 0, lphase = 0;
    bool failed = false, load_pending = false;
    constexpr bool STAGED = sizeof(TIO) == 2;
    uint8_t *stg = sm + OFF_STG;

    // waits for the MMAs committed so far; false on time-out (reported, then the CTA stops)
    auto mma_wait = [&]() -> bool {
        const bool ok = ptx::mbar_wait_bounded(&sh.bar, phase, WAIT_LIMIT);
        phase ^= 1u;
        ptx::tc_fence_after();
        return __syncthreads_and(ok);
    };
    auto mma_ready = [&]() {  // make this thread's smem / tmem writes visible to the next MMA
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
    };

    const int n_items = ws[1] * p.Hv;
    const TIO *qg = static_cast<const TIO *>(p.q);
    const TIO *kg = static_cast<const TIO *>(p.k);
    const TIO *vg = static_cast<const TIO *>(p.v);
    TIO *og = static_cast<TIO *>(p.out);
    const long long ubase = (long long)p.Hv + (long long)p.Hk * DH;

    while (!failed) {
        if (tid == 0) sh.item = atomicAdd(&ws[0], 1);
        __syncthreads();
        const int item = sh.item;
        __syncthreads();
        if (item >= n_items) break;
        const int b = ws[2 + item / p.Hv], h = item % p.Hv, kh = h / p.r;
        const int bos = seq_start(p.cu, p.dense_S, b), eos = seq_start(p.cu, p.dense_S, b + 1);
        const int slot = p.slots ? p.slots[b] : b;
        if (slot < 0 || slot >= p.num_slots) {
            if (tid == 0 && h == 0) flag_error(p.status, GDN_DEVERR_STATE_SLOT);
            continue;
        }
        const size_t head_off = ((size_t)slot * p.Hv + h) * (size_t)DH * DH;
        const bool has_init = p.init != nullptr;

        // TMA copies of the q, k, v rows of the chunk starting at token tc into
        // the staging area (row s of tensor j at stg + j*16 KiB + s*256 B); rows
        // past the sequence are loaded (or zero-filled past T) and ignored.
        auto prefetch = [&](int tc) {
            if (tid == 0) {
                ptx::mbar_arrive_expect_tx(&sh.lbar, (uint32_t)(3 * CH * DH * 2));
                ptx::tma_load_2d(stg, &map_q, kh * DH, tc, &sh.lbar);
                ptx::tma_load_2d(stg + CH * DH * 2, &map_k, kh * DH, tc, &sh.lbar);
                ptx::tma_load_2d(stg + 2 * CH * DH * 2, &map_v, h * DH, tc, &sh.lbar);
            }
        };
        // raw gate inputs of the chunk starting at tc, two tokens per lane of warp 0
        float ga[2] = {0.f, 0.f}, gb[2] = {0.f, 0.f};
        auto prefetch_gates = [&](int tc) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const long long t = tc + lane + 32 * u;
                if (t < eos) {
                    ga[u] = p.a[t * p.Hv + h];
                    gb[u] = p.b[t * p.Hv + h];
                }
            }
        };
        if (STAGED && bos < eos) {
            prefetch(bos);
            load_pending = true;
        }
        // Gates of the chunk starting at tc (warp 0, two tokens per lane) from
        // the prefetched raw inputs ga/gb, then the raw inputs of the chunk after
        // it: effective decay, beta, and the within-chunk cumulative log decay.
        // per-head gate parameters, loaded once per chain
        const float expA = (warp == 0 && p.gate_raw) ? expf(p.A_log[h]) : 0.f;
        const float dtb = (warp == 0 && p.gate_raw) ? p.dt_bias[h] : 0.f;
        auto chunk_gates = [&](int tc) {
            const int nn = min(CH, eos - tc);
            float lg[2], bt[2], gt[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int s = lane + 32 * u;
                lg[u] = 0.f; bt[u] = 0.f; gt[u] = 1.f;
                if (s < nn) {
                    const float av = ga[u], bv = gb[u];
                    if (p.gate_raw) {
                        const float l = -expA * softplus_f(av + dtb);
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
            if (tc + CH < eos) prefetch_gates(tc + CH);  // in flight until this is called again
            float c0 = lg[0], c1 = lg[1];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y0 = __shfl_up_sync(0xffffffffu, c0, o);
                const float y1 = __shfl_up_sync(0xffffffffu, c1, o);
                if (lane >= o) { c0 += y0; c1 += y1; }
            }
            c1 += __shfl_sync(0xffffffffu, c0, 31);
            sh.Gam[lane] = c0 * LOG2E;  // log2 units: every decay factor below is one ex2
            sh.Gam[lane + 32] = c1 * LOG2E;
            sh.gam[lane] = expf(c0);
            sh.gam[lane + 32] = expf(c1);
            sh.beta[lane] = bt[0];
            sh.beta[lane + 32] = bt[1];
            sh.gate[lane] = gt[0];
            sh.gate[lane + 32] = gt[1];
            if (p.caps) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int s = lane + 32 * u, tl = tc + s - bos;
                    if (s < nn && tl < p.cap) p.caps[((long long)b * p.cap + tl) * p.W + h] = gt[u];
                }
            }
        };
        if (warp == 0 && bos < eos) {
            prefetch_gates(bos);
            chunk_gates(bos);  // the first chunk's; later chunks' are computed during the previous chunk
        }

        // ---- chain start: the initial state into tensor memory
        if (has_init) {
            const float *src = p.init + head_off + (size_t)row * DH + c32;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(src + j);
                v[j] = x.x; v[j + 1] = x.y; v[j + 2] = x.z; v[j + 3] = x.w;
            }
            ptx::tmem_st32(tm + lane_sel + TM_S + c32, v);
            ptx::tmem_st_wait();
        }
        bool state_live = has_init;  // does TM_S hold the state (else it is zero)?

        for (int t0 = bos; t0 < eos && !failed; t0 += CH) {
            const int n = min(CH, eos - t0);
            // ---- A1: (the gates of this chunk were computed by warp 0 during the
            //      previous chunk's last MMA wait, or at the chain start)
            if (STAGED) {
                const bool ok = ptx::mbar_wait_bounded(&sh.lbar, lphase, WAIT_LIMIT);
                lphase ^= 1u;
                load_pending = false;
                if (!__syncthreads_and(ok)) { failed = true; break; }
            }
            // ---- A2: v rows (fp32) of the chunk
            for (int e = tid; e < CH * (DH / 4); e += NT) {
                const int s = e >> 5, c4 = (e & 31) * 4;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (s < n) {
                    if (STAGED)
                        ld4<TIO>(reinterpret_cast<const TIO *>(stg + 2 * CH * DH * 2 + s * DH * 2) + c4, v);
                    else
                        ld4<TIO>(vg + (long long)(t0 + s) * p.v_stride + (long long)h * DH + c4, v);
                }
                *reinterpret_cast<float4 *>(V_s + s * DH + c4) = make_float4(v[0], v[1], v[2], v[3]);
            }
            // ---- A3: normalised q and k into the [Q;K;gamma Q] tile; each warp handles
            //      its 4 tokens together so their loads and reductions overlap
            {
                constexpr int TPW = CH / (NT / 32);  // tokens per warp
                float qv[TPW][4], kv[TPW][4], sq[TPW], sk[TPW];
#pragma unroll
                for (int u = 0; u < TPW; ++u) {
                    const int s = warp + (NT / 32) * u;
#pragma unroll
                    for (int e = 0; e < 4; ++e) qv[u][e] = kv[u][e] = 0.f;
                    if (s < n) {
                        if (STAGED) {
                            ld4<TIO>(reinterpret_cast<const TIO *>(stg + s * DH * 2) + lane * 4, qv[u]);
                            ld4<TIO>(reinterpret_cast<const TIO *>(stg + CH * DH * 2 + s * DH * 2) + lane * 4, kv[u]);
                        } else {
                            const long long t = t0 + s;
                            ld4<TIO>(qg + t * p.q_stride + (long long)kh * DH + lane * 4, qv[u]);
                            ld4<TIO>(kg + t * p.k_stride + (long long)kh * DH + lane * 4, kv[u]);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < TPW; ++u) {
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
                    for (int u = 0; u < TPW; ++u) {
                        sq[u] += __shfl_xor_sync(0xffffffffu, sq[u], off);
                        sk[u] += __shfl_xor_sync(0xffffffffu, sk[u], off);
                    }
                }
                const int c = lane * 4;
#pragma unroll
                for (int u = 0; u < TPW; ++u) {
                    const int s = warp + (NT / 32) * u;
                    const float iq = 1.f / fmaxf(sqrtf(sq[u]), EPS), ik = 1.f / fmaxf(sqrtf(sk[u]), EPS);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        qv[u][e] *= iq;
                        kv[u][e] *= ik;
                    }
                    st_h4(sm + OFF_QKG, sw(s, c, QKG_ROWS), qv[u][0], qv[u][1], qv[u][2], qv[u][3]);
                    st_h4(sm + OFF_QKG, sw(64 + s, c, QKG_ROWS), kv[u][0], kv[u][1], kv[u][2], kv[u][3]);
                    const int tl = t0 + s - bos;
                    if (p.caps && h % p.r == 0 && s < n && tl < p.cap) {
                        float *dst = p.caps + ((long long)b * p.cap + tl) * p.W + p.Hv + (long long)kh * DH + c;
#pragma unroll
                        for (int e = 0; e < 4; ++e) dst[e] = kv[u][e];
                    }
                }
            }
            __syncthreads();
            // ---- A4: gamma Q (from the fp16 Q rows); the state update reads K from the
            //      K rows as an MN-major operand, so no transposed copy is built
            {
                const uint8_t *kq = sm + OFF_QKG;
#pragma unroll
                for (int it = 0; it < 2; ++it) {
                    const int e = tid + NT * it;       // 64 rows x 16 pieces of 8 elements
                    const int s = e >> 4, k8 = (e & 15) * 8;
                    const uint4 raw = *reinterpret_cast<const uint4 *>(kq + sw(s, k8, QKG_ROWS));
                    const float gm = sh.gam[s];
                    const __half2 *hq = reinterpret_cast<const __half2 *>(&raw);
                    uint4 o;
                    __half2 *ho = reinterpret_cast<__half2 *>(&o);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 f = __half22float2(hq[q]);
                        ho[q] = __floats2half2_rn(gm * f.x, gm * f.y);
                    }
                    *reinterpret_cast<uint4 *>(sm + OFF_QKG + sw(128 + s, k8, QKG_ROWS)) = o;
                }
            }
            // ---- B: S0 -> fp16 operand tile; the tensor-memory state becomes gamma_last S0
            {
                const float gl = sh.gam[n - 1];
                float v[32];
                if (state_live) {
                    ptx::tmem_ld32(tm + lane_sel + TM_S + c32, v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 32; j += 4) st_h4(sm + OFF_S16, sw(row, c32 + j, 128), v[j], v[j + 1], v[j + 2], v[j + 3]);
                if (state_live) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= gl;
                    ptx::tmem_st32(tm + lane_sel + TM_S + c32, v);
                    ptx::tmem_st_wait();
                }
            }
            mma_ready();
            // ---- C: MMA1 (committed on its own, so the inverse can start while
            //      MMA2 still runs) and MMA2
            if (tid == 0) {
                ptx::tc_fence_after();
                const uint32_t i64 = ptx::idesc_f16_f32(128, 64);
                const uint32_t i128 = ptx::idesc_f16_f32(128, 128);
                for (int ks = 0; ks < DH / 16; ++ks) {
                    const uint32_t ko = (ks >> 2) * QKG_KB + (ks & 3) * 32;
                    ptx::mma_f16(tm + TM_D1, ptx::sdesc_k_sw128(a_QKG + ko),
                                 ptx::sdesc_k_sw128(a_QKG + 64 * 128 + ko), i64, ks > 0);
                }
                ptx::mma_commit(&sh.bar1);
                for (int ks = 0; ks < DH / 16; ++ks) {
                    const uint32_t ko = (ks >> 2) * QKG_KB + (ks & 3) * 32;
                    ptx::mma_f16(tm + TM_X, ptx::sdesc_k_sw128(a_S16 + (ks >> 2) * 16384 + (ks & 3) * 32),
                                 ptx::sdesc_k_sw128(a_QKG + 64 * 128 + ko), i128, ks > 0);  // X and S0 (gamma Q)^T
                }
                ptx::mma_commit(&sh.bar);
            }
            {
                const bool ok = ptx::mbar_wait_bounded(&sh.bar1, phase1, WAIT_LIMIT);
                phase1 ^= 1u;
                ptx::tc_fence_after();
                if (!__syncthreads_and(ok)) { failed = true; break; }
            }
            // ---- D1: A (fp32 staging) and P o D (fp16 tile) from G and P
            {
                float v[16];
                ptx::tmem_ld16(tm + lane_sel + TM_D1 + c16, v);
                const int r = row & 63;
                const float Gr = sh.Gam[r];
                if (quarter >= 2) {  // lanes 64-127: G
                    const float br = sh.beta[r];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s = c16 + j;
                        A32[r * AS + s] = (s < r) ? br * ex2_approx(Gr - sh.Gam[s]) * v[j] : 0.f;
                    }
                } else {  // lanes 0-63: P
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        float w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s = c16 + j + e;
                            w[e] = (s <= r) ? v[j + e] * ex2_approx(Gr - sh.Gam[s]) : 0.f;
                        }
                        st_h4(sm + OFF_PD, sw(r, c16 + j, 64), w[0], w[1], w[2], w[3]);
                    }
                }
            }
            __syncthreads();
            // ---- D2: T = (I + A)^-1 on the CUDA cores, then its fp16 tile
            tri_inverse(A32, T32, Mws, tid);
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int e = tid + NT * it;
                const int r = e >> 4, s0 = (e & 15) * 4;
                const float4 w = (r < 32 && s0 >= 32) ? make_float4(0.f, 0.f, 0.f, 0.f)  // upper-right quadrant
                                                      : *reinterpret_cast<const float4 *>(T32 + r * TS + s0);
                st_h4(sm + OFF_T, sw(r, s0, 64), w.x, w.y, w.z, w.w);
            }
            // ---- D2w: wait for MMA2
            if (!mma_wait()) { failed = true; break; }
            // the staging area is free again: fetch the next chunk while this one finishes
            if (STAGED && t0 + CH < eos) {
                prefetch(t0 + CH);
                load_pending = true;
            }
            // ---- D3: R^T = (V - diag(gamma) K S0^T)^T diag(beta) from X^T
            {
                float v[16];
                ptx::tmem_ld16(tm + lane_sel + TM_X + c16, v);
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    float w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s = c16 + j + e;
                        w[e] = sh.beta[s] * (V_s[s * DH + row] - sh.gam[s] * v[j + e]);
                    }
                    st_h4(sm + OFF_RT, sw(row, c16 + j, 128), w[0], w[1], w[2], w[3]);
                }
            }
            mma_ready();
            // ---- E: MMA3  U^T = R^T T^T
            if (tid == 0) {
                ptx::tc_fence_after();
                const uint32_t i64 = ptx::idesc_f16_f32(128, 64);
                for (int ks = 0; ks < CH / 16; ++ks)
                    ptx::mma_f16(tm + TM_D3, ptx::sdesc_k_sw128(a_RT + ks * 32), ptx::sdesc_k_sw128(a_T + ks * 32),
                                 i64, ks > 0);
                ptx::mma_commit(&sh.bar);
            }
            if (!mma_wait()) { failed = true; break; }
            // ---- F: U^T -> fp16 operands (plain and decayed to the chunk end); capsule deltas
            {
                float v[16];
                ptx::tmem_ld16(tm + lane_sel + TM_D3 + c16, v);
                const float Gl = sh.Gam[n - 1];
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    float w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) w[e] = ex2_approx(Gl - sh.Gam[c16 + j + e]) * v[j + e];
                    st_h4(sm + OFF_RT, sw(row, c16 + j, 128), v[j], v[j + 1], v[j + 2], v[j + 3]);
                    st_h4(sm + OFF_UD, sw(row, c16 + j, 128), w[0], w[1], w[2], w[3]);
                }
                if (p.caps) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s = c16 + j, tl = t0 + s - bos;
                        if (s < n && tl < p.cap)
                            p.caps[((long long)b * p.cap + tl) * p.W + ubase + (long long)h * DH + row] = v[j];
                    }
                }
            }
            mma_ready();
            // ---- G: MMA4 (output) and MMA5 (state)
            if (tid == 0) {
                ptx::tc_fence_after();
                const uint32_t i64 = ptx::idesc_f16_f32(128, 64), i128_bmn = ptx::idesc_f16_f32(128, 128, true);
                for (int ks = 0; ks < CH / 16; ++ks) {
                    ptx::mma_f16(tm + TM_O, ptx::sdesc_k_sw128(a_RT + ks * 32), ptx::sdesc_k_sw128(a_PD + ks * 32),
                                 i64, 1u);
                    // K rows (64..127) of the [Q;K;gamma Q] tile as MN-major B: 16 tokens = 2048 B per step
                    ptx::mma_f16(tm + TM_S, ptx::sdesc_k_sw128(a_UD + ks * 32),
                                 ptx::sdesc_mn_sw128(a_QKG + 64 * 128 + ks * 2048, QKG_KB),
                                 i128_bmn, (state_live || ks > 0) ? 1u : 0u);
                }
                ptx::mma_commit(&sh.bar);
            }
            // the next chunk's gates while MMA4/5 run (nothing reads them after F)
            if (warp == 0 && t0 + CH < eos) chunk_gates(t0 + CH);
            if (!mma_wait()) { failed = true; break; }
            state_live = true;
            // ---- H: outputs, staged through shared memory (the v tile is free) and
            //      written as contiguous 16-byte pieces of each token's dv row
            {
                float v[16];
                ptx::tmem_ld16(tm + lane_sel + TM_O + c16, v);
                TIO *ost = reinterpret_cast<TIO *>(sm + OFF_V);
#pragma unroll
                for (int j = 0; j < 16; ++j) ost[(c16 + j) * DH + row] = from_f32<TIO>(p.scale * v[j]);
                __syncthreads();
                constexpr int VEC = 16 / sizeof(TIO);  // elements per 16-byte piece
                for (int e = tid; e < n * (DH / VEC); e += NT) {
                    const int r = e / (DH / VEC), c = (e % (DH / VEC)) * VEC;
                    *reinterpret_cast<uint4 *>(og + ((long long)(t0 + r) * p.Hv + h) * DH + c) =
                        *reinterpret_cast<const uint4 *>(ost + r * DH + c);
                }
            }
            ptx::tc_fence_before();
            __syncthreads();
            ptx::tc_fence_after();
        }
        if (failed) break;
        // ---- chain end: the final state (unless the caller asked for none)
        if (p.final_state) {
            float *dst = p.final_state + head_off + (size_t)row * DH + c32;
            float v[32];
            if (state_live) {
                ptx::tmem_ld32(tm + lane_sel + TM_S + c32, v);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
    }

    if (failed && tid == 0) {
        flag_error(p.status, GDN_DEVERR_TIMEOUT);
        ptx::mbar_wait_bounded(&sh.bar, phase ^ 1u, WAIT_LIMIT);  // let in-flight MMAs drain
        ptx::mbar_wait_bounded(&sh.bar, phase, WAIT_LIMIT);
        ptx::mbar_wait_bounded(&sh.bar1, phase1 ^ 1u, WAIT_LIMIT);
        if (load_pending) ptx::mbar_wait_bounded(&sh.lbar, lphase, WAIT_LIMIT);  // and staged copies
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tm, TMEM_COLS);
    }
}

// Builds the chain list: ws[0] = 0 (work counter), ws[1] = number of
// sequences on this path, ws[2..] = those sequences, longest first (counting
// sort on the number of chunks).  Sequences with a bad packing are left out
// (the recurrent kernel reports them).
constexpr int PLAN_BINS = 1024;
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t *cu, int dense_S, int B, int T, int min_len,
                                                    int32_t *ws, int32_t *status) {
    dependent_prologue();
    __shared__ int hist[PLAN_BINS];
    __shared__ int total;
    const int tid = threadIdx.x;
    for (int i = tid; i < PLAN_BINS; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    auto key = [&](int b) -> int {
        const int lo = seq_start(cu, dense_S, b), hi = seq_start(cu, dense_S, b + 1);
        if (lo < 0 || hi < lo || hi > T || hi - lo <= min_len) return -1;
        const int chunks = min((hi - lo + CH - 1) / CH, PLAN_BINS - 1);
        return PLAN_BINS - 1 - chunks;  // descending length
    };
    // a packing error is flagged here too: under the forced chunked plan no other
    // kernel sees the batch
    if (tid == 0 && cu && (cu[0] != 0 || cu[B] != T)) flag_error(status, GDN_DEVERR_CU_SEQLENS);
    for (int b = tid; b < B; b += blockDim.x) {
        const int lo = seq_start(cu, dense_S, b), hi = seq_start(cu, dense_S, b + 1);
        if (lo < 0 || hi < lo || hi > T) flag_error(status, GDN_DEVERR_CU_SEQLENS);
        const int k = key(b);
        if (k >= 0) atomicAdd(&hist[k], 1);
    }
    __syncthreads();
    if (tid == 0) {  // exclusive scan (1024 bins, once per call)
        int run = 0;
        for (int i = 0; i < PLAN_BINS; ++i) {
            const int c = hist[i];
            hist[i] = run;
            run += c;
        }
        total = run;
    }
    __syncthreads();
    for (int b = tid; b < B; b += blockDim.x) {
        const int k = key(b);
        if (k >= 0) ws[2 + atomicAdd(&hist[k], 1)] = b;
    }
    if (tid == 0) {
        ws[0] = 0;
        ws[1] = total;
    }
}

int num_sms() { return current_device_sms(); }

template <typename TIO>
cudaError_t launch_io(const ForwardParams &p, int min_len, int32_t *ws, cudaStream_t stream) {
    CUtensorMap mq{}, mk{}, mv{};
    if (sizeof(TIO) == 2 && p.T > 0) {  // (no tokens: no chunk reads q, k or v)
        if (!encode_rows_f16(&mq, p.q, (long long)p.Hk * DH, p.q_stride, p.T, DH, CH, false) ||
            !encode_rows_f16(&mk, p.k, (long long)p.Hk * DH, p.k_stride, p.T, DH, CH, false) ||
            !encode_rows_f16(&mv, p.v, (long long)p.Hv * DH, p.v_stride, p.T, DH, CH, false))
            return cudaErrorInvalidValue;
    }
    cudaError_t e =
        launch_dependent(plan_kernel, dim3(1), dim3(1024), 0, stream, p.cu, p.dense_S, p.B, p.T, min_len, ws, p.status);
    if (e != cudaSuccess) return e;
    auto kern = chunked_kernel<TIO>;
    constexpr int smem = SMEM_ALLOC;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long chains = (long long)p.B * p.Hv;
    const int grid = (int)(chains < num_sms() ? chains : num_sms());
    return launch_dependent(kern, dim3(grid), dim3(NT), smem, stream, p, ws, mq, mk, mv);
}

}  // namespace

// cuTensorMapEncodeTiled from the driver, looked up once.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool encode_rows_f16(CUtensorMap *map, const void *base, long long row_elems, long long stride, int T, int box_x,
                     int box_y, bool swizzle128) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)(T > 0 ? T : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)box_y};
    const cuuint32_t estride[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_f32(CUtensorMap *map, const float *base, long long row_elems, long long rows, int box_x, int box_y,
                     bool swizzle128) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)row_elems * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)box_y};
    const cuuint32_t estride[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_state_tiles(CUtensorMap *map, const float *base, int d, long long rows, int box_rows) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    // [rows, d] viewed as (32 features, rows, d / 32 feature blocks): one box of
    // box_rows rows lands as d / 32 consecutive 128-byte swizzled tiles
    const cuuint64_t dims[3] = {32, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)(d / 32)};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 4, 128};
    const cuuint32_t box[3] = {32, (cuuint32_t)box_rows, (cuuint32_t)(d / 32)};
    const cuuint32_t estride[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_f32_strided(CUtensorMap *map, const float *base, long long row_elems, long long stride, int T,
                             int box_x, int box_y) {
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)(T > 0 ? T : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)stride * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)box_y};
    const cuuint32_t estride[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t chunked_workspace_bytes(int B) { return ((size_t)(B + 2) * sizeof(int32_t) + 255) & ~size_t(255); }

bool chunked_supported(int dk, int dv) { return dk == DH && dv == DH; }

cudaError_t launch_chunked(const ForwardParams &p, int min_len, void *workspace, cudaStream_t stream) {
    if (p.B == 0) return cudaSuccess;
    int32_t *ws = static_cast<int32_t *>(workspace);
    return p.io_f16 ? launch_io<__half>(p, min_len, ws, stream) : launch_io<float>(p, min_len, ws, stream);
}

}  // namespace gdn
