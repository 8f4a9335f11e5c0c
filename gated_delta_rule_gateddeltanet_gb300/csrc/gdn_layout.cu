// Conversion between the two recurrent-state layouts of the GatedDeltaNet
// operator.
//
// Source: "Add GatedDeltaNet evaluation export for Qwen hybrid models" (review
// of the Qwen builder): the dense export keeps the recurrent state K-major,
// [B, heads, key_dim, value_dim], while the packed operator keeps it V-major,
// [B, heads, value_dim, key_dim].  Converting one to the other is a transpose
// of every (slot, head) matrix; this library's kernels read and write the
// V-major form.
//
// The transpose is HBM-bound (one read and one write of every element): a
// CTA moves a 32 x 32 tile through shared memory (row stride 33, so both the
// column reads and the row writes are conflict-free), each thread 4 elements,
// reads and writes coalesced along the 128-byte rows of source and
// destination.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int TILE = 32, ROWS_PER_PASS = 8;

__global__ void __launch_bounds__(TILE * ROWS_PER_PASS) transpose_kernel(const float *__restrict__ src,
                                                                         float *__restrict__ dst, int rows, int cols,
                                                                         int tiles_c) {
    dependent_prologue();
    __shared__ float tile[TILE][TILE + 1];
    const long long m = blockIdx.y;  // matrix index
    const int tr = blockIdx.x / tiles_c, tc = blockIdx.x % tiles_c;
    const float *s = src + m * rows * cols;
    float *d = dst + m * rows * cols;
    const int c = tc * TILE + threadIdx.x;
#pragma unroll
    for (int i = 0; i < TILE; i += ROWS_PER_PASS) {
        const int r = tr * TILE + threadIdx.y + i;
        if (r < rows && c < cols) tile[threadIdx.y + i][threadIdx.x] = s[(long long)r * cols + c];
    }
    __syncthreads();
    // destination is cols x rows: its row index is the source column
    const int dc = tr * TILE + threadIdx.x;
#pragma unroll
    for (int i = 0; i < TILE; i += ROWS_PER_PASS) {
        const int dr = tc * TILE + threadIdx.y + i;
        if (dr < cols && dc < rows) d[(long long)dr * rows + dc] = tile[threadIdx.x][threadIdx.y + i];
    }
}

}  // namespace

cudaError_t launch_transpose(const float *src, float *dst, long long num, int rows, int cols, cudaStream_t stream) {
    if (num == 0 || rows == 0 || cols == 0) return cudaSuccess;
    const int tiles_r = (rows + TILE - 1) / TILE, tiles_c = (cols + TILE - 1) / TILE;
    // grid.y is limited to 65535: large batches go in several launches
    for (long long m0 = 0; m0 < num; m0 += 65535) {
        const long long n = num - m0 < 65535 ? num - m0 : 65535;
        dim3 grid((unsigned)(tiles_r * tiles_c), (unsigned)n);
        const cudaError_t e = launch_dependent(transpose_kernel, grid, dim3(TILE, ROWS_PER_PASS), 0, stream,
                                               src + m0 * rows * cols, dst + m0 * rows * cols, rows, cols, tiles_c);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gdn
