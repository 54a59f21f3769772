// prepack.cu -- the scale prepack kernel.
//
// Layout (page 4, submission 482006, `to_blocked_gpu`, and the same page's
// layout atom with shape ((32,4),(16,4)) and strides ((16,4),(0,1))):
//  - zero-pad the rows to a multiple of 128 and the columns to a multiple of 4;
//  - cut the result into 128 x 4 blocks of 512 bytes, row-tile major, column
//    blocks inner;
//  - inside a block, row 32*i + j and column c go to byte 16*j + 4*i + c.
// A 512-byte block is exactly what one `tcgen05.cp .32x128b.warpx4` moves into
// four TMEM columns.
//
// Work split. The kernel only moves bytes, so it is bound by HBM bandwidth and
// by how many bytes are in flight. A work item is one warp's: a 128-row tile of
// one operand and 32 of its source columns (8 output blocks). Lane j loads 32
// bytes (two 16-byte words, one whole 32-byte sector) from each of rows j,
// j + 32, j + 64 and j + 96 of the tile, all eight loads before any use, then
// transposes them in registers: output row j of block b is the four 4-byte
// words of column group b from those four rows, so it writes one 16-byte word
// per block and a warp's store fills a whole 512-byte block. No shared memory
// and no barrier: every warp of the launch has its loads in flight at once, and
// a launch is a single wave for any realistic set of operands.
// Operands whose rows are not a multiple of 16 bytes (K % 256 != 0) take the
// byte path: 16 source columns per item, loaded byte by byte, same stores.
#include "prepack.cuh"

#include <algorithm>
#include <climits>

namespace nvfp4 {

struct PrepackBatch {
    PrepackJob job[kPrepackMaxJobs];
    int32_t n;
};

constexpr int kPrepackThreads = 256;  // 8 warps, one work item each
constexpr int kPrepackWarps = kPrepackThreads / 32;

__device__ __forceinline__ uint4 pick_words(const uint4 (&w)[4], int k)
{
    // word k of each of the four rows: the 16-byte output row of column block k
    switch (k) {
    case 0: return make_uint4(w[0].x, w[1].x, w[2].x, w[3].x);
    case 1: return make_uint4(w[0].y, w[1].y, w[2].y, w[3].y);
    case 2: return make_uint4(w[0].z, w[1].z, w[2].z, w[3].z);
    default: return make_uint4(w[0].w, w[1].w, w[2].w, w[3].w);
    }
}

__global__ void __launch_bounds__(kPrepackThreads) prepack_scales_kernel(const __grid_constant__ PrepackBatch batch,
                                                                         int total_items)
{
    const int item = (int)blockIdx.x * kPrepackWarps + (int)(threadIdx.x >> 5);
    if (item >= total_items)
        return;
    const int j = (int)(threadIdx.x & 31);
    int jn = 0;
    while (jn + 1 < batch.n && item >= batch.job[jn + 1].item_begin)
        ++jn;
    const PrepackJob &J = batch.job[jn];
    const int local = item - J.item_begin;
    const int rt = local / J.units, u = local % J.units;
    const int r0 = rt * 128 + j;
    // output row j of this tile's blocks
    uint8_t *dst = J.dst + (size_t)rt * J.col_blocks * 512 + 16 * j;

    if (J.vec) {
        // columns 32u .. 32u + 31: one or two 16-column pieces, 4 blocks each
        const int pieces = min(2, J.cols / 16 - 2 * u);
        uint4 w[2][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + 32 * i;
            const uint4 *src = reinterpret_cast<const uint4 *>(J.src + (size_t)r * J.cols + 32 * u);
            const bool row_in = r < J.rows;
            w[0][i] = row_in ? __ldcs(src) : make_uint4(0, 0, 0, 0);
            w[1][i] = (row_in && pieces > 1) ? __ldcs(src + 1) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            if (p < pieces) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4 *>(dst + (size_t)(8 * u + 4 * p + k) * 512) = pick_words(w[p], k);
            }
        }
    } else {
        // columns 16u .. 16u + 15 byte by byte, zero past the matrix (the padding columns
        // of the last block included)
        uint4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + 32 * i;
            uint32_t word[4] = {0, 0, 0, 0};
            if (r < J.rows) {
                const uint8_t *src = J.src + (size_t)r * J.cols;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int col = 16 * u + c;
                    if (col < J.cols)
                        word[c >> 2] |= (uint32_t)src[col] << (8 * (c & 3));
                }
            }
            w[i] = make_uint4(word[0], word[1], word[2], word[3]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b = 4 * u + k;
            if (b < J.col_blocks)
                *reinterpret_cast<uint4 *>(dst + (size_t)b * 512) = pick_words(w, k);
        }
    }
}

cudaError_t launch_prepack(PrepackJob *jobs, int n, cudaStream_t stream)
{
    int k = 0;
    while (k < n) {
        PrepackBatch b{};
        b.n = 0;
        long long items = 0;
        // up to kPrepackMaxJobs jobs per launch, and few enough items for int indexing
        for (; k < n && b.n < kPrepackMaxJobs; ++k) {
            PrepackJob J = jobs[k];
            if (J.rows <= 0 || J.cols <= 0)
                continue;
            J.vec = (J.cols % 16 == 0) && (reinterpret_cast<uintptr_t>(J.src) % 16 == 0);
            J.col_blocks = (J.cols + 3) / 4;
            J.units = J.vec ? (J.cols + 31) / 32 : (J.cols + 15) / 16;
            const long long mine = (long long)((J.rows + 127) / 128) * J.units;
            if (mine > INT_MAX / 2)
                return cudaErrorInvalidValue;
            if (items + mine > INT_MAX / 2)
                break;  // this job opens the next launch
            J.item_begin = (int32_t)items;
            items += mine;
            b.job[b.n++] = J;
        }
        if (b.n == 0)
            continue;
        const long long grid = (items + kPrepackWarps - 1) / kPrepackWarps;
        prepack_scales_kernel<<<(unsigned)grid, kPrepackThreads, 0, stream>>>(b, (int)items);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace nvfp4
