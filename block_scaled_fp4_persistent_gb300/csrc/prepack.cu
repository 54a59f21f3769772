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
// Work split. A tile is (128-row tile, up to 128 source columns = 32 blocks) of
// one operand; persistent CTAs walk the tiles of every operand of the launch. The
// kernel moves bytes and is bound by HBM bandwidth, so both sides move 16 bytes per
// access, and a CTA's next tile's loads are in flight while it writes the current one:
//  1. the CTA reads its 128 x 128-byte source tile with 16-byte loads (eight
//     threads per 128-byte row segment; narrower loads only when rows are not
//     16-byte aligned), into shared memory;
//  2. each thread then assembles whole 16-byte rows of the output blocks (four
//     4-byte words from rows j, j+32, j+64, j+96 of the tile) and stores them,
//     so a warp writes 512 contiguous bytes: one whole block.
// Shared-memory rows are 132 bytes apart, so the 4-byte reads of step 2 (32
// consecutive rows, one column) fall in 32 different banks.
#include "prepack.cuh"

#include <algorithm>

namespace nvfp4 {

struct PrepackBatch {
    PrepackJob job[kPrepackMaxJobs];
    int32_t n;
};

constexpr int kPrepackCols = 128;                    // source columns (bytes) per CTA: 32 blocks
constexpr int kPrepackStride = kPrepackCols + 4;     // shared-memory row pitch
constexpr int kPrepackThreads = 256;

// One tile of one job: its 128-row tile rt and its chunk of 128 source columns.
struct PrepackTile {
    const PrepackJob *J;
    int rt, ch;
};

__device__ __forceinline__ PrepackTile prepack_tile(const PrepackBatch &batch, int t)
{
    int jn = 0;
    while (jn + 1 < batch.n && t >= batch.job[jn + 1].cta_begin)
        ++jn;
    const PrepackJob &J = batch.job[jn];
    const int local = t - J.cta_begin;
    return PrepackTile{&J, local / J.chunks, local % J.chunks};
}

// A thread's four 16-byte source words of a tile (16-byte rows only), zero past the matrix.
__device__ __forceinline__ void prepack_load(const PrepackTile &T, uint4 (&v)[4])
{
    const PrepackJob &J = *T.J;
    const int c0 = T.ch * kPrepackCols, r0 = T.rt * 128;
    const int ncols = min(kPrepackCols, J.cols - c0), nrows = min(128, J.rows - r0);
    const uint8_t *src = J.src + (size_t)r0 * J.cols + c0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = (int)threadIdx.x + k * kPrepackThreads;
        const int r = i >> 3, q = i & 7;
        v[k] = make_uint4(0, 0, 0, 0);
        if (r < nrows && q * 16 < ncols)
            v[k] = __ldcs(reinterpret_cast<const uint4 *>(src + (size_t)r * J.cols + q * 16));
    }
}

// Persistent CTAs walk the tiles of every job of the launch. While a CTA writes one
// tile's blocks it already has the next tile's loads in flight, so reads and writes
// overlap instead of coming in two waves.
__global__ void __launch_bounds__(kPrepackThreads) prepack_scales_kernel(const __grid_constant__ PrepackBatch batch,
                                                                         int total_tiles)
{
    __shared__ __align__(16) uint8_t tile[128 * kPrepackStride];
    int t = (int)blockIdx.x;
    if (t >= total_tiles)
        return;
    PrepackTile cur = prepack_tile(batch, t);
    bool vec16 = ((cur.J->cols & 15) == 0) && ((reinterpret_cast<uintptr_t>(cur.J->src) & 15) == 0);
    uint4 v[4];
    if (vec16)
        prepack_load(cur, v);
    for (;;) {
        const PrepackJob &J = *cur.J;
        const int c0 = cur.ch * kPrepackCols, r0 = cur.rt * 128;
        const int ncols = min(kPrepackCols, J.cols - c0), nrows = min(128, J.rows - r0);
        const int nblk = min(kPrepackCols / 4, J.col_blocks - cur.ch * (kPrepackCols / 4));
        // 1. this tile -> shared memory (rows and columns past the matrix read as zero)
        if (vec16) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = (int)threadIdx.x + k * kPrepackThreads;
                const int r = i >> 3, q = i & 7;
                uint32_t *d = reinterpret_cast<uint32_t *>(tile + r * kPrepackStride + q * 16);
                d[0] = v[k].x, d[1] = v[k].y, d[2] = v[k].z, d[3] = v[k].w;
            }
        } else {
            const uint8_t *src = J.src + (size_t)r0 * J.cols + c0;
            for (int i = threadIdx.x; i < 128 * kPrepackCols; i += kPrepackThreads) {
                const int r = i / kPrepackCols, c = i % kPrepackCols;
                tile[r * kPrepackStride + c] = (r < nrows && c < ncols) ? src[(size_t)r * J.cols + c] : (uint8_t)0;
            }
        }
        __syncthreads();
        // 2. the next tile's loads go out now
        const int tn = t + (int)gridDim.x;
        PrepackTile nxt{};
        bool nvec = false;
        if (tn < total_tiles) {
            nxt = prepack_tile(batch, tn);
            nvec = ((nxt.J->cols & 15) == 0) && ((reinterpret_cast<uintptr_t>(nxt.J->src) & 15) == 0);
            if (nvec)
                prepack_load(nxt, v);
        }
        // 3. whole 16-byte rows of this tile's output blocks: word (block b, row j) = the
        //    four columns of block b in rows j, j + 32, j + 64 and j + 96 of the tile
        uint8_t *dst = J.dst + ((size_t)cur.rt * J.col_blocks + (size_t)cur.ch * (kPrepackCols / 4)) * 512;
        for (int i = threadIdx.x; i < nblk * 32; i += kPrepackThreads) {
            const int b = i >> 5, j = i & 31;
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                w[q] = *reinterpret_cast<const uint32_t *>(tile + (q * 32 + j) * kPrepackStride + b * 4);
            __stcs(reinterpret_cast<uint4 *>(dst + (size_t)b * 512 + j * 16), make_uint4(w[0], w[1], w[2], w[3]));
        }
        if (tn >= total_tiles)
            break;
        __syncthreads();  // the shared tile is read before it is rewritten
        t = tn;
        cur = nxt;
        vec16 = nvec;
    }
}

cudaError_t launch_prepack(PrepackJob *jobs, int n, cudaStream_t stream)
{
    for (int base = 0; base < n; base += kPrepackMaxJobs) {
        PrepackBatch b{};
        b.n = 0;
        int ctas = 0;
        for (int k = base; k < n && k < base + kPrepackMaxJobs; ++k) {
            PrepackJob J = jobs[k];
            if (J.rows <= 0 || J.cols <= 0)
                continue;
            J.col_blocks = (J.cols + 3) / 4;
            J.chunks = (J.cols + kPrepackCols - 1) / kPrepackCols;
            J.cta_begin = ctas;
            ctas += ((J.rows + 127) / 128) * J.chunks;
            b.job[b.n++] = J;
        }
        if (b.n == 0)
            continue;
        // persistent CTAs: about two tiles each on a full device, so that each CTA's
        // second tile's loads overlap its first tile's stores
        static int sms = 0;
        if (sms == 0) {
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                        cudaSuccess || sms <= 0)
                sms = 1;
        }
        const int grid = std::max(1, std::min(ctas, 4 * sms));
        prepack_scales_kernel<<<grid, kPrepackThreads, 0, stream>>>(b, ctas);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace nvfp4
