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
// Work split. One CTA per (128-row tile, 8 column blocks). Its 256 threads first
// load the 128 x 32-byte source tile into shared memory (reads coalesced along
// each row). Then each thread writes one 16-byte row of a 512-byte block, so
// consecutive threads write consecutive 16 bytes. The kernel moves bytes and
// is bound by HBM bandwidth.
#include "prepack.cuh"

namespace nvfp4 {

struct PrepackBatch {
    PrepackJob job[kPrepackMaxJobs];
    int32_t n;
};

__global__ void __launch_bounds__(256) prepack_scales_kernel(const __grid_constant__ PrepackBatch batch)
{
    __shared__ uint8_t tile[128][36];  // 32 bytes per row + 4 padding (keeps rows 4-byte aligned, spreads banks)
    int j = 0;
    while (j + 1 < batch.n && (int)blockIdx.x >= batch.job[j + 1].cta_begin)
        ++j;
    const PrepackJob &J = batch.job[j];
    const int local = (int)blockIdx.x - J.cta_begin;
    const int rt = local / J.chunks, ch = local % J.chunks;
    const int c0 = ch * 32;  // first source column of this CTA (8 blocks x 4 columns)

    for (int i = threadIdx.x; i < 128 * 32; i += 256) {
        const int r = i / 32, c = i % 32;
        const int gr = rt * 128 + r, gc = c0 + c;
        tile[r][c] = (gr < J.rows && gc < J.cols) ? J.src[(size_t)gr * J.cols + gc] : (uint8_t)0;
    }
    __syncthreads();

    const int cb = threadIdx.x / 32, jj = threadIdx.x % 32;  // block within the chunk, row within the block
    const int gcb = ch * 8 + cb;
    if (gcb < J.col_blocks) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = *reinterpret_cast<const uint32_t *>(&tile[i * 32 + jj][cb * 4]);
        uint8_t *dst = J.dst + ((size_t)rt * J.col_blocks + gcb) * 512 + jj * 16;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
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
            J.chunks = (J.col_blocks + 7) / 8;
            J.cta_begin = ctas;
            ctas += ((J.rows + 127) / 128) * J.chunks;
            b.job[b.n++] = J;
        }
        if (b.n == 0)
            continue;
        prepack_scales_kernel<<<ctas, 256, 0, stream>>>(b);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace nvfp4
