// prepack.cuh -- scale-factor relayout from row-major [rows][K/16] E4M3 bytes
// to the 128 x 4 blocked layout that tcgen05.cp reads (declarations).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace nvfp4 {

struct PrepackJob {
    const uint8_t *src;  // row-major [rows][cols]
    uint8_t *dst;        // blocked, 128*ceil(rows/128) * 4*ceil(cols/4) bytes, 16-byte aligned
    int32_t rows;
    int32_t cols;        // K / 16
    int32_t col_blocks;  // ceil(cols / 4): 512-byte blocks per 128-row tile
    int32_t chunks;      // ceil(col_blocks / 8): CTAs per 128-row tile
    int32_t cta_begin;   // first CTA of this job within the launch
};

constexpr int kPrepackMaxJobs = 32;

// Fills in col_blocks/chunks/cta_begin and launches one kernel for up to
// kPrepackMaxJobs jobs (more are split into several launches).
cudaError_t launch_prepack(PrepackJob *jobs, int n, cudaStream_t stream);

inline size_t blocked_scale_bytes(int rows, int cols)
{
    if (rows <= 0 || cols <= 0)
        return 0;
    return (size_t)((rows + 127) / 128) * 128 * (size_t)((cols + 3) / 4) * 4;
}

}  // namespace nvfp4
