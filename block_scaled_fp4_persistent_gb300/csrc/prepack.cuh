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
    int32_t units;       // warp work items per 128-row tile: 32 source columns each (16 on the byte path)
    int32_t item_begin;  // first work item of this job within the launch
    int32_t vec;         // 1: 16-byte loads (cols % 16 == 0 and src 16-byte aligned); 0: byte loads
};

constexpr int kPrepackMaxJobs = 32;

// Fills in col_blocks/units/item_begin/vec and launches one kernel for up to
// kPrepackMaxJobs jobs (more are split into several launches).
cudaError_t launch_prepack(PrepackJob *jobs, int n, cudaStream_t stream);

inline size_t blocked_scale_bytes(int rows, int cols)
{
    if (rows <= 0 || cols <= 0)
        return 0;
    return (size_t)((rows + 127) / 128) * 128 * (size_t)((cols + 3) / 4) * 4;
}

}  // namespace nvfp4
