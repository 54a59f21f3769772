// table.h -- the device-side problem table read by the grouped GEMM kernel.
//
// The host builds one table per distinct problem set and uploads it once.
// The table lives in one device buffer:
//
//   [TableHeader (128 B)] [GroupEntry x num_groups] [uint32 cta_begin[grid+1]] [WorkItem x num_items]
//
// Each GroupEntry holds the group's two TMA tensor maps (A and B), its scale and
// output pointers and its sizes. CTA c processes work items
// cta_begin[c] .. cta_begin[c+1]-1 in order. Each item is one 128 x BLOCK_N
// output tile of one group.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace nvfp4 {

constexpr int kStatusTimeout = -5;  // NVFP4_ERR_TIMEOUT

struct alignas(128) GroupEntry {
    CUtensorMap tmap_a;   // uint8 [M][K/2], box 128 B x 128 rows, 128-byte swizzle
    CUtensorMap tmap_b;   // uint8 [N][K/2], box 128 B x BLOCK_N rows, 128-byte swizzle
    const uint8_t *sfa;   // blocked scales of A: ceil(M/128) x kblocks64 blocks of 512 B
    const uint8_t *sfb;   // blocked scales of B: ceil(N/128) x kblocks64 blocks of 512 B
    __half *C;            // [M][N] fp16
    int32_t M, N, K;
    int32_t kblocks64;    // K / 64
    int32_t tiles_m, tiles_n;
};

struct WorkItem {
    int32_t group;
    int32_t tile_m;
    int32_t tile_n;
    int32_t reserved;
};

struct alignas(128) TableHeader {
    int32_t num_groups;
    int32_t num_items;
    int32_t grid;
    int32_t block_n;
    uint32_t off_cta_begin;  // byte offsets from the table's start
    uint32_t off_items;
    uint32_t total_bytes;
};

struct Table {
    TableHeader h;
    __host__ __device__ const GroupEntry &group(int g) const
    {
        return reinterpret_cast<const GroupEntry *>(reinterpret_cast<const char *>(this) + sizeof(TableHeader))[g];
    }
    __host__ __device__ uint32_t cta_begin(int c) const
    {
        return reinterpret_cast<const uint32_t *>(reinterpret_cast<const char *>(this) + h.off_cta_begin)[c];
    }
    __host__ __device__ WorkItem item(uint32_t i) const
    {
        const int4 v = reinterpret_cast<const int4 *>(reinterpret_cast<const char *>(this) + h.off_items)[i];
        return WorkItem{v.x, v.y, v.z, v.w};
    }
    int num_groups_host() const { return h.num_groups; }
};

struct KernelArgs {
    const Table *table;
    int *status;            // 4 words: code, role, item, stage
    uint64_t timeout_ns;    // bound of every wait
    int32_t fault_skip_load;  // -1 off; else CTA 0 skips the copies of that k-stage
    int32_t num_groups;
    int32_t prefetch_stages;  // L2 prefetch distance of the producer, in stages (0 = none)
};

}  // namespace nvfp4
