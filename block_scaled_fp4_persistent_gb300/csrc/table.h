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
    CUtensorMap tmap_c;   // fp16 [M][N], box 32 x 32, 64-byte swizzle (the epilogues' stores)
    // Row-major scales (kItemSfRowMajor): uint8 [M][K/16] and [N][K/16], boxes of 16 B
    // (one K-stage) x 128 rows (A) and x the tile's B rows, no swizzle. For prepacked
    // scales, valid but unused maps of the scale buffers' first 16 bytes.
    CUtensorMap tmap_sfa;
    CUtensorMap tmap_sfb;
    const uint8_t *sfa;   // scales of A: blocked, ceil(M/128) x kblocks64 blocks of 512 B, or row-major
    const uint8_t *sfb;   // scales of B: the same
    __half *C;            // [M][N] fp16
    int32_t M, N, K;
    int32_t kblocks64;    // K / 64
    int32_t tiles_m, tiles_n;
    int32_t sf_rowmajor;  // 1: the scales are row-major, read through tmap_sfa / tmap_sfb
};

// One segment of an output tile: K-stages kb_begin .. kb_end-1 (256 K each).
// A tile that is not split has one segment covering all its K-stages
// (split = -1). A split tile has nseg segments on different CTAs; each writes
// its fp32 partial to workspace slot ws_slot, and the one that finishes last
// (counted in counters[split]) sums the slots ws_slot - seg .. ws_slot - seg +
// nseg - 1 in that order and stores C.
//
// The item also carries what the TMA producer needs before its first copy, so
// that copy waits for one load (the item) rather than a chain of them:
// kblocks64 = K / 64, the scale blocks of the tile's first 128-row tiles of A
// and B, and flags telling whether the second 128-row half of the A tile (CTA
// pairs) and of the B tile (256-wide tiles) holds any rows.
struct WorkItem {
    int32_t group;
    int32_t tile_m;
    int32_t tile_n;
    int32_t kb_begin;
    int32_t kb_end;
    int32_t split;
    int32_t seg;
    int32_t nseg;
    int32_t ws_slot;
    int32_t kblocks64;
    int32_t flags;  // kItemBShared | kItemA2 | kItemB2 | kItemSfRowMajor | a_map << kItemAMapShift
    // Row of the tile's first A row in the A tensor map of group a_map (and, for
    // row-major scales, in its SFA map). Groups whose A rows follow one another in
    // memory share one map (M-fusion): the map of the first group of the run. Read
    // by the pair kernel; the single-CTA kernel's tables are never fused.
    int32_t a_row;
    const uint8_t *sfa;  // scale blocks of the tile's first 128 A rows (kblocks64 blocks of 512 B)
    const uint8_t *sfb;  // scale blocks of the tile's first 128 B rows
};

constexpr int32_t kItemBShared = 1;  // the group has several m-tiles: its B tiles are read more than once
constexpr int32_t kItemA2 = 2;       // rows 128..255 of the tile's A rows exist (their scales follow sfa)
constexpr int32_t kItemB2 = 4;       // rows 128..255 of the tile's B rows exist (their scales follow sfb)
constexpr int32_t kItemSfRowMajor = 8;  // the group's scales are row-major, read through tmap_sfa / tmap_sfb
constexpr int kItemAMapShift = 8;       // flags >> kItemAMapShift: the group whose tmap_a (tmap_sfa) the item reads
constexpr int kMaxGroups = 1 << 23;     // a_map fits the flags' upper bits

static_assert(sizeof(WorkItem) == 64, "WorkItem is read as four int4");

// An item from its four int4 words (the layout of WorkItem).
__host__ __device__ inline WorkItem unpack_item(int4 a, int4 b, int4 c, int4 d)
{
    WorkItem w;
    w.group = a.x, w.tile_m = a.y, w.tile_n = a.z, w.kb_begin = a.w;
    w.kb_end = b.x, w.split = b.y, w.seg = b.z, w.nseg = b.w;
    w.ws_slot = c.x, w.kblocks64 = c.y, w.flags = c.z, w.a_row = c.w;
    w.sfa = reinterpret_cast<const uint8_t *>((uint64_t)(uint32_t)d.x | ((uint64_t)(uint32_t)d.y << 32));
    w.sfb = reinterpret_cast<const uint8_t *>((uint64_t)(uint32_t)d.z | ((uint64_t)(uint32_t)d.w << 32));
    return w;
}

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
    int num_groups_host() const { return h.num_groups; }
};

// Tile lists per launch: one per CTA, or per CTA pair.
constexpr int kMaxLists = 256;

// The A, B and C tensor maps of the first kParamMapGroups groups travel in the launch
// parameters (param space, read by TMA directly): they need neither a fetch from
// global memory at start-up nor the acquire fence that a map written by the host into
// global memory needs before its first use (see tensormap_acquire). 3 KB of
// parameters; the maps of further groups are read from the table.
constexpr int kParamMapGroups = 8;

struct KernelArgs {
    CUtensorMap pmaps[2 * kParamMapGroups];  // A, B of group g at 2g, 2g + 1 (g < min(groups, kParamMapGroups))
    CUtensorMap cmaps[kParamMapGroups];      // C of group g
    const Table *table;
    const int4 *items;      // the table's work items (four int4 each), so that no read waits for the header
    // List l holds items list_begin[l] .. list_begin[l+1]-1. A copy of the table's
    // cta_begin array, passed with the launch so that no CTA waits for it.
    uint32_t list_begin[kMaxLists + 1];
    int *status;            // 4 words: code, role, item, stage
    uint64_t timeout_ns;    // bound of every wait
    int32_t fault_skip_load;  // -1 off; else CTA 0 skips the copies of that k-stage
    int32_t num_groups;
    int32_t prefetch_stages;  // L2 prefetch distance of the producer, in stages (0 = none)
    float *workspace;         // fp32 partial tiles of split tiles (slots of 128 x BN floats)
    int *counters;            // per split tile: segments finished so far (0 between launches)
};

// The fields of a list's first work item that the TMA producer needs for its first
// copies, in the launch parameters of the CTA-pair kernels and of the single-CTA kernel:
// the producer's first copy then waits for no load from the (cold) table. 48 bytes a list.
struct FirstItem {
    int32_t group, tile_m, tile_n, kb_begin, kb_end, kblocks64, flags, a_row;
    const uint8_t *sfa;
    const uint8_t *sfb;
};
constexpr int kParamFirstItems = 80;  // lists (CTA pairs) whose first item travels in the parameters

struct PairArgs : KernelArgs {
    FirstItem first[kParamFirstItems];
};

constexpr int kSingleFirstItems = 160;  // lists (CTAs) of the single-CTA kernel, the same way

struct SingleArgs : KernelArgs {
    FirstItem first[kSingleFirstItems];
};

__host__ __device__ inline FirstItem first_item_of(const WorkItem &w)
{
    return FirstItem{w.group, w.tile_m, w.tile_n, w.kb_begin, w.kb_end, w.kblocks64, w.flags, w.a_row, w.sfa, w.sfb};
}

// A work item with the fields a FirstItem carries (the split fields are those of a whole tile;
// the producer does not read them).
__host__ __device__ inline WorkItem item_of(const FirstItem &f)
{
    WorkItem w{};
    w.group = f.group, w.tile_m = f.tile_m, w.tile_n = f.tile_n, w.kb_begin = f.kb_begin, w.kb_end = f.kb_end;
    w.split = -1, w.nseg = 1, w.kblocks64 = f.kblocks64, w.flags = f.flags, w.a_row = f.a_row;
    w.sfa = f.sfa, w.sfb = f.sfb;
    return w;
}

}  // namespace nvfp4
