// gemm_kernel.cuh -- the persistent, warp-specialised grouped NVFP4 GEMM kernel.
//
// One CTA per SM (a kernel that allocates TMEM gets no second CTA on an SM).
// Each CTA walks its own list of output tiles of 128 rows x BN columns
// (group, tile m, tile n). Fourteen warps share the work:
//   warp 0      TMA producer. It streams 256-wide K-stages of A and B (E2M1,
//               128-byte swizzled rows) and the matching 512-byte scale blocks
//               into a ring of STAGES shared-memory slots.
//   warp 1      MMA issuer; it also owns the TMEM allocation. Per stage it
//               issues four block-scaled MMAs (kind::mxf4nvf4, 16-element scale
//               blocks, M = 128, N = BN, K = 64 each) into the TMEM accumulator,
//               then commits the stage back to the producer.
//   warps 2-5   scale stagers. Per stage each warp reads its rows of the scale
//               blocks from shared memory and writes them into the stage's TMEM
//               scale slot with tcgen05.st, in the layout that
//               tcgen05.cp .32x128b.warpx4 would produce. The scales arrive either
//               as prepacked 512-byte atoms (bulk copies) or as row-major rows of
//               16 bytes per stage (TMA tensor copies); the stagers transpose the
//               latter on the way, so row-major scales need no separate pass.
//   warps 6-13  epilogue. Two warps per TMEM lane quarter, each owning BN/2
//               columns. They read their columns of the accumulator (16 at a time)
//               into fp16 registers and free it for the next tile, then send each
//               32 x 32 block out through a swizzled shared-memory buffer and a TMA
//               store (which clips rows past M and columns past N).
//
// Why this shape. Measurements on this GPU drove it:
//  * One tcgen05.cp of a 512-byte scale block costs about as much tensor-pipe
//    time as an N = 128 MMA (~46 vs ~64 cycles), and a stage needs 8 or 12.
//    So the scales are written with tcgen05.st by other warps while MMAs run.
//  * The issuing thread pays ~100 cycles per tcgen05 instruction and ~300 per
//    stage for its barrier wait and commit, whatever the MMA's N. N = 256 MMAs
//    (BN = 256) halve the issue cost per output and the A re-reads per output.
//  * With BN = 256 the accumulator takes half of TMEM. It is single-buffered:
//    eight epilogue warps read it out in ~0.45 us, and the next tile's MMAs start
//    while those warps store the previous tile.
//
// The pages' kernels (page 1 `grouped_gemm_kernel_v4`, page 2
// `group_gemm_kernel_impl`) copy the scales with tcgen05.cp from the MMA thread,
// and page 1 also runs 128 x 256 tiles for N >= 4096. Other differences:
//  * ring phases are monotone counters carried across tiles, so no barrier is
//    re-initialised;
//  * the schedule is a per-CTA list built on the host;
//  * there is no cluster multicast;
//  * every wait is bounded. When one runs out, the kernel records an error
//    word and returns, and it never traps.
#pragma once
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"
#include "table.h"

namespace nvfp4 {

constexpr int kPipes = 1;                // tile lists per CTA
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kStagerWarp0 = 2;          // warps 2..5
constexpr int kEpilogueWarp0 = 6;        // warps 6..13
constexpr int kEpilogueWarps = 8;
constexpr int kThreads = (kEpilogueWarp0 + kEpilogueWarps) * 32;
constexpr int kBlockM = 128;
constexpr int kBlockK = 256;             // K per stage = 128 bytes of E2M1 per row
constexpr int kRowBytes = kBlockK / 2;   // 128
constexpr int kScaleBlockBytes = 512;    // scales of 128 rows x 64 K
constexpr int kSfRowBytes = kBlockK / 16;  // one row's scales of one K-stage in the row-major layout: 16
constexpr uint32_t kTmemCols = 512;
constexpr int kEpiBufBytes = 32 * 64;    // one epilogue staging buffer: 32 rows x 64 bytes

// Roles reported in the status words.
constexpr int kRoleProducer = 0, kRoleMma = 1, kRoleEpilogue = 2, kRoleTeardown = 3, kRoleScales = 4;

// Named barriers: 0 is __syncthreads, 1 the epilogue warps', 2 the start-up one.
constexpr uint32_t kEpilogueBarrier = 1, kSetupBarrier = 2;

template <int BN, int STAGES>
struct Layout {
    static constexpr int kHalves = BN / 128;                       // 128-row halves of the B tile
    static constexpr int kABytes = kBlockM * kRowBytes;            // 16 KB
    static constexpr int kBBytes = BN * kRowBytes;                 // 32 KB for BN = 256
    static constexpr int kSfaBytes = 4 * kScaleBlockBytes;         // 2 KB
    static constexpr int kSfbBytes = kHalves * 4 * kScaleBlockBytes;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static constexpr int kOffB = kABytes;
    static constexpr int kOffSfa = kABytes + kBBytes;
    static constexpr int kOffSfb = kOffSfa + kSfaBytes;            // half h, k-block j at + (4h + j) * 512
    static constexpr int kRingBytes = STAGES * kStageBytes;
    // epilogue staging: two buffers per epilogue warp (see EpilogueStager)
    static constexpr int kOffEpi = kRingBytes;
    static constexpr int kEpiBytes = kEpilogueWarps * 2 * kEpiBufBytes;
    // barriers: full[S], empty[S], sf_full[S], acc_full, acc_empty, drain, then the TMEM base word
    static constexpr int kBarBytes = (3 * STAGES + 3) * 8 + 16;
    static constexpr int kSmemBytes = 1024 + kRingBytes + kEpiBytes + kBarBytes + 64;  // the SharedState lives in the last 64
    // TMEM columns: the accumulator at 0 .. BN-1, then one scale slot per stage:
    //   SFA at +0 .. 15 (k-block j at +4j),
    //   SFB at +16 .. (k-block j at +16 + 4*kHalves*j; its half h at +4h within that).
    static constexpr uint32_t kSfbCol = 16;
    static constexpr uint32_t kSfColsPerStage = 16 + 16 * kHalves;
    static constexpr uint32_t kSfCol0 = BN;
    static_assert(kStageBytes % 1024 == 0, "stage slots must keep 1024-byte alignment");
    static_assert(BN + STAGES * kSfColsPerStage <= (int)kTmemCols, "TMEM budget");
};

// Item `it` of the table. Read through the items pointer passed with the launch, it
// is one load: through the table header's offset it would be two dependent ones,
// each a DRAM round trip at the start of a launch.
// A stager lane's view of one 128-row region of a stage's scales: the four 16-byte
// rows at base + 512 t (t = 0..3), base including the lane's 16-byte offset. The
// word the MMA wants for K-block j and row lane + 32 i is word i of row t = j in
// the blocked layout (atom j, the 4 scales of rows lane, lane + 32, ...), and word j
// of row t = i in the row-major layout (row lane + 32 i's 16 scales of the stage,
// 4 per K-block): the same four loads, transposed.
struct ScaleRows {
    uint4 q[4];
    __device__ __forceinline__ void load(const uint8_t *base)
    {
#pragma unroll
        for (int t = 0; t < 4; ++t)
            q[t] = *reinterpret_cast<const uint4 *>(base + t * kScaleBlockBytes);
    }
    static __device__ __forceinline__ uint32_t part(const uint4 &v, int c)
    {
        return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
    }
    template <bool kRowMajor>
    __device__ __forceinline__ uint32_t word(int j, int i) const
    {
        return kRowMajor ? part(q[i], j) : part(q[j], i);
    }
};

// One stager warp's part of one stage: SFA (one 128-row region at src) to TMEM
// columns col .. col+15, then SFB (kHalves regions after kSfaBytes) to columns
// col + kSfbCol ..., 16 per store, in the order (K-block j, half h, word i).
template <bool kRowMajor, int kHalves>
__device__ __forceinline__ void stage_scales(const uint8_t *src, int sfa_bytes, uint32_t col, uint32_t sfb_col)
{
    ScaleRows a;
    a.load(src);
    uint32_t ra[16];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            ra[4 * j + i] = a.word<kRowMajor>(j, i);
    tmem_store_16cols(col, ra);
    ScaleRows b[kHalves];
#pragma unroll
    for (int h = 0; h < kHalves; ++h)
        b[h].load(src + sfa_bytes + h * 4 * kScaleBlockBytes);
#pragma unroll
    for (int batch = 0; batch < kHalves; ++batch) {
        uint32_t rb[16];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int idx = batch * 4 + x;  // 0 .. 4*kHalves-1: the (j, h) block in column order
            const int j = idx / kHalves, h = idx % kHalves;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                rb[4 * x + i] = b[h].template word<kRowMajor>(j, i);
        }
        tmem_store_16cols(col + sfb_col + 16 * batch, rb);
    }
}

// Prefetches the scale tensor maps of the groups whose scales are row-major, by
// the lanes of one warp that has nothing else to do at start-up (each lane reads
// its group's flag first).
__device__ __forceinline__ void prefetch_scale_maps(const Table *tab, int num_groups, uint32_t lane)
{
    for (int i = (int)lane; i < 2 * min(num_groups, 64); i += 32) {
        const GroupEntry &g = tab->group(i / 2);
        if (g.sf_rowmajor)
            tensormap_prefetch(i % 2 == 0 ? &g.tmap_sfa : &g.tmap_sfb);
    }
}

// The A and B maps of group g: from the launch parameters for the first
// kParamMapGroups groups, else from the table (those take an acquire fence before a
// thread's first use, see acquire_table_maps).
__device__ __forceinline__ const CUtensorMap *map_a(const KernelArgs &args, const Table *tab, int g)
{
    return g < kParamMapGroups ? &args.pmaps[2 * g] : &tab->group(g).tmap_a;
}
__device__ __forceinline__ const CUtensorMap *map_b(const KernelArgs &args, const Table *tab, int g)
{
    return g < kParamMapGroups ? &args.pmaps[2 * g + 1] : &tab->group(g).tmap_b;
}

// The C map of group g (the epilogues' stores), by the same rule.
__device__ __forceinline__ const CUtensorMap *map_c(const KernelArgs &args, const Table *tab, int g)
{
    return g < kParamMapGroups ? &args.cmaps[g] : &tab->group(g).tmap_c;
}

// Prefetch of the table's A and B maps of groups kParamMapGroups .. 63, by a warp's lanes.
__device__ __forceinline__ void prefetch_table_maps(const Table *tab, int num_groups, uint32_t lane)
{
    for (int i = 2 * kParamMapGroups + (int)lane; i < 2 * min(num_groups, 64); i += 32) {
        const GroupEntry &g = tab->group(i / 2);
        tensormap_prefetch(i % 2 == 0 ? &g.tmap_a : &g.tmap_b);
    }
}

__device__ __forceinline__ WorkItem global_item(const KernelArgs &args, uint32_t it)
{
    const int4 *p = args.items + 4 * (size_t)it;
    return unpack_item(p[0], p[1], p[2], p[3]);
}

struct SharedState {
    volatile int abort;  // set by the first role that gives up a wait
    volatile int last;   // epilogue: this CTA completes the split tile being stored
};

// Records the first error of the launch in the device status words.
__device__ __forceinline__ void record_error(int *status, int code, int role, int item, int stage)
{
    if (atomicCAS(status, 0, code) == 0) {
        status[1] = role;
        status[2] = item;
        status[3] = stage;
        __threadfence();
    }
}

// Bounded wait on an mbarrier phase. Returns false if the wait ran out or
// another role already gave up. In both cases the caller leaves its loop.
// It first polls with test_wait, which never suspends: try_wait may suspend the
// thread for up to about a microsecond, and a phase that a peer CTA's remote
// arrival completes does not always wake it sooner (measured: 1 us per stage on
// the CTA-pair kernel's tile changes, 3 % of the whole launch).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, SharedState *sh, const KernelArgs &args,
                                           int role, int item, int stage)
{
    for (int i = 0; i < 64; ++i)
        if (mbar_test_wait(bar, parity))
            return true;
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((spin & 63u) == 0) {
            if (sh->abort)
                return false;
            if (global_timer_ns() - t0 > args.timeout_ns) {
                sh->abort = 1;
                record_error(args.status, kStatusTimeout, role, item, stage);
                return false;
            }
        }
    }
}

// The same wait for a whole warp: lane 0 polls, the verdict is shared, and
// every lane then takes its own acquire of the completed phase (which cannot
// move on before this warp releases it).
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, SharedState *sh,
                                                const KernelArgs &args, int role, int item, int stage)
{
    int ok = 1;
    if (lane_id() == 0)
        ok = wait_phase(bar, parity, sh, args, role, item, stage) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok)
        (void)mbar_try_wait(bar, parity);
    return ok != 0;
}

// Bounded wait that ignores the abort flag, for the teardown drains.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const KernelArgs &args, int stage)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > args.timeout_ns) {
            record_error(args.status, kStatusTimeout, kRoleTeardown, -1, stage);
            return;
        }
    }
}

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo, uint32_t hi)
{
    __half2 h = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t *>(&h);
}

// An epilogue warp's way out for C: two 2 KB shared-memory buffers of 32 rows x 64
// bytes (32 fp16 columns), alternated, each the source of one TMA store of a
// 32 x 32 box. Before a buffer is rewritten, the store that read it two chunks ago
// must have finished reading shared memory. Rows go in with the 64-byte swizzle
// (16-byte chunk j of row r at position j ^ ((r >> 1) & 3)), which is what the
// tensor map expects and keeps the warp's writes free of bank conflicts.
struct EpilogueStager {
    uint8_t *bufs;  // 2 * kEpiBufBytes, 1024-byte aligned
    uint32_t n = 0;

    // Row `lane` of the box comes from h[0..15]; (x, y) is the box's first column and row.
    __device__ __forceinline__ void store(const CUtensorMap *tmap, int x, int y, const uint32_t *h, uint32_t lane)
    {
        uint8_t *buf = bufs + (n & 1) * kEpiBufBytes;
        ++n;
        if (lane == 0)
            bulk_wait_group_read<1>();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4 *>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(h[4 * j + 0], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmap, x, y, smem_addr(buf));
            bulk_commit_group();
        }
    }

    // Every store must be complete before the CTA exits.
    __device__ __forceinline__ void finish(uint32_t lane)
    {
        if (lane == 0)
            bulk_wait_group<0>();
        __syncwarp();
    }
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) nvfp4_grouped_gemm_kernel(const __grid_constant__ SingleArgs args)
{
    static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
    using L = Layout<BN, STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern of the operand tiles
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffEpi + L::kEpiBytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *sf_full = bars + 2 * STAGES;
    uint64_t *acc_full = bars + 3 * STAGES;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *drain = acc_empty + 1;
    uint32_t *tmem_base_word = reinterpret_cast<uint32_t *>(drain + 1);
    SharedState *sh = reinterpret_cast<SharedState *>(tmem_base_word + 2);

    const int warp = threadIdx.x / 32;
    const uint32_t lane = threadIdx.x % 32;
    const Table *tab = args.table;
    const uint32_t item_begin = args.list_begin[blockIdx.x];
    const uint32_t item_end = args.list_begin[blockIdx.x + 1];
    // The producer's first item is read before anything else, so that its latency
    // overlaps the set-up below.
    WorkItem first_item{};
    if (warp == kProducerWarp && lane == 0 && item_begin < item_end)
        first_item = blockIdx.x < (unsigned)kSingleFirstItems ? item_of(args.first[blockIdx.x])
                                                              : global_item(args, item_begin);
    // The operand maps of groups past those in the launch parameters, fetched ahead by
    // the producer warp's lanes in parallel.
    if (warp == kProducerWarp)
        prefetch_table_maps(tab, args.num_groups, lane);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
            mbar_init(smem_addr(&sf_full[s]), 4);  // one elected arrive per stager warp
        }
        mbar_init(smem_addr(acc_full), 1);
        mbar_init(smem_addr(acc_empty), kEpilogueWarps);  // one elected arrive per epilogue warp
        mbar_init(smem_addr(drain), 1);
        sh->abort = 0;
        fence_barrier_init();
    }
    // The producer needs nothing but the barriers its lane 0 just initialised, so
    // it starts at once; the other warps also wait for the TMEM allocation.
    uint32_t tmem_base = 0;
    if (warp == kProducerWarp) {
        __syncwarp();
        named_barrier_arrive(kSetupBarrier, kThreads);
    } else {
        if (warp == kMmaWarp) {
            tmem_alloc(smem_addr(tmem_base_word), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        named_barrier_sync(kSetupBarrier, kThreads);
        tc_fence_after();
        tmem_base = *tmem_base_word;
    }
    const uint32_t tmem_sf = tmem_base + L::kSfCol0;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ TMA producer
        // Besides the ring's loads, the producer keeps an L2 prefetch cursor
        // args.prefetch_stages stages ahead of them, across tile boundaries: the
        // ring holds only STAGES stages, and a stage that comes from DRAM takes
        // ~1.5 us to land, while one that comes from L2 lands several times sooner.
        if (lane == 0) {
            // Inputs may come from the previous kernel in the stream (programmatic
            // dependent launch): nothing of the caller's is read before this wait.
            grid_dependency_wait();
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_b_stream = policy_evict_first();
            const uint64_t pol_b_shared = policy_evict_normal();
            struct Src {  // where one tile's stages come from
                int group;
                const void *tmap_a, *tmap_b;
                int32_t ya, yb;
                int kb64, kb_begin, kb_end;
                bool b_shared;
                bool sf_rowmajor;              // scales through tmap_sfa / tmap_sfb at rows ya / yb
                const void *tmap_sfa, *tmap_sfb;
                const uint8_t *sfa;            // else blocked scale atoms
                const uint8_t *sfb[L::kHalves];
            };
            // Everything but the tensor maps' addresses comes from the item itself.
            auto source = [&](uint32_t it) {
                Src r;
                const WorkItem w = it == item_begin ? first_item : global_item(args, it);
                const GroupEntry &ge = tab->group(w.group);  // address only: no load
                r.group = w.group;
                r.tmap_a = map_a(args, tab, w.group);  // one A map per group: M-fusion is for CTA pairs only
                r.tmap_b = map_b(args, tab, w.group);
                r.ya = w.tile_m * kBlockM;
                r.yb = w.tile_n * BN;
                r.kb64 = w.kblocks64;
                r.kb_begin = w.kb_begin;
                r.kb_end = w.kb_end;
                r.b_shared = (w.flags & kItemBShared) != 0;
                r.sf_rowmajor = (w.flags & kItemSfRowMajor) != 0;
                r.tmap_sfa = &ge.tmap_sfa;
                r.tmap_sfb = &ge.tmap_sfb;
                r.sfa = w.sfa;
                // The scales of B come in 128-row tiles. A half of the B tile that lies
                // wholly past N reads the first half's scales instead: its B rows are
                // zero (TMA fills them), so the scales only need to be finite.
                r.sfb[0] = w.sfb;
                if (L::kHalves > 1)
                    r.sfb[L::kHalves - 1] = w.sfb + ((w.flags & kItemB2) ? (size_t)r.kb64 * kScaleBlockBytes : 0);
                return r;
            };
            // Maps read from the table (A and B of groups past the launch parameters, and
            // the row-major scale maps) get their acquire fence here, before this thread's
            // first copy (or prefetch) through them.
            int fenced = -1;
            auto acquire_maps = [&](const Src &s) {
                if (s.group == fenced)
                    return;
                fenced = s.group;
                if (s.group >= kParamMapGroups) {
                    tensormap_acquire(s.tmap_a);
                    tensormap_acquire(s.tmap_b);
                }
                if (s.sf_rowmajor) {
                    tensormap_acquire(s.tmap_sfa);
                    tensormap_acquire(s.tmap_sfb);
                }
            };
            // prefetch cursor
            uint32_t pf_it = item_begin, pf_g = 0;
            Src pf{};
            if (pf_it < item_end)
                pf = source(pf_it);
            int pf_kb = pf.kb_begin;
            auto prefetch_until = [&](uint32_t g_end) {
                while (pf_g < g_end && pf_it < item_end) {
                    acquire_maps(pf);
                    const uint32_t sfb_bytes = (uint32_t)min(4, pf.kb64 - pf_kb * 4) * kScaleBlockBytes;
                    tma_prefetch_2d(pf.tmap_a, pf_kb * kRowBytes, pf.ya);
                    tma_prefetch_2d(pf.tmap_b, pf_kb * kRowBytes, pf.yb);
                    if (pf.sf_rowmajor) {
                        tma_prefetch_2d(pf.tmap_sfa, pf_kb * kSfRowBytes, pf.ya);
                        tma_prefetch_2d(pf.tmap_sfb, pf_kb * kSfRowBytes, pf.yb);
                    } else {
                        bulk_prefetch(pf.sfa + (size_t)pf_kb * 4 * kScaleBlockBytes, sfb_bytes);
#pragma unroll
                        for (int h = 0; h < L::kHalves; ++h)
                            bulk_prefetch(pf.sfb[h] + (size_t)pf_kb * 4 * kScaleBlockBytes, sfb_bytes);
                    }
                    ++pf_g;
                    if (++pf_kb == pf.kb_end) {
                        if (++pf_it < item_end) {
                            pf = source(pf_it);
                            pf_kb = pf.kb_begin;
                        }
                    }
                }
            };
            const uint32_t pf_dist = (uint32_t)args.prefetch_stages;
            uint32_t stage = 0, phase = 0, kiter = 0;
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const Src src = source(it);
                acquire_maps(src);
                const uint64_t pol_b = src.b_shared ? pol_b_shared : pol_b_stream;
                for (int kb = src.kb_begin; kb < src.kb_end; ++kb, ++kiter) {
                    if (pf_dist > 0)
                        prefetch_until(kiter + pf_dist);
                    if (!wait_phase(smem_addr(&empty[stage]), phase ^ 1u, sh, args, kRoleProducer, (int)it, kb)) {
                        ok = false;
                        break;
                    }
                    const int ksub = min(4, src.kb64 - kb * 4);
                    const uint32_t sf_bytes = (uint32_t)ksub * kScaleBlockBytes;
                    const uint32_t bytes = L::kABytes + L::kBBytes + sf_bytes * (1 + L::kHalves);
                    const uint32_t slot = smem_addr(ring + stage * L::kStageBytes);
                    const uint32_t fb = smem_addr(&full[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    if (!(args.fault_skip_load >= 0 && blockIdx.x == 0 && kiter == (uint32_t)args.fault_skip_load)) {
                        tma_load_2d(slot, src.tmap_a, kb * kRowBytes, src.ya, fb, pol_a);
                        tma_load_2d(slot + L::kOffB, src.tmap_b, kb * kRowBytes, src.yb, fb, pol_b);
                        if (src.sf_rowmajor) {  // K % 256 == 0: always a whole stage (sf_bytes = 2 KB)
                            tma_load_2d(slot + L::kOffSfa, src.tmap_sfa, kb * kSfRowBytes, src.ya, fb, pol_a);
                            tma_load_2d(slot + L::kOffSfb, src.tmap_sfb, kb * kSfRowBytes, src.yb, fb, pol_b);
                        } else {
                            bulk_load(slot + L::kOffSfa, src.sfa + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb, pol_a);
#pragma unroll
                            for (int h = 0; h < L::kHalves; ++h)
                                bulk_load(slot + L::kOffSfb + h * 4 * kScaleBlockBytes,
                                          src.sfb[h] + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb, pol_b);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            grid_launch_dependents();  // every copy of this CTA is issued
            // Before the CTA may exit, every copy it started must have landed.
            // A full barrier whose last fill was consumed has already flipped its
            // phase, so these waits return at once in a normal run.
            const uint32_t issued = kiter < (uint32_t)STAGES ? kiter : (uint32_t)STAGES;
            for (uint32_t i = 0; i < issued; ++i) {
                const uint32_t f = kiter - 1 - i;
                drain_wait(smem_addr(&full[f % STAGES]), (f / STAGES) & 1u, args, (int)(f % STAGES));
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------ MMA issuer
        // This thread is on the critical path, so its loop is short: descriptors
        // and TMEM addresses advance by constant steps and are never rebuilt.
        if (lane == 0) {
            constexpr uint32_t idesc = mma_idesc_nvfp4(kBlockM, BN);
            constexpr uint64_t kDescStep = (uint64_t)(L::kStageBytes >> 4);  // one ring slot, in 16-byte units
            constexpr uint32_t kB = L::kSfbCol, kJ = 4 * L::kHalves;          // SFB column of k-block j: kB + kJ*j
            const uint64_t desc_a0 = operand_desc(smem_addr(ring));
            const uint64_t desc_b0 = operand_desc(smem_addr(ring) + L::kOffB);
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            uint64_t da = desc_a0, db = desc_b0;
            uint32_t sf = tmem_sf;
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const WorkItem w = global_item(args, it);
                const int kb64 = w.kblocks64;
                // the epilogue warps must have drained the previous tile's accumulator
                if (!wait_phase(smem_addr(acc_empty), acc_phase ^ 1u, sh, args, kRoleMma, (int)it, -1)) {
                    ok = false;
                    break;
                }
                acc_phase ^= 1u;
                tc_fence_after();
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
                    // sf_full is released by the stagers only after they acquired the
                    // stage's full barrier, so the TMA writes of A and B are ordered
                    // before this wait.
                    if (!wait_phase(smem_addr(&sf_full[stage]), phase, sh, args, kRoleMma, (int)it, kb)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acc0 = kb > w.kb_begin ? 1u : 0u;
                    if (kb64 - kb * 4 >= 4) {
                        // K step of 64 E2M1 = 32 bytes inside the 128-byte swizzled row: +2 in the
                        // descriptor's 16-byte address field
                        tc_mma_nvfp4(tmem_base, da + 0, db + 0, idesc, sf + 0, sf + kB, acc0);
                        tc_mma_nvfp4(tmem_base, da + 2, db + 2, idesc, sf + 4, sf + kB + kJ, 1u);
                        tc_mma_nvfp4(tmem_base, da + 4, db + 4, idesc, sf + 8, sf + kB + 2 * kJ, 1u);
                        tc_mma_nvfp4(tmem_base, da + 6, db + 6, idesc, sf + 12, sf + kB + 3 * kJ, 1u);
                    } else {
                        const int ksub = kb64 - kb * 4;
                        for (int j = 0; j < ksub; ++j)
                            tc_mma_nvfp4(tmem_base, da + 2 * j, db + 2 * j, idesc, sf + 4 * j, sf + kB + kJ * j,
                                         (acc0 | (uint32_t)j) ? 1u : 0u);
                    }
                    tc_commit(smem_addr(&empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                        da = desc_a0;
                        db = desc_b0;
                        sf = tmem_sf;
                    } else {
                        da += kDescStep;
                        db += kDescStep;
                        sf += L::kSfColsPerStage;
                    }
                }
                if (!ok)
                    break;
                tc_commit(smem_addr(acc_full));
            }
            // Every MMA this thread issued must finish before TMEM is freed.
            tc_commit(smem_addr(drain));
            drain_wait(smem_addr(drain), 0, args, -1);
        }
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------ scale stagers
        // Lane r of the warp for TMEM lane quarter q writes TMEM lane 32q + r. The 4
        // k-scales of row r + 32c for K-block j go to column base(j) + c (see
        // ScaleRows for where they sit in shared memory, blocked or row-major). That
        // is the layout tcgen05.cp .32x128b.warpx4 produces, repeated in all four
        // quarters.
        const int quarter = warp % 4;  // warps 2,3,4,5 -> quarters 2,3,0,1
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (uint32_t it = item_begin; ok && it < item_end; ++it) {
            const WorkItem w = global_item(args, it);
            for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
                if (!warp_wait_phase(smem_addr(&full[stage]), phase, sh, args, kRoleScales, (int)it, kb)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = ring + stage * L::kStageBytes + L::kOffSfa + lane * 16;
                const uint32_t col = tmem_sf + lane_off + stage * L::kSfColsPerStage;
                if (w.flags & kItemSfRowMajor)
                    stage_scales<true, L::kHalves>(src, L::kSfaBytes, col, L::kSfbCol);
                else
                    stage_scales<false, L::kHalves>(src, L::kSfaBytes, col, L::kSfbCol);
                tmem_store_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&sf_full[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        // Warp w owns TMEM lane quarter w % 4 and the column half (w - 6) / 4 of the
        // accumulator: output rows tile_m*128 + 32*(w % 4) + lane, columns
        // half*BN/2 .. half*BN/2 + BN/2 - 1 of the tile. C leaves through staged TMA
        // stores, which clip rows past M and columns past N.
        const int quarter = warp % 4;  // warps 6..13 -> quarters 2,3,0,1,2,3,0,1
        const int chalf = (warp - kEpilogueWarp0) / 4;
        constexpr int kCols = BN / 2;
        const uint32_t t_addr = tmem_base + ((uint32_t)(quarter * 32) << 16) + chalf * kCols;
        EpilogueStager out{smem + L::kOffEpi + (warp - kEpilogueWarp0) * 2 * kEpiBufBytes};
        if (warp == kEpilogueWarp0)
            prefetch_scale_maps(tab, args.num_groups, lane);
        uint32_t acc_phase = 0;
        int fenced = -1;  // the group whose C map lane 0 (which issues the stores) last fenced
        grid_dependency_wait();  // C and the split workspace may still be in use by the previous kernel
        for (uint32_t it = item_begin; it < item_end; ++it) {
            const WorkItem w = global_item(args, it);
            const GroupEntry &ge = tab->group(w.group);
            const int M = ge.M, N = ge.N;
            // before the wait for the accumulator, so that the fence overlaps the MMAs
            if (lane == 0 && w.group >= kParamMapGroups && w.group != fenced) {
                tensormap_acquire(map_c(args, tab, w.group));
                fenced = w.group;
            }
            if (!warp_wait_phase(smem_addr(acc_full), acc_phase, sh, args, kRoleEpilogue, (int)it, -1))
                break;
            acc_phase ^= 1u;
            tc_fence_after();
            const int m_row0 = w.tile_m * kBlockM + quarter * 32;  // first of this warp's 32 rows
            const bool rows_in = m_row0 < M;                       // warp-uniform
            const int n0 = w.tile_n * BN + chalf * kCols;
            if (w.split < 0) {
                // whole tile: the warp's columns TMEM -> fp16 registers, the accumulator
                // released (the next tile's MMAs wait for it), then 32 columns at a time
                // -> staging -> TMA store: the release never waits for the store path.
                uint32_t h[kCols / 32][16];
#pragma unroll
                for (int c = 0; c < kCols / 16; ++c) {
                    uint32_t v[16];
                    tmem_load_16cols(t_addr + c * 16, v);
                    tmem_load_wait();
                    reg_fence(v);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        h[c / 2][(c % 2) * 8 + i] = pack_half2(v[2 * i], v[2 * i + 1]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(acc_empty));
                if (rows_in) {
#pragma unroll
                    for (int c = 0; c < kCols / 32; ++c)
                        if (n0 + c * 32 < N)
                            out.store(map_c(args, tab, w.group), n0 + c * 32, m_row0, h[c], lane);
                }
            } else {
                // One segment of a split tile: its fp32 partial goes to the workspace slot.
                // Thread e of the epilogue keeps its elements at float4 index (c*8 + f)*256 + e
                // of the slot, so every store and load of a warp covers 512 contiguous bytes.
                // Warps whose 32 rows lie past M neither write nor read partials.
                const int e = (warp - kEpilogueWarp0) * 32 + (int)lane;
                constexpr int kSlotFloats = kBlockM * BN;
                float4 *ws = reinterpret_cast<float4 *>(args.workspace + (size_t)w.ws_slot * kSlotFloats);
                if (rows_in) {
#pragma unroll
                    for (int c = 0; c < kCols / 32; ++c) {
                        uint32_t v[32];
                        tmem_load_32cols(t_addr + c * 32, v);
                        tmem_load_wait();
                        reg_fence(v);
#pragma unroll
                        for (int f = 0; f < 8; ++f)
                            ws[(c * 8 + f) * 256 + e] =
                                make_float4(__uint_as_float(v[4 * f + 0]), __uint_as_float(v[4 * f + 1]),
                                            __uint_as_float(v[4 * f + 2]), __uint_as_float(v[4 * f + 3]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(acc_empty));
                // Count this segment in. The segment that completes the count sums all of
                // them; nothing ever waits for another CTA.
                __threadfence();
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
                if (e == 0)
                    sh->last = (atomicAdd(&args.counters[w.split], 1) == w.nseg - 1) ? 1 : 0;
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
                if (sh->last) {
                    __threadfence();
                    const float4 *ws0 = reinterpret_cast<const float4 *>(args.workspace +
                                                                         (size_t)(w.ws_slot - w.seg) * kSlotFloats);
                    // Each partial is read once, here: its L2 lines are then dropped, so they
                    // are never written back to DRAM. Lane l < 4 drops the 128-byte line of
                    // lanes 8l .. 8l+7, after the whole warp has read it.
                    auto drop = [&](const float4 *wp, int c) {
                        __syncwarp();
                        if (lane < 4) {
#pragma unroll
                            for (int f = 0; f < 8; ++f)
                                discard_l2_line(&wp[(c * 8 + f) * 256 + (e - (int)lane) + 8 * (int)lane]);
                        }
                    };
                    if (rows_in) {
#pragma unroll 1
                        for (int c = 0; c < kCols / 32; ++c) {
                            // 32 columns at a time, eight independent loads per segment in
                            // flight; segments are added in K order, so the rounding does not
                            // depend on which segment finished last
                            float4 acc[8];
#pragma unroll
                            for (int f = 0; f < 8; ++f)
                                acc[f] = __ldcg(&ws0[(c * 8 + f) * 256 + e]);
                            for (int sg = 1; sg < w.nseg; ++sg) {
                                const float4 *wp = ws0 + (size_t)sg * (kSlotFloats / 4);
                                float4 q[8];
#pragma unroll
                                for (int f = 0; f < 8; ++f)
                                    q[f] = __ldcg(&wp[(c * 8 + f) * 256 + e]);
#pragma unroll
                                for (int f = 0; f < 8; ++f)
                                    acc[f].x += q[f].x, acc[f].y += q[f].y, acc[f].z += q[f].z, acc[f].w += q[f].w;
                                drop(wp, c);
                            }
                            drop(ws0, c);
                            if (n0 + c * 32 < N) {
                                uint32_t h[16];
#pragma unroll
                                for (int f = 0; f < 8; ++f) {
                                    h[2 * f] = pack_half2(__float_as_uint(acc[f].x), __float_as_uint(acc[f].y));
                                    h[2 * f + 1] = pack_half2(__float_as_uint(acc[f].z), __float_as_uint(acc[f].w));
                                }
                                out.store(map_c(args, tab, w.group), n0 + c * 32, m_row0, h, lane);
                            }
                        }
                    }
                    if (e == 0)
                        args.counters[w.split] = 0;  // ready for the next launch
                }
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);  // sh->last is read before it is rewritten
            }
        }
        out.finish(lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace nvfp4
