// pair_kernel.cuh -- the CTA-pair variant of the grouped NVFP4 GEMM kernel.
//
// A cluster of two CTAs (one per SM) computes 256 x 256 output tiles with the
// pair form of the block-scaled MMA (tcgen05.mma.cta_group::2, M = 256,
// N = 256, K = 64). Per K-stage each CTA of the pair loads
//   * its own 128 rows of the A tile (CTA rank r: rows 128r .. 128r+127),
//   * its half of the B tile (B rows 128r .. 128r+127 of the 256),
//   * the scale blocks of its A rows and of all 256 B rows,
// so each SM moves 32 KB of E2M1 operands per stage for a 128 x 256 block of
// outputs: half the bytes per output of the single-CTA 128 x 128 tile. The even
// CTA (the leader) issues the MMAs for both; each CTA's TMEM receives its own
// 128 rows of the accumulator.
//
// Warp roles are those of the single-CTA kernel (warp 0 producer, warp 1 MMA
// and TMEM owner, warps 2-5 scale stagers, warps 6-13 epilogue), in both CTAs,
// except that only the leader's warp 1 issues MMAs. Synchronisation across the
// pair:
//   full[s]     per CTA: its own copies of stage s landed (TMA transaction count).
//   sf_full[s]  leader only, 8 arrivals: the stager warps of BOTH CTAs saw their
//               own full[s] and wrote their scale slots into their own TMEM. So
//               when it completes, both CTAs' operands and scales are in place.
//   empty[s]    per CTA, completed by the leader's multicast commit when the
//               MMAs that read stage s are done: the slot may be refilled.
//   acc_full    per CTA, leader's multicast commit after a tile's last MMA.
//   acc_empty   leader only, 16 arrivals: the epilogue warps of both CTAs
//               drained their accumulator rows.
//   drain       per CTA, leader's multicast commit after its last MMA: TMEM
//               may be freed.
// The leader's own warps arrive on its barriers as usual. The peer's warps arrive
// remotely and relaxed: each arrival announces work that has already completed
// (the warp saw its TMA bytes land on its own full barrier, and its tcgen05.st /
// tcgen05.ld returned from tcgen05.wait), so it needs no release of memory. A
// cluster barrier at both ends keeps every remote arrival inside the lifetime of
// both CTAs.
//
// Split tiles: each CTA keeps its own 128 rows. Segment partials go to
// workspace slot 2 * ws_slot + rank, and the counter of the split tile's half is
// counters[2 * split + rank], so the two halves finish independently.
#pragma once
#include "gemm_kernel.cuh"

namespace nvfp4 {

constexpr int kPairBlockM = 256;  // output rows per pair tile (128 per CTA)
constexpr int kPairBlockN = 256;  // output columns per pair tile

template <int STAGES>
struct PairLayout {
    static constexpr int kABytes = 128 * kRowBytes;              // this CTA's 128 A rows: 16 KB
    static constexpr int kBBytes = 128 * kRowBytes;              // this CTA's half of the B rows: 16 KB
    static constexpr int kSfaBytes = 4 * kScaleBlockBytes;       // 2 KB
    static constexpr int kSfbBytes = 8 * kScaleBlockBytes;       // 4 KB: both 128-row halves of B
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;  // 38 KB
    static constexpr int kOffB = kABytes;
    static constexpr int kOffSfa = kABytes + kBBytes;
    static constexpr int kOffSfb = kOffSfa + kSfaBytes;          // half h, k-block j at + (4h + j) * 512
    static constexpr int kRingBytes = STAGES * kStageBytes;
    // epilogue staging: two buffers per epilogue warp (see EpilogueStager)
    static constexpr int kOffEpi = kRingBytes;
    static constexpr int kEpiBytes = kEpilogueWarps * 2 * kEpiBufBytes;
    static constexpr int kBarBytes = (3 * STAGES + 3) * 8 + 16;
    static constexpr int kSmemBytes = 1024 + kRingBytes + kEpiBytes + kBarBytes + 64;
    // TMEM columns: the accumulator at 0 .. 255, then one scale slot per stage:
    //   SFA at +0 .. 15 (k-block j at +4j), SFB at +16 .. 47 (k-block j at +16 + 8j, half h at +4h).
    static constexpr uint32_t kSfCol0 = kPairBlockN;
    static constexpr uint32_t kSfbCol = 16;
    static constexpr uint32_t kSfColsPerStage = 48;
    static_assert(kStageBytes % 1024 == 0, "stage slots must keep 1024-byte alignment");
    static_assert(kPairBlockN + STAGES * kSfColsPerStage <= (int)kTmemCols, "TMEM budget");
};

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    nvfp4_pair_gemm_kernel(const __grid_constant__ PairArgs args)
{
    using L = PairLayout<STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
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
    const uint32_t rank = cluster_rank();
    const Table *tab = args.table;
    const int pair = blockIdx.x >> 1;
    const uint32_t item_begin = args.list_begin[pair];
    const uint32_t item_end = args.list_begin[pair + 1];
    // The producer's first item is read before anything else, so that its latency
    // overlaps the set-up below.
    WorkItem first_item{};
    if (warp == kProducerWarp && lane == 0 && item_begin < item_end)
        first_item = pair < kParamFirstItems ? item_of(args.first[pair]) : global_item(args, item_begin);
    // The operand maps of groups past those in the launch parameters, fetched ahead by
    // the producer warp's lanes in parallel.
    if (warp == kProducerWarp)
        prefetch_table_maps(tab, args.num_groups, lane);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
            mbar_init(smem_addr(&sf_full[s]), 8);  // 4 stager warps in each CTA
        }
        mbar_init(smem_addr(acc_full), 1);
        mbar_init(smem_addr(acc_empty), 2 * kEpilogueWarps);
        mbar_init(smem_addr(drain), 1);
        sh->abort = 0;
        fence_barrier_init();
    }
    // The producer needs nothing but the barriers its lane 0 just initialised, so
    // it starts at once (it sends nothing to the peer). The other warps also wait
    // for the TMEM allocation and for the peer's barriers to exist, since the
    // leader's commits and the peer's arrivals cross the pair. The producer's
    // cluster arrival is relaxed: the barrier initialisation it did is published
    // by the other warps' release arrivals, which follow the named barrier (a
    // cluster-scope release costs about half a microsecond here).
    uint32_t tmem_base = 0;
    if (warp == kProducerWarp) {
        __syncwarp();
        named_barrier_arrive(kSetupBarrier, kThreads);
        cluster_arrive_relaxed();
    } else {
        if (warp == kMmaWarp) {
            tmem_alloc_pair(smem_addr(tmem_base_word), kTmemCols);
            tmem_relinquish_pair();
        }
        tc_fence_before();
        named_barrier_sync(kSetupBarrier, kThreads);
        cluster_arrive();
        cluster_wait();
        tc_fence_after();
        tmem_base = *tmem_base_word;
    }
    const uint32_t tmem_sf = tmem_base + L::kSfCol0;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            // Inputs may come from the previous kernel in the stream (programmatic
            // dependent launch): nothing of the caller's is read before this wait.
            grid_dependency_wait();
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_b_stream = policy_evict_first();
            const uint64_t pol_b_shared = policy_evict_normal();
            uint32_t stage = 0, phase = 0, kiter = 0;
            int fenced_b = -1, fenced_a = -1;  // groups whose maps this thread has fenced (tensormap_acquire)
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const WorkItem w = it == item_begin ? first_item : global_item(args, it);
                const GroupEntry &ge = tab->group(w.group);  // address only: the tensor maps
                const int a_map = w.flags >> kItemAMapShift;
                const GroupEntry &ga = tab->group(a_map);  // the (possibly shared) A map
                const bool sf_rm_item = (w.flags & kItemSfRowMajor) != 0;
                // maps read from the table take an acquire fence before their first use
                const CUtensorMap *tmap_a = map_a(args, tab, a_map), *tmap_b = map_b(args, tab, w.group);
                if (w.group != fenced_b) {
                    fenced_b = w.group;
                    if (w.group >= kParamMapGroups)
                        tensormap_acquire(tmap_b);
                    if (sf_rm_item)
                        tensormap_acquire(&ge.tmap_sfb);
                }
                if (a_map != fenced_a) {
                    fenced_a = a_map;
                    if (a_map >= kParamMapGroups)
                        tensormap_acquire(tmap_a);
                    if (sf_rm_item)
                        tensormap_acquire(&ga.tmap_sfa);
                }
                const int kb64 = w.kblocks64;
                const int32_t ya = w.a_row + (int)rank * 128;
                const int32_t yb = w.tile_n * kPairBlockN + (int)rank * 128;
                // Scale blocks come in 128-row tiles. A 128-row half that lies wholly
                // past M (or N) reads the tile's first half's scales instead: its
                // operand rows are zero (TMA fills them), so the scales need only be
                // finite.
                const size_t half = (size_t)kb64 * kScaleBlockBytes;
                const uint8_t *sfa = w.sfa + ((rank == 1 && (w.flags & kItemA2)) ? half : 0);
                const uint8_t *sfb[2] = {w.sfb, w.sfb + ((w.flags & kItemB2) ? half : 0)};
                const uint64_t pol_b = (w.flags & kItemBShared) ? pol_b_shared : pol_b_stream;
                const bool sf_rm = (w.flags & kItemSfRowMajor) != 0;
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++kiter) {
                    if (!wait_phase(smem_addr(&empty[stage]), phase ^ 1u, sh, args, kRoleProducer, (int)it, kb)) {
                        ok = false;
                        break;
                    }
                    const int ksub = min(4, kb64 - kb * 4);
                    const uint32_t sf_bytes = (uint32_t)ksub * kScaleBlockBytes;
                    const uint32_t bytes = L::kABytes + L::kBBytes + sf_bytes * 3;
                    const uint32_t slot = smem_addr(ring + stage * L::kStageBytes);
                    const uint32_t fb = smem_addr(&full[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    if (!(args.fault_skip_load >= 0 && blockIdx.x == 0 && kiter == (uint32_t)args.fault_skip_load)) {
                        tma_load_2d(slot, tmap_a, kb * kRowBytes, ya, fb, pol_a);
                        tma_load_2d(slot + L::kOffB, tmap_b, kb * kRowBytes, yb, fb, pol_b);
                        if (sf_rm) {  // K % 256 == 0: a whole stage; B's box is both halves, 256 rows
                            tma_load_2d(slot + L::kOffSfa, &ga.tmap_sfa, kb * kSfRowBytes, ya, fb, pol_a);
                            tma_load_2d(slot + L::kOffSfb, &ge.tmap_sfb, kb * kSfRowBytes, w.tile_n * kPairBlockN, fb,
                                        pol_b);
                        } else {
                            bulk_load(slot + L::kOffSfa, sfa + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb, pol_a);
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                bulk_load(slot + L::kOffSfb + h * 4 * kScaleBlockBytes,
                                          sfb[h] + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb, pol_b);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            grid_launch_dependents();  // every copy of this CTA is issued
            // Every copy this CTA started must land before it may exit.
            const uint32_t issued = kiter < (uint32_t)STAGES ? kiter : (uint32_t)STAGES;
            for (uint32_t i = 0; i < issued; ++i) {
                const uint32_t f = kiter - 1 - i;
                drain_wait(smem_addr(&full[f % STAGES]), (f / STAGES) & 1u, args, (int)(f % STAGES));
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------ MMA issuer (leader)
        if (rank == 0 && lane == 0) {
            constexpr uint32_t idesc = mma_idesc_nvfp4(kPairBlockM, kPairBlockN);
            constexpr uint64_t kDescStep = (uint64_t)(L::kStageBytes >> 4);
            constexpr uint32_t kB = L::kSfbCol, kJ = 8;  // SFB column of k-block j: kB + kJ*j
            const uint64_t desc_a0 = operand_desc(smem_addr(ring));
            const uint64_t desc_b0 = operand_desc(smem_addr(ring) + L::kOffB);
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            uint64_t da = desc_a0, db = desc_b0;
            uint32_t sf = tmem_sf;
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const WorkItem w = global_item(args, it);
                const int kb64 = w.kblocks64;
                if (!wait_phase(smem_addr(acc_empty), acc_phase ^ 1u, sh, args, kRoleMma, (int)it, -1)) {
                    ok = false;
                    break;
                }
                acc_phase ^= 1u;
                tc_fence_after();
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
                    if (!wait_phase(smem_addr(&sf_full[stage]), phase, sh, args, kRoleMma, (int)it, kb)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acc0 = kb > w.kb_begin ? 1u : 0u;
                    if (kb64 - kb * 4 >= 4) {
                        tc_mma_nvfp4_pair(tmem_base, da + 0, db + 0, idesc, sf + 0, sf + kB, acc0);
                        tc_mma_nvfp4_pair(tmem_base, da + 2, db + 2, idesc, sf + 4, sf + kB + kJ, 1u);
                        tc_mma_nvfp4_pair(tmem_base, da + 4, db + 4, idesc, sf + 8, sf + kB + 2 * kJ, 1u);
                        tc_mma_nvfp4_pair(tmem_base, da + 6, db + 6, idesc, sf + 12, sf + kB + 3 * kJ, 1u);
                    } else {
                        const int ksub = kb64 - kb * 4;
                        for (int j = 0; j < ksub; ++j)
                            tc_mma_nvfp4_pair(tmem_base, da + 2 * j, db + 2 * j, idesc, sf + 4 * j, sf + kB + kJ * j,
                                              (acc0 | (uint32_t)j) ? 1u : 0u);
                    }
                    tc_commit_pair(smem_addr(&empty[stage]), 0x3);
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
                tc_commit_pair(smem_addr(acc_full), 0x3);
            }
            // Every MMA must finish before either CTA frees TMEM or its shared memory.
            tc_commit_pair(smem_addr(drain), 0x3);
        }
        if (lane == 0)
            drain_wait(smem_addr(drain), 0, args, -1);
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------ scale stagers
        // As in the single-CTA kernel (the layout of tcgen05.cp .32x128b.warpx4),
        // with both 128-row halves of the B scales; then one arrival per warp on
        // the leader's sf_full.
        const int quarter = warp % 4;
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
                    stage_scales<true, 2>(src, L::kSfaBytes, col, L::kSfbCol);
                else
                    stage_scales<false, 2>(src, L::kSfaBytes, col, L::kSfbCol);
                tmem_store_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0)
                        mbar_arrive(smem_addr(&sf_full[stage]));
                    else
                        mbar_arrive_remote_relaxed(cluster_map(smem_addr(&sf_full[stage]), 0));
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        // Warp w drains TMEM lane quarter w % 4, column half (w - 6) / 4 (128
        // columns) of this CTA's 128 accumulator rows.
        const int quarter = warp % 4;
        const int chalf = (warp - kEpilogueWarp0) / 4;
        constexpr int kCols = kPairBlockN / 2;
        const uint32_t t_addr = tmem_base + ((uint32_t)(quarter * 32) << 16) + chalf * kCols;
        const int row_in_tile = (int)rank * 128 + quarter * 32 + (int)lane;
        // the leader's acc_empty: a local arrival in the leader, a remote relaxed one in the peer
        const uint32_t acc_empty_leader = cluster_map(smem_addr(acc_empty), 0);
        auto release_accumulator = [&]() {
            if (rank == 0)
                mbar_arrive(smem_addr(acc_empty));
            else
                mbar_arrive_remote_relaxed(acc_empty_leader);
        };
        // C goes out through this warp's two staging buffers and TMA stores
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
            const int m = w.tile_m * kPairBlockM + row_in_tile;
            const int n0 = w.tile_n * kPairBlockN + chalf * kCols;
            const int m_row0 = m - (int)lane;    // first of this warp's 32 rows
            const bool rows_in = m_row0 < M;     // warp-uniform
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
                    release_accumulator();
                if (rows_in) {
#pragma unroll
                    for (int c = 0; c < kCols / 32; ++c)
                        if (n0 + c * 32 < N)
                            out.store(map_c(args, tab, w.group), n0 + c * 32, m_row0, h[c], lane);
                }
            } else {
                // One segment of a split tile, this CTA's 128 rows. Thread e keeps its
                // elements at float4 index (c*8 + f)*256 + e of the slot. Warps whose 32
                // rows lie past M neither write nor read partials; a CTA half with no row
                // inside the group skips the whole exchange (the same for every segment
                // of the tile, so its counter stays untouched).
                const int e = (warp - kEpilogueWarp0) * 32 + (int)lane;
                constexpr int kSlotFloats = 128 * kPairBlockN;
                const bool half_in = w.tile_m * kPairBlockM + (int)rank * 128 < M;  // CTA-uniform
                float4 *ws = reinterpret_cast<float4 *>(args.workspace + (size_t)(2 * w.ws_slot + (int)rank) * kSlotFloats);
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
                    release_accumulator();
                if (!half_in)
                    continue;
                __threadfence();
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
                if (e == 0)
                    sh->last = (atomicAdd(&args.counters[2 * w.split + (int)rank], 1) == w.nseg - 1) ? 1 : 0;
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
                if (sh->last) {
                    __threadfence();
                    // this half's slot of segment sg is 2 * (ws_slot - seg + sg) + rank
                    const float4 *ws0 = reinterpret_cast<const float4 *>(
                        args.workspace + (size_t)(2 * (w.ws_slot - w.seg) + (int)rank) * kSlotFloats);
                    constexpr size_t kSegStride = 2 * (size_t)kSlotFloats / 4;  // float4 units
                    // Each partial is read once, here: its L2 lines are then dropped, so
                    // they are never written back to DRAM. Lane l < 4 drops the 128-byte
                    // line of lanes 8l .. 8l+7, after the whole warp has read it.
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
                            float4 acc[8];
#pragma unroll
                            for (int f = 0; f < 8; ++f)
                                acc[f] = __ldcg(&ws0[(c * 8 + f) * 256 + e]);
                            for (int sg = 1; sg < w.nseg; ++sg) {
                                const float4 *wp = ws0 + (size_t)sg * kSegStride;
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
                        args.counters[2 * w.split + (int)rank] = 0;  // ready for the next launch
                }
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
            }
        }
        out.finish(lane);
    }

    if (warp == kProducerWarp)
        cluster_wait();  // the producer's part of the start-up cluster barrier
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no arrival from the peer after this point
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace nvfp4
