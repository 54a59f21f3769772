// swapab_pair_kernel.cuh -- the swapped-operand kernel on CTA pairs.
//
// The output tile is computed transposed, as in swapab_kernel.cuh, with the pair
// form of the block-scaled MMA (tcgen05.mma.cta_group::2, M = 256, N = the tile's
// rows of A rounded up to 16, at most 256):
//
//   D[n][m] = sum_k B[n][k] sb . A[m][k] sa   (n: 256 rows of B, m: up to 256 rows of A)
//
// Per K-stage each CTA of the pair loads
//   * its own 128 rows of B (rank r: rows 128r .. 128r+127 of the tile),
//   * its half of the tile's rows of A (rank r: rows r*NT/2 .. (r+1)*NT/2 - 1),
//   * the scale blocks of its own B rows and of all the tile's A rows,
// so an SM moves 16 KB of B plus NT/2 rows of A per stage, where a 256 x 256 tile
// of the unswapped pair kernel moves 16 KB of each. Each CTA's TMEM receives its own
// 128 rows of B (lanes) x NT columns of A; the epilogue writes them transposed.
//
// Everything else (warp roles, barriers across the pair, relaxed remote arrivals,
// bounded waits) follows pair_kernel.cuh; split tiles (stream-K) follow
// swapab_kernel.cuh, per CTA half: partial slot 2 * slot + rank, counter 2 * split +
// rank.
#pragma once
#include "pair_kernel.cuh"
#include "swapab_kernel.cuh"

namespace nvfp4 {

constexpr int kSwapPairStages = 5;
constexpr int kSwapPairRows = 256;  // rows of B per pair tile; and the most rows of A per tile

// Item flags of this kernel (beside kItemSfRowMajor):
//   kItemA2   rows 128..255 of the tile's B exist (else rank 1 reads rank 0's scale blocks)
//   kItemB2   rows 128..255 of the tile's A exist (else the second scale half repeats the first)
//   bits 8-12 the MMA's N / 16 (the group's rows of A, rounded up to 16, at most 256); each
//             CTA's box of A has N/2 rows
constexpr int kSwapPairNtShift = 8;
__host__ __device__ inline int swap_pair_nt(int flags) { return ((flags >> kSwapPairNtShift) & 31) * 16; }

template <int STAGES>
struct SwapPairLayout {
    static constexpr int kWBytes = 128 * kRowBytes;          // this CTA's 128 rows of B: 16 KB
    static constexpr int kTBytes = 128 * kRowBytes;          // its half of the tile's A rows: up to 16 KB
    static constexpr int kSfwBytes = 4 * kScaleBlockBytes;   // 2 KB
    static constexpr int kSftBytes = 8 * kScaleBlockBytes;   // 4 KB: both 128-row halves of A's scales
    static constexpr int kStageBytes = kWBytes + kTBytes + kSfwBytes + kSftBytes;  // 38 KB
    static constexpr int kOffT = kWBytes;
    static constexpr int kOffSfw = kWBytes + kTBytes;
    static constexpr int kOffSft = kOffSfw + kSfwBytes;
    static constexpr int kRingBytes = STAGES * kStageBytes;
    static constexpr int kEpiBuf = 16 * 64;
    static constexpr int kOffEpi = kRingBytes;
    static constexpr int kEpiBytes = kEpilogueWarps * 2 * kEpiBuf;
    static constexpr int kBarBytes = (3 * STAGES + 3) * 8 + 16;
    static constexpr int kSmemBytes = 1024 + kRingBytes + kEpiBytes + kBarBytes + 64;
    // TMEM: the accumulator at columns 0 .. 255, then a scale slot of 48 columns per stage
    // (B's scales at +0 .. 15, A's two halves at +16 .. 47), as in the pair kernel.
    static constexpr uint32_t kSfCol0 = 256;
    static constexpr uint32_t kSfbCol = 16;
    static constexpr uint32_t kSfColsPerStage = 48;
    static constexpr int kPartialFloats = 128 * 256;  // one CTA's half of a split tile's fp32 partial
    static_assert(kStageBytes % 1024 == 0, "stage slots must keep 1024-byte alignment");
    static_assert(kSfCol0 + STAGES * kSfColsPerStage <= kTmemCols, "TMEM budget");
};

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    nvfp4_swapab_pair_kernel(const __grid_constant__ PairArgs args)
{
    using L = SwapPairLayout<STAGES>;
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
    WorkItem first_item{};
    if (warp == kProducerWarp && lane == 0 && item_begin < item_end)
        first_item = pair < kParamFirstItems ? item_of(args.first[pair]) : global_item(args, item_begin);
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
            grid_dependency_wait();
            const uint64_t pol_t = policy_evict_last();  // A: re-read for every tile of B
            const uint64_t pol_w = policy_evict_first();
            uint32_t stage = 0, phase = 0, kiter = 0;
            int fenced = -1;
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const WorkItem w = it == item_begin ? first_item : global_item(args, it);
                const GroupEntry &ge = tab->group(w.group);  // address only: the tensor maps
                const bool sf_rm = (w.flags & kItemSfRowMajor) != 0;
                const CUtensorMap *tmap_a = map_a(args, tab, w.group), *tmap_b = map_b(args, tab, w.group);
                if (w.group != fenced) {  // maps read from the table: an acquire fence before first use
                    fenced = w.group;
                    if (w.group >= kParamMapGroups) {
                        tensormap_acquire(tmap_a);
                        tensormap_acquire(tmap_b);
                    }
                    if (sf_rm) {
                        tensormap_acquire(&ge.tmap_sfa);
                        tensormap_acquire(&ge.tmap_sfb);
                    }
                }
                const int kb64 = w.kblocks64;
                const int half_rows = swap_pair_nt(w.flags) / 2;  // rows of A in each CTA's box
                const int32_t yw = w.tile_n * kSwapPairRows + (int)rank * 128;
                const int32_t yt = w.tile_m * kSwapPairRows + (int)rank * half_rows;
                const size_t half = (size_t)kb64 * kScaleBlockBytes;
                // a 128-row half wholly past the matrix reads the first half's scale blocks:
                // its operand rows are zero (TMA fills them), so the scales need only be finite
                const uint8_t *sfw = w.sfb + ((rank == 1 && (w.flags & kItemA2)) ? half : 0);
                const uint8_t *sft[2] = {w.sfa, w.sfa + ((w.flags & kItemB2) ? half : 0)};
                const uint32_t tbytes = (uint32_t)half_rows * kRowBytes;
                for (int kb = w.kb_begin; kb < w.kb_end; ++kb, ++kiter) {
                    if (!wait_phase(smem_addr(&empty[stage]), phase ^ 1u, sh, args, kRoleProducer, (int)it, kb)) {
                        ok = false;
                        break;
                    }
                    const int ksub = min(4, kb64 - kb * 4);
                    const uint32_t sf_bytes = (uint32_t)ksub * kScaleBlockBytes;
                    const uint32_t slot = smem_addr(ring + stage * L::kStageBytes);
                    const uint32_t fb = smem_addr(&full[stage]);
                    mbar_arrive_expect_tx(fb, L::kWBytes + tbytes + 3 * sf_bytes);
                    if (!(args.fault_skip_load >= 0 && blockIdx.x == 0 && kiter == (uint32_t)args.fault_skip_load)) {
                        tma_load_2d(slot, tmap_b, kb * kRowBytes, yw, fb, pol_w);
                        tma_load_2d(slot + L::kOffT, tmap_a, kb * kRowBytes, yt, fb, pol_t);
                        if (sf_rm) {  // K % 256 == 0: B's 128 rows, A's box of 256 rows (both halves)
                            tma_load_2d(slot + L::kOffSfw, &ge.tmap_sfb, kb * kSfRowBytes, yw, fb, pol_w);
                            tma_load_2d(slot + L::kOffSft, &ge.tmap_sfa, kb * kSfRowBytes, w.tile_m * kSwapPairRows, fb,
                                        pol_t);
                        } else {
                            bulk_load(slot + L::kOffSfw, sfw + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb, pol_w);
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                bulk_load(slot + L::kOffSft + h * 4 * kScaleBlockBytes,
                                          sft[h] + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb, pol_t);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            grid_launch_dependents();
            const uint32_t issued = kiter < (uint32_t)STAGES ? kiter : (uint32_t)STAGES;
            for (uint32_t i = 0; i < issued; ++i) {
                const uint32_t f = kiter - 1 - i;
                drain_wait(smem_addr(&full[f % STAGES]), (f / STAGES) & 1u, args, (int)(f % STAGES));
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------ MMA issuer (leader)
        if (rank == 0 && lane == 0) {
            constexpr uint64_t kDescStep = (uint64_t)(L::kStageBytes >> 4);
            constexpr uint32_t kB = L::kSfbCol, kJ = 8;  // A-scale column of k-block j: kB + kJ*j
            const uint64_t desc_w0 = operand_desc(smem_addr(ring));
            const uint64_t desc_t0 = operand_desc(smem_addr(ring) + L::kOffT);
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            uint64_t dw = desc_w0, dt = desc_t0;
            uint32_t sf = tmem_sf;
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const WorkItem w = global_item(args, it);
                const int kb64 = w.kblocks64;
                const uint32_t idesc = mma_idesc_nvfp4(256, (uint32_t)swap_pair_nt(w.flags));
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
                        tc_mma_nvfp4_pair(tmem_base, dw + 0, dt + 0, idesc, sf + 0, sf + kB, acc0);
                        tc_mma_nvfp4_pair(tmem_base, dw + 2, dt + 2, idesc, sf + 4, sf + kB + kJ, 1u);
                        tc_mma_nvfp4_pair(tmem_base, dw + 4, dt + 4, idesc, sf + 8, sf + kB + 2 * kJ, 1u);
                        tc_mma_nvfp4_pair(tmem_base, dw + 6, dt + 6, idesc, sf + 12, sf + kB + 3 * kJ, 1u);
                    } else {
                        const int ksub = kb64 - kb * 4;
                        for (int j = 0; j < ksub; ++j)
                            tc_mma_nvfp4_pair(tmem_base, dw + 2 * j, dt + 2 * j, idesc, sf + 4 * j, sf + kB + kJ * j,
                                              (acc0 | (uint32_t)j) ? 1u : 0u);
                    }
                    tc_commit_pair(smem_addr(&empty[stage]), 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                        dw = desc_w0;
                        dt = desc_t0;
                        sf = tmem_sf;
                    } else {
                        dw += kDescStep;
                        dt += kDescStep;
                        sf += L::kSfColsPerStage;
                    }
                }
                if (!ok)
                    break;
                tc_commit_pair(smem_addr(acc_full), 0x3);
            }
            tc_commit_pair(smem_addr(drain), 0x3);
        }
        if (lane == 0)
            drain_wait(smem_addr(drain), 0, args, -1);
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------ scale stagers
        // As in the pair kernel: B's scales (the MMA's A side) and both halves of A's.
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
                const uint8_t *src = ring + stage * L::kStageBytes + L::kOffSfw + lane * 16;
                const uint32_t col = tmem_sf + lane_off + stage * L::kSfColsPerStage;
                if (w.flags & kItemSfRowMajor)
                    stage_scales<true, 2>(src, L::kSfwBytes, col, L::kSfbCol);
                else
                    stage_scales<false, 2>(src, L::kSfwBytes, col, L::kSfbCol);
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
        // Warp w reads TMEM lane quarter w % 4 (this CTA's rows 32q .. 32q+31 of B, i.e.
        // columns of C) and every other 16-column chunk of the tile's rows of A, from
        // (w - 6) / 4 on; each chunk leaves as a transposed 16 x 32 box of C.
        const int quarter = warp % 4;
        const int chalf = (warp - kEpilogueWarp0) / 4;
        const uint32_t t_addr = tmem_base + ((uint32_t)(quarter * 32) << 16);
        const int row = quarter * 32 + (int)lane;  // this thread's row of B within this CTA's half
        const uint32_t acc_empty_leader = cluster_map(smem_addr(acc_empty), 0);
        auto release_accumulator = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0)
                    mbar_arrive(smem_addr(acc_empty));
                else
                    mbar_arrive_remote_relaxed(acc_empty_leader);
            }
        };
        TransposeStager out{smem + L::kOffEpi + (warp - kEpilogueWarp0) * 2 * L::kEpiBuf};
        if (warp == kEpilogueWarp0)
            prefetch_scale_maps(tab, args.num_groups, lane);
        uint32_t acc_phase = 0;
        int fenced = -1;  // the group whose C map lane 0 (which issues the stores) last fenced
        grid_dependency_wait();
        for (uint32_t it = item_begin; it < item_end; ++it) {
            const WorkItem w = global_item(args, it);
            const GroupEntry &ge = tab->group(w.group);
            const int M = ge.M, N = ge.N;
            if (lane == 0 && w.group >= kParamMapGroups && w.group != fenced) {
                tensormap_acquire(map_c(args, tab, w.group));
                fenced = w.group;
            }
            if (!warp_wait_phase(smem_addr(acc_full), acc_phase, sh, args, kRoleEpilogue, (int)it, -1))
                break;
            acc_phase ^= 1u;
            tc_fence_after();
            const int nch = swap_pair_nt(w.flags) / 16;
            const int n0 = w.tile_n * kSwapPairRows + (int)rank * 128 + quarter * 32;  // this warp's first column of C
            const int m0 = w.tile_m * kSwapPairRows;                                  // the tile's first row of C
            auto store_chunk = [&](int c, const uint32_t (&h)[8]) {
                if (n0 < N && m0 + 16 * c < M)
                    out.store(map_c(args, tab, w.group), n0, m0 + 16 * c, h, lane);
            };
            if (w.split < 0) {
                // 8 columns per load keeps the temporaries small beside the 64 packed words
                uint32_t h[8][8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int c = chalf + 2 * k;
                    if (c < nch) {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            uint32_t v[8];
                            tmem_load_8cols(t_addr + c * 16 + 8 * q, v);
                            tmem_load_wait();
                            reg_fence(v);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                h[k][4 * q + i] = pack_half2(v[2 * i], v[2 * i + 1]);
                        }
                    }
                }
                release_accumulator();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int c = chalf + 2 * k;
                    if (c < nch)
                        store_chunk(c, h[k]);
                }
                continue;
            }
            // One segment of a split tile, this CTA's 128 rows of B. A CTA half whose rows
            // of B all lie past N skips the exchange (the same for every segment of the
            // tile, so its counter stays untouched).
            const int e = (warp - kEpilogueWarp0) * 32 + (int)lane;
            const bool half_in = w.tile_n * kSwapPairRows + (int)rank * 128 < N;  // CTA-uniform
            if (!half_in) {
                release_accumulator();
                continue;
            }
            int *counter = args.counters + 2 * w.split + (int)rank;
            float4 *slot0 = reinterpret_cast<float4 *>(args.workspace) +
                            (size_t)(2 * (w.ws_slot - w.seg) + (int)rank) * (L::kPartialFloats / 4);
            const size_t seg_stride = 2 * (size_t)(L::kPartialFloats / 4);
            if (e == 0)
                sh->last = ld_acquire_gpu(counter) == w.nseg - 1 ? 2 : 0;  // 2: every other segment published
            named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
            const bool fast = sh->last == 2;
            named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
            bool last = fast;
            if (!fast) {
                const uint64_t pol_keep = policy_evict_last();
                float4 *mine = slot0 + (size_t)w.seg * seg_stride;
#pragma unroll 1
                for (int k = 0; k < 8; ++k) {
                    const int c = chalf + 2 * k;
                    if (c >= nch)
                        break;
                    uint32_t v[16];
                    tmem_load_16cols(t_addr + c * 16, v);
                    tmem_load_wait();
                    reg_fence(v);
#pragma unroll
                    for (int f = 0; f < 4; ++f)
                        st_global_keep(&mine[(4 * c + f) * 128 + row], v[4 * f], v[4 * f + 1], v[4 * f + 2],
                                       v[4 * f + 3], pol_keep);
                }
                release_accumulator();
                __threadfence();
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
                if (e == 0)
                    sh->last = (atomicAdd(counter, 1) == w.nseg - 1) ? 1 : 0;
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
                last = sh->last != 0;
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
            }
            if (last) {
                __threadfence();
#pragma unroll 1
                for (int k = 0; k < 8; ++k) {
                    const int c = chalf + 2 * k;
                    if (c >= nch)
                        break;
                    uint32_t own[16];
                    if (fast) {
                        tmem_load_16cols(t_addr + c * 16, own);
                        tmem_load_wait();
                        reg_fence(own);
                    }
                    float a[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        a[i] = 0.f;
                    for (int sg = 0; sg < w.nseg; ++sg) {
                        if (fast && sg == w.seg) {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                a[i] += __uint_as_float(own[i]);
                            continue;
                        }
                        const float4 *p = slot0 + (size_t)sg * seg_stride;
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            const float4 q = __ldcg(&p[(4 * c + f) * 128 + row]);
                            a[4 * f] += q.x, a[4 * f + 1] += q.y, a[4 * f + 2] += q.z, a[4 * f + 3] += q.w;
                        }
                    }
                    uint32_t h[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        h[i] = pack_half2(__float_as_uint(a[2 * i]), __float_as_uint(a[2 * i + 1]));
                    store_chunk(c, h);
                }
                if (fast)
                    release_accumulator();
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);  // every partial read
                if (e == 0)
                    *counter = 0;  // ready for the next launch
                for (int sg = 0; sg < w.nseg; ++sg) {
                    if (fast && sg == w.seg)
                        continue;
                    const float4 *p = slot0 + (size_t)sg * seg_stride;
                    for (int l = e; l < nch * 4 * 128 / 8; l += kEpilogueWarps * 32)
                        discard_l2_line(p + 8 * l);
                }
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
