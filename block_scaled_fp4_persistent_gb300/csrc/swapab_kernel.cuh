// swapab_kernel.cuh -- the grouped NVFP4 GEMM with the operands swapped (swap-AB).
//
// For the MoE-shaped sets (few rows of A per group, thousands of rows of B) the
// output tile is computed transposed: the MMA's M side holds 128 rows of B (the
// weights, C's columns) and its N side the group's rows of A (the tokens, C's
// rows), so the MMA is exactly as wide as the group has rows, rounded up to 16,
// instead of being padded to a 128- or 256-row A tile:
//
//   D[n][m] (TMEM, lanes n, columns m) = sum_k B[n][k] sb . A[m][k] sa,  C[m][n] = fp16(D[n][m])
//
// Work item. One 128-row tile of B (weight tile w) against up to two 128-row
// tiles of A (token tiles t0, t0+1), over a range of 256-wide K-stages. The
// K-stages are walked as (k-stage outer, token tile inner): each token tile has
// its own shared-memory stage and its own accumulator, and the second stage's
// B bytes come from L2, fetched from DRAM one stage earlier. So B leaves DRAM
// once however many token tiles a group has (up to 256 rows per item).
//
// One CTA per SM, 14 warps, roles as in the other kernels:
//   warp 0      TMA producer: per stage B (16 KB, the MMA's A operand), A (the
//               group's token box, up to 16 KB, the MMA's B operand) and both
//               scale sets (2 KB each).
//   warp 1      MMA issuer and TMEM owner: per stage four block-scaled MMAs
//               M = 128, N = the token tile's rows rounded up to 16, K = 64.
//   warps 2-5   scale stagers (B's scales in the A-scale slot, A's in the B-scale
//               slot).
//   warps 6-13  epilogue: two warps per TMEM lane quarter; each reads 16 token
//               columns at a time and writes them transposed (a 16 x 32 fp16 box
//               of C: 16 rows of A, 32 rows of B) through shared memory and a TMA
//               store.
// The accumulator is double-buffered (TMEM columns 0-127 and 128-255), so the
// MMAs of the next token tile run while the epilogue drains the last one.
//
// Stream-K. The host may cut items along K anywhere (at K-stage boundaries) so
// that every CTA gets the same number of stages. The segments of a split tile
// write fp32 partials; the last to finish adds them in K order, so the bits do
// not depend on timing. A segment that finds every other segment already
// published (the usual case: a CTA's last segment is the tail-end of a tile whose
// other part another CTA ran first) adds the partials straight to its own
// accumulator and writes none of its own.
#pragma once
#include "gemm_kernel.cuh"

namespace nvfp4 {

constexpr int kSwapStages = 5;
constexpr int kSwapTileRows = 128;  // rows of B per tile, and the most rows of A per token tile

// Item flags of this kernel (beside kItemBShared and kItemSfRowMajor):
//   bits  8-12  N of token tile 0 / 16       bits 13-17  N of token tile 1 / 16 (0: one token tile)
//   bits 18-22  rows of the group's A box / 16 (what each A copy brings, zero-filled past M)
constexpr int kSwapNt0Shift = 8, kSwapNt1Shift = 13, kSwapBoxShift = 18;
__host__ __device__ inline int swap_nt(int flags, int j) { return ((flags >> (j ? kSwapNt1Shift : kSwapNt0Shift)) & 31) * 16; }
__host__ __device__ inline int swap_ntok(int flags) { return ((flags >> kSwapNt1Shift) & 31) ? 2 : 1; }
__host__ __device__ inline int swap_box_rows(int flags) { return ((flags >> kSwapBoxShift) & 31) * 16; }

template <int STAGES>
struct SwapLayout {
    static constexpr int kWBytes = kSwapTileRows * kRowBytes;   // 128 rows of B: 16 KB
    static constexpr int kTBytes = kSwapTileRows * kRowBytes;   // up to 128 rows of A: 16 KB
    static constexpr int kSfwBytes = 4 * kScaleBlockBytes;      // 2 KB
    static constexpr int kSftBytes = 4 * kScaleBlockBytes;      // 2 KB
    static constexpr int kStageBytes = kWBytes + kTBytes + kSfwBytes + kSftBytes;  // 36 KB
    static constexpr int kOffT = kWBytes;
    static constexpr int kOffSfw = kWBytes + kTBytes;
    static constexpr int kRingBytes = STAGES * kStageBytes;
    static constexpr int kEpiBuf = 16 * 64;  // one transposed box: 16 rows of A x 32 fp16 columns
    static constexpr int kOffEpi = kRingBytes;
    static constexpr int kEpiBytes = kEpilogueWarps * 2 * kEpiBuf;
    // barriers: full[S], empty[S], sf_full[S], acc_full[2], acc_empty[2], drain, then the TMEM base word
    static constexpr int kBarBytes = (3 * STAGES + 5) * 8 + 16;
    static constexpr int kSmemBytes = 1024 + kRingBytes + kEpiBytes + kBarBytes + 64;
    // TMEM: accumulators at columns 0 and 128, then one scale slot of 32 columns per
    // stage: B's scales at +0 .. 15 (k-block j at +4j), A's at +16 .. 31.
    static constexpr uint32_t kAccCols = 128;
    static constexpr uint32_t kSfCol0 = 2 * kAccCols;
    static constexpr uint32_t kSfColsPerStage = 32;
    static constexpr int kPartialFloats = kSwapTileRows * kSwapTileRows;  // one fp32 partial slot
    static_assert(kStageBytes % 1024 == 0, "stage slots must keep 1024-byte alignment");
    static_assert(kSfCol0 + STAGES * kSfColsPerStage <= kTmemCols, "TMEM budget");
};

// An epilogue warp's transposed way out for C: two 1 KB buffers of 16 rows x 64
// bytes, alternated, each the source of one TMA store of a box of 16 rows of C
// (rows of A) x 32 columns (rows of B). Lane l holds column l of the box.
struct TransposeStager {
    uint8_t *bufs;  // 2 * 1 KB
    uint32_t n = 0;

    // h[i] holds the fp16 values of box rows 2i (low half) and 2i + 1 (high half) of column `lane`.
    __device__ __forceinline__ void store(const CUtensorMap *tmap, int x, int y, const uint32_t (&h)[8], uint32_t lane)
    {
        uint8_t *buf = bufs + (n & 1) * 1024;
        ++n;
        if (lane == 0)
            bulk_wait_group_read<1>();
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            *reinterpret_cast<uint16_t *>(buf + (2 * i) * 64 + lane * 2) = (uint16_t)(h[i] & 0xffffu);
            *reinterpret_cast<uint16_t *>(buf + (2 * i + 1) * 64 + lane * 2) = (uint16_t)(h[i] >> 16);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmap, x, y, smem_addr(buf));
            bulk_commit_group();
        }
    }

    __device__ __forceinline__ void finish(uint32_t lane)
    {
        if (lane == 0)
            bulk_wait_group<0>();
        __syncwarp();
    }
};

__device__ __forceinline__ void pack16(const uint32_t (&v)[16], uint32_t (&h)[8])
{
#pragma unroll
    for (int i = 0; i < 8; ++i)
        h[i] = pack_half2(v[2 * i], v[2 * i + 1]);
}

template <int STAGES>
__global__ void __launch_bounds__(kThreads, 1) nvfp4_swapab_gemm_kernel(const __grid_constant__ KernelArgs args)
{
    using L = SwapLayout<STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffEpi + L::kEpiBytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *sf_full = bars + 2 * STAGES;
    uint64_t *acc_full = bars + 3 * STAGES;   // [2]
    uint64_t *acc_empty = acc_full + 2;       // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_base_word = reinterpret_cast<uint32_t *>(drain + 1);
    SharedState *sh = reinterpret_cast<SharedState *>(tmem_base_word + 2);

    const int warp = threadIdx.x / 32;
    const uint32_t lane = threadIdx.x % 32;
    const Table *tab = args.table;
    const uint32_t item_begin = args.list_begin[blockIdx.x];
    const uint32_t item_end = args.list_begin[blockIdx.x + 1];
    WorkItem first_item{};
    if (warp == kProducerWarp && lane == 0 && item_begin < item_end)
        first_item = global_item(args, item_begin);
    if (warp == kProducerWarp)
        prefetch_table_maps(tab, args.num_groups, lane);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
            mbar_init(smem_addr(&sf_full[s]), 4);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_addr(&acc_full[x]), 1);
            mbar_init(smem_addr(&acc_empty[x]), kEpilogueWarps);
        }
        mbar_init(smem_addr(drain), 1);
        sh->abort = 0;
        fence_barrier_init();
    }
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
        if (lane == 0) {
            grid_dependency_wait();
            const uint64_t pol_t = policy_evict_last();     // A: re-read for every tile of B
            const uint64_t pol_w_stream = policy_evict_first();
            const uint64_t pol_w_shared = policy_evict_normal();
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
                const int ntok = swap_ntok(w.flags);
                const uint32_t tbytes = (uint32_t)swap_box_rows(w.flags) * kRowBytes;
                const int32_t yw = w.tile_n * kSwapTileRows;
                // B's copy for the first of two token tiles is read again one stage later
                // (from L2), so it is not marked for early eviction; nor where another item
                // reads the same B tile.
                const bool w_shared = (w.flags & kItemBShared) != 0;
                const size_t tok_sf_step = (size_t)kb64 * kScaleBlockBytes;  // the next 128 rows of A's scales
                for (int kb = w.kb_begin; ok && kb < w.kb_end; ++kb) {
                    for (int j = 0; j < ntok; ++j, ++kiter) {
                        if (!wait_phase(smem_addr(&empty[stage]), phase ^ 1u, sh, args, kRoleProducer, (int)it, kb)) {
                            ok = false;
                            break;
                        }
                        const int ksub = min(4, kb64 - kb * 4);
                        const uint32_t sf_bytes = (uint32_t)ksub * kScaleBlockBytes;
                        const uint32_t slot = smem_addr(ring + stage * L::kStageBytes);
                        const uint32_t fb = smem_addr(&full[stage]);
                        const int32_t yt = w.a_row + j * kSwapTileRows;
                        mbar_arrive_expect_tx(fb, L::kWBytes + tbytes + 2 * sf_bytes);
                        if (!(args.fault_skip_load >= 0 && blockIdx.x == 0 && kiter == (uint32_t)args.fault_skip_load)) {
                            const uint64_t pol_w = (w_shared || j + 1 < ntok) ? pol_w_shared : pol_w_stream;
                            tma_load_2d(slot, tmap_b, kb * kRowBytes, yw, fb, pol_w);
                            tma_load_2d(slot + L::kOffT, tmap_a, kb * kRowBytes, yt, fb, pol_t);
                            if (sf_rm) {  // K % 256 == 0: a whole stage, 16 bytes x 128 rows each
                                tma_load_2d(slot + L::kOffSfw, &ge.tmap_sfb, kb * kSfRowBytes, yw, fb, pol_w);
                                tma_load_2d(slot + L::kOffSfw + L::kSfwBytes, &ge.tmap_sfa, kb * kSfRowBytes, yt, fb,
                                            pol_t);
                            } else {
                                bulk_load(slot + L::kOffSfw, w.sfb + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb,
                                          pol_w);
                                bulk_load(slot + L::kOffSfw + L::kSfwBytes,
                                          w.sfa + j * tok_sf_step + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb,
                                          pol_t);
                            }
                        }
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
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
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint64_t kDescStep = (uint64_t)(L::kStageBytes >> 4);
            const uint64_t desc_w0 = operand_desc(smem_addr(ring));
            const uint64_t desc_t0 = operand_desc(smem_addr(ring) + L::kOffT);
            uint32_t stage = 0, phase = 0, acc_use = 0;
            uint64_t dw = desc_w0, dt = desc_t0;
            uint32_t sf = tmem_sf;
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const WorkItem w = global_item(args, it);
                const int kb64 = w.kblocks64;
                const int ntok = swap_ntok(w.flags);
                const uint32_t idesc[2] = {mma_idesc_nvfp4(128, (uint32_t)swap_nt(w.flags, 0)),
                                           mma_idesc_nvfp4(128, (uint32_t)max(16, swap_nt(w.flags, 1)))};
                for (int kb = w.kb_begin; ok && kb < w.kb_end; ++kb) {
                    for (int j = 0; j < ntok; ++j) {
                        const uint32_t u = acc_use + (uint32_t)j, x = u & 1u;
                        if (kb == w.kb_begin) {
                            // the epilogue must have drained this accumulator's previous tile
                            if (!wait_phase(smem_addr(&acc_empty[x]), ((u >> 1) & 1u) ^ 1u, sh, args, kRoleMma, (int)it,
                                            -1)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        if (!wait_phase(smem_addr(&sf_full[stage]), phase, sh, args, kRoleMma, (int)it, kb)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + x * L::kAccCols;
                        const uint32_t acc0 = kb > w.kb_begin ? 1u : 0u;
                        const uint32_t id = idesc[j];
                        if (kb64 - kb * 4 >= 4) {
                            tc_mma_nvfp4(d, dw + 0, dt + 0, id, sf + 0, sf + 16, acc0);
                            tc_mma_nvfp4(d, dw + 2, dt + 2, id, sf + 4, sf + 20, 1u);
                            tc_mma_nvfp4(d, dw + 4, dt + 4, id, sf + 8, sf + 24, 1u);
                            tc_mma_nvfp4(d, dw + 6, dt + 6, id, sf + 12, sf + 28, 1u);
                        } else {
                            const int ksub = kb64 - kb * 4;
                            for (int q = 0; q < ksub; ++q)
                                tc_mma_nvfp4(d, dw + 2 * q, dt + 2 * q, id, sf + 4 * q, sf + 16 + 4 * q,
                                             (acc0 | (uint32_t)q) ? 1u : 0u);
                        }
                        tc_commit(smem_addr(&empty[stage]));
                        if (kb == w.kb_end - 1)
                            tc_commit(smem_addr(&acc_full[x]));
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
                }
                acc_use += (uint32_t)ntok;
            }
            tc_commit(smem_addr(drain));
            drain_wait(smem_addr(drain), 0, args, -1);
        }
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------ scale stagers
        // B's scales (the MMA's A side) from the slot's first 2 KB, A's (its B side)
        // from the next 2 KB: the single-CTA kernel's stage_scales with one half.
        const int quarter = warp % 4;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (uint32_t it = item_begin; ok && it < item_end; ++it) {
            const WorkItem w = global_item(args, it);
            const int nst = (w.kb_end - w.kb_begin) * swap_ntok(w.flags);
            for (int s = 0; s < nst; ++s) {
                if (!warp_wait_phase(smem_addr(&full[stage]), phase, sh, args, kRoleScales, (int)it, s)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = ring + stage * L::kStageBytes + L::kOffSfw + lane * 16;
                const uint32_t col = tmem_sf + lane_off + stage * L::kSfColsPerStage;
                if (w.flags & kItemSfRowMajor)
                    stage_scales<true, 1>(src, L::kSfwBytes, col, 16);
                else
                    stage_scales<false, 1>(src, L::kSfwBytes, col, 16);
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
        // Warp w reads TMEM lane quarter w % 4 (rows 32q .. 32q+31 of the B tile) and
        // every other 16-column chunk of the token tile, starting at (w - 6) / 4.
        const int quarter = warp % 4;
        const int chalf = (warp - kEpilogueWarp0) / 4;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        const int row = quarter * 32 + (int)lane;  // row of the B tile this thread holds
        TransposeStager out{smem + L::kOffEpi + (warp - kEpilogueWarp0) * 2 * L::kEpiBuf};
        if (warp == kEpilogueWarp0)
            prefetch_scale_maps(tab, args.num_groups, lane);
        uint32_t acc_use = 0;
        int fenced = -1;  // the group whose C map lane 0 (which issues the stores) last fenced
        grid_dependency_wait();
        for (uint32_t it = item_begin; it < item_end; ++it) {
            const WorkItem w = global_item(args, it);
            const GroupEntry &ge = tab->group(w.group);
            const int M = ge.M, N = ge.N;
            if (lane == 0 && w.group >= kParamMapGroups && w.group != fenced) {  // before the wait: the fence overlaps the MMAs
                tensormap_acquire(map_c(args, tab, w.group));
                fenced = w.group;
            }
            const int ntok = swap_ntok(w.flags);
            const int n0 = w.tile_n * kSwapTileRows + quarter * 32;  // this warp's first column of C
            bool stop = false;
            for (int j = 0; j < ntok; ++j) {
                const uint32_t u = acc_use + (uint32_t)j, x = u & 1u;
                if (!warp_wait_phase(smem_addr(&acc_full[x]), (u >> 1) & 1u, sh, args, kRoleEpilogue, (int)it, j)) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                const uint32_t t_addr = lane_base + x * L::kAccCols;
                const int nch = swap_nt(w.flags, j) / 16;  // 16-column chunks of this token tile
                const int m0 = (w.tile_m + j) * kSwapTileRows;  // first row of A (and of C) of this token tile
                auto release = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_addr(&acc_empty[x]));
                };
                auto store_chunk = [&](int c, const uint32_t (&h)[8]) {
                    if (n0 < N && m0 + 16 * c < M)
                        out.store(map_c(args, tab, w.group), n0, m0 + 16 * c, h, lane);
                };
                if (w.split < 0) {
                    // whole tile: every chunk of this warp -> fp16 registers, the
                    // accumulator released, then the transposed stores
                    uint32_t h[4][8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = chalf + 2 * k;
                        if (c < nch) {
                            uint32_t v[16];
                            tmem_load_16cols(t_addr + c * 16, v);
                            tmem_load_wait();
                            reg_fence(v);
                            pack16(v, h[k]);
                        }
                    }
                    release();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = chalf + 2 * k;
                        if (c < nch)
                            store_chunk(c, h[k]);
                    }
                    continue;
                }
                // One segment of a split tile (token tile j). Partial slot of this
                // segment: ws_slot + j; of segment sg: ws_slot + (sg - seg) * ntok + j.
                // Thread (row) keeps chunk c's 16 floats as float4 index (4c + f) * 128 + row.
                const int e = (warp - kEpilogueWarp0) * 32 + (int)lane;
                int *counter = args.counters + w.split + j;
                float4 *slot0 = reinterpret_cast<float4 *>(args.workspace) +
                                (size_t)(w.ws_slot - w.seg * ntok + j) * (L::kPartialFloats / 4);
                const size_t seg_stride = (size_t)ntok * (L::kPartialFloats / 4);
                if (e == 0)
                    sh->last = ld_acquire_gpu(counter) == w.nseg - 1 ? 2 : 0;  // 2: every other segment published
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);
                const bool fast = sh->last == 2;
                named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);  // sh->last read before rewritten
                bool last = fast;
                if (!fast) {
                    // the partial waits in L2 until the tile's last segment reads it (then drops it)
                    const uint64_t pol_keep = policy_evict_last();
                    float4 *mine = slot0 + (size_t)w.seg * seg_stride;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = chalf + 2 * k;
                        if (c < nch) {
                            uint32_t v[16];
                            tmem_load_16cols(t_addr + c * 16, v);
                            tmem_load_wait();
                            reg_fence(v);
#pragma unroll
                            for (int f = 0; f < 4; ++f)
                                st_global_keep(&mine[(4 * c + f) * 128 + row], v[4 * f], v[4 * f + 1], v[4 * f + 2],
                                               v[4 * f + 3], pol_keep);
                        }
                    }
                    release();
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
                    for (int k = 0; k < 4; ++k) {
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
                        release();
                    named_barrier_sync(kEpilogueBarrier, kEpilogueWarps * 32);  // every partial read
                    if (e == 0)
                        *counter = 0;  // ready for the next launch
                    // the partials were read once: drop their L2 lines without writing them back
                    for (int sg = 0; sg < w.nseg; ++sg) {
                        if (fast && sg == w.seg)
                            continue;
                        const float4 *p = slot0 + (size_t)sg * seg_stride;
                        for (int l = e; l < nch * 4 * 128 / 8; l += kEpilogueWarps * 32)
                            discard_l2_line(p + 8 * l);
                    }
                }
            }
            if (stop)
                break;
            acc_use += (uint32_t)ntok;
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
