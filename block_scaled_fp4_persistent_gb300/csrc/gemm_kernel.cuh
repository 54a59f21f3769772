// gemm_kernel.cuh -- the persistent, warp-specialised grouped NVFP4 GEMM kernel.
//
// One CTA per SM walks its own list of output tiles (group, 128-row tile m,
// BLOCK_N-column tile n). Ten warps share the work:
//   warp 0      TMA producer. It streams 256-wide K-stages of A and B (E2M1,
//               128-byte swizzled rows) and the matching 512-byte scale blocks
//               into a ring of STAGES shared-memory slots.
//   warp 1      MMA issuer; it also owns the TMEM allocation. Per stage it issues
//               four block-scaled MMAs (kind::mxf4nvf4, 16-element scale blocks,
//               K = 64 each) into one of two TMEM accumulators, then commits the
//               stage back to the producer.
//   warps 2-5   epilogue. They load the fp32 accumulator from TMEM, free it for
//               the next tile, round to fp16 and store the rows that lie inside
//               the group.
//   warps 6-9   scale stagers. Per stage each warp reads its rows of the scale
//               blocks from shared memory and writes them into the stage's TMEM
//               scale slot with tcgen05.st, in the layout tcgen05.cp .warpx4
//               would produce.
// The two accumulators let tile t+1's MMAs run while tile t is stored.
//
// Why the stagers exist. On this GPU one tcgen05.cp of a 512-byte scale block
// costs about as much tensor-pipe time as an MMA (measured: ~46 vs ~64 cycles),
// and a 256-wide stage needs 8 of them for 4 MMAs. Issued from the MMA thread,
// the copies more than double the per-stage pipe time. tcgen05.st from four
// other warps writes the same TMEM contents while the MMAs run.
//
// The pages' kernels (page 1 `grouped_gemm_kernel_v4`, page 2
// `group_gemm_kernel_impl`) use the producer/MMA/epilogue split and copy the
// scales with tcgen05.cp from the MMA thread. This kernel differs from them in
// several ways. Scale staging is moved off the MMA thread. Ring and accumulator
// phases are monotone counters carried across tiles, so no barrier is
// re-initialised. The schedule is a per-CTA list built on the host. There is no
// cluster multicast. Every wait is bounded: when one runs out, the kernel
// records an error word and returns, and it never traps.
#pragma once
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"
#include "table.h"

namespace nvfp4 {

constexpr int kThreads = 320;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kEpilogueWarp0 = 2;  // warps 2..5
constexpr int kScaleWarp0 = 6;     // warps 6..9
constexpr int kBlockM = 128;
constexpr int kBlockK = 256;             // K per stage = 128 bytes of E2M1 per row
constexpr int kRowBytes = kBlockK / 2;   // 128
constexpr int kMmaK = 64;                // K per MMA
constexpr int kScaleBlockBytes = 512;    // scales of 128 rows x 64 K
constexpr uint32_t kTmemCols = 512;

// Roles reported in the status words.
constexpr int kRoleProducer = 0, kRoleMma = 1, kRoleEpilogue = 2, kRoleTeardown = 3, kRoleScales = 4;

template <int BN, int STAGES>
struct Layout {
    static constexpr int kABytes = kBlockM * kRowBytes;            // 16 KB
    static constexpr int kBBytes = BN * kRowBytes;                 // 16 KB for BN = 128
    static constexpr int kSfaBytes = 4 * kScaleBlockBytes;         // 2 KB
    static constexpr int kSfbBytes = (BN / 128) * 4 * kScaleBlockBytes;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static constexpr int kOffB = kABytes;
    static constexpr int kOffSfa = kABytes + kBBytes;
    static constexpr int kOffSfb = kOffSfa + kSfaBytes;
    static constexpr int kRingBytes = STAGES * kStageBytes;
    // barriers: full[S], empty[S], sf_full[S], acc_full[2], acc_empty[2], drain, then the TMEM base word
    static constexpr int kBarBytes = (3 * STAGES + 5) * 8 + 16;
    static constexpr int kSmemBytes = 1024 + kRingBytes + kBarBytes + 64;
    // TMEM columns: accumulators at 0 and BN; a 32-column scale slot per stage after them
    // (SFA at +0..15: k-block j at +4j; SFB at +16..31)
    static constexpr uint32_t kSfCol0 = 2 * BN;
    static constexpr uint32_t kSfColsPerStage = 32;
    static_assert(kStageBytes % 1024 == 0, "stage slots must keep 1024-byte alignment");
    static_assert(2 * BN + STAGES * kSfColsPerStage <= (int)kTmemCols, "TMEM budget");
};

struct SharedState {
    volatile int abort;  // set by the first role that gives up a wait
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
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, SharedState *sh, const KernelArgs &args,
                                           int role, int item, int stage)
{
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
// move on before this warp releases the slot).
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

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) nvfp4_grouped_gemm_kernel(const __grid_constant__ KernelArgs args)
{
    static_assert(BN == 128, "only 128-column tiles: the TMEM scale layout of N = 256 is not used");
    using L = Layout<BN, STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern of the operand tiles
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kRingBytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *sf_full = bars + 2 * STAGES;
    uint64_t *acc_full = bars + 3 * STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_base_word = reinterpret_cast<uint32_t *>(drain + 1);
    SharedState *sh = reinterpret_cast<SharedState *>(tmem_base_word + 2);

    const int warp = threadIdx.x / 32;
    const uint32_t lane = threadIdx.x % 32;
    const Table *tab = args.table;
    const uint32_t item_begin = tab->cta_begin(blockIdx.x);
    const uint32_t item_end = tab->cta_begin(blockIdx.x + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
            mbar_init(smem_addr(&sf_full[s]), 4);  // one elected arrive per stager warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&acc_full[b]), 1);
            mbar_init(smem_addr(&acc_empty[b]), 4 * 32);
        }
        mbar_init(smem_addr(drain), 1);
        sh->abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_base_word), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_word;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_b_stream = policy_evict_first();
            const uint64_t pol_b_shared = policy_evict_normal();
            for (int gi = 0; gi < args.num_groups && gi < 64; ++gi) {
                tensormap_prefetch(&tab->group(gi).tmap_a);
                tensormap_prefetch(&tab->group(gi).tmap_b);
            }
            uint32_t stage = 0, phase = 0, kiter = 0;
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const WorkItem w = tab->item(it);
                const GroupEntry &ge = tab->group(w.group);
                const int kb64 = ge.kblocks64;
                const int nk = (kb64 + 3) / 4;
                const uint64_t pol_b = ge.tiles_m > 1 ? pol_b_shared : pol_b_stream;
                const void *tmap_a = &ge.tmap_a;
                const void *tmap_b = &ge.tmap_b;
                const int32_t ya = w.tile_m * kBlockM, yb = w.tile_n * BN;
                const uint8_t *sfa = ge.sfa + (size_t)w.tile_m * kb64 * kScaleBlockBytes;
                const uint8_t *sfb = ge.sfb + (size_t)w.tile_n * (BN / 128) * kb64 * kScaleBlockBytes;
                for (int kb = 0; kb < nk; ++kb, ++kiter) {
                    if (!wait_phase(smem_addr(&empty[stage]), phase ^ 1u, sh, args, kRoleProducer, (int)it, kb)) {
                        ok = false;
                        break;
                    }
                    const int ksub = min(4, kb64 - kb * 4);
                    const uint32_t sf_bytes = (uint32_t)ksub * kScaleBlockBytes;
                    const uint32_t bytes = L::kABytes + L::kBBytes + sf_bytes * (1 + BN / 128);
                    const uint32_t slot = smem_addr(ring + stage * L::kStageBytes);
                    const uint32_t fb = smem_addr(&full[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    if (!(args.fault_skip_load >= 0 && blockIdx.x == 0 && kiter == (uint32_t)args.fault_skip_load)) {
                        tma_load_2d(slot, tmap_a, kb * kRowBytes, ya, fb, pol_a);
                        tma_load_2d(slot + L::kOffB, tmap_b, kb * kRowBytes, yb, fb, pol_b);
                        bulk_load(slot + L::kOffSfa, sfa + (size_t)kb * 4 * kScaleBlockBytes, sf_bytes, fb, pol_a);
#pragma unroll
                        for (int h = 0; h < BN / 128; ++h)
                            bulk_load(slot + L::kOffSfb + h * 4 * kScaleBlockBytes,
                                      sfb + ((size_t)h * kb64 + kb * 4) * kScaleBlockBytes, sf_bytes, fb, pol_b);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Before the CTA may exit, every copy it started must have landed.
            // A full barrier whose last fill was consumed has already flipped its
            // phase, so these waits return at once in a normal run.
            const uint32_t issued = kiter < (uint32_t)STAGES ? kiter : (uint32_t)STAGES;
            for (uint32_t i = 0; i < issued; ++i) {
                const uint32_t f = kiter - 1 - i;
                const uint32_t s = f % STAGES, ph = (f / STAGES) & 1u;
                uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(smem_addr(&full[s]), ph)) {
                    if (global_timer_ns() - t0 > args.timeout_ns) {
                        record_error(args.status, kStatusTimeout, kRoleTeardown, -1, (int)s);
                        break;
                    }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = mma_idesc_nvfp4(kBlockM, BN);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (uint32_t it = item_begin; ok && it < item_end; ++it) {
                const WorkItem w = tab->item(it);
                const int kb64 = tab->group(w.group).kblocks64;
                const int nk = (kb64 + 3) / 4;
                if (!wait_phase(smem_addr(&acc_empty[acc]), acc_phase ^ 1u, sh, args, kRoleMma, (int)it, -1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < nk; ++kb) {
                    // The stagers arrive on sf_full only after the stage's copies landed, so
                    // the full wait below returns at once; it gives this thread its own
                    // acquire of the TMA writes that the MMAs read.
                    if (!wait_phase(smem_addr(&sf_full[stage]), phase, sh, args, kRoleMma, (int)it, kb) ||
                        !wait_phase(smem_addr(&full[stage]), phase, sh, args, kRoleMma, (int)it, kb)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int ksub = min(4, kb64 - kb * 4);
                    const uint32_t slot = smem_addr(ring + stage * L::kStageBytes);
                    const uint32_t sfa_col = tmem_base + L::kSfCol0 + stage * L::kSfColsPerStage;
                    const uint32_t sfb_col = sfa_col + 16;
                    const uint32_t acc_in = kb > 0 ? 1u : 0u;
                    if (ksub == 4) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tc_mma_nvfp4(d_tmem, operand_desc(slot + j * 32), operand_desc(slot + L::kOffB + j * 32),
                                         idesc, sfa_col + 4 * j, sfb_col + 4 * j, (acc_in | (uint32_t)j) ? 1u : 0u);
                    } else {
                        for (int j = 0; j < ksub; ++j)
                            tc_mma_nvfp4(d_tmem, operand_desc(slot + j * 32), operand_desc(slot + L::kOffB + j * 32),
                                         idesc, sfa_col + 4 * j, sfb_col + 4 * j, (acc_in | (uint32_t)j) ? 1u : 0u);
                    }
                    tc_commit(smem_addr(&empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                tc_commit(smem_addr(&acc_full[acc]));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA this thread issued must finish before TMEM is freed.
            tc_commit(smem_addr(drain));
            uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_addr(drain), 0)) {
                if (global_timer_ns() - t0 > args.timeout_ns) {
                    record_error(args.status, kStatusTimeout, kRoleTeardown, -1, -1);
                    break;
                }
            }
        }
    } else if (warp < kScaleWarp0) {
        // ------------------------------------------------------ epilogue
        const int quarter = warp % 4;  // warps 2,3,4,5 -> TMEM lane quarters 2,3,0,1
        const int row_in_tile = quarter * 32 + (int)lane;
        uint32_t acc = 0, acc_phase = 0;
        for (uint32_t it = item_begin; it < item_end; ++it) {
            const WorkItem w = tab->item(it);
            const GroupEntry &ge = tab->group(w.group);
            const int M = ge.M, N = ge.N;
            __half *const C = ge.C;
            if (!wait_phase(smem_addr(&acc_full[acc]), acc_phase, sh, args, kRoleEpilogue, (int)it, -1))
                break;
            tc_fence_after();
            const uint32_t t_addr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
            uint32_t v[BN / 32][32];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
                tmem_load_32cols(t_addr + c * 32, v[c]);
            tmem_load_wait();
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
                reg_fence(v[c]);
            tc_fence_before();
            mbar_arrive(smem_addr(&acc_empty[acc]));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            const int m = w.tile_m * kBlockM + row_in_tile;
            if (m < M) {
                const int n0 = w.tile_n * BN;
                __half *crow = C + (size_t)m * N + n0;
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int col = c * 32 + q * 8;
                        if (n0 + col < N) {
                            uint4 pk;
                            __half2 h0 = __floats2half2_rn(__uint_as_float(v[c][q * 8 + 0]), __uint_as_float(v[c][q * 8 + 1]));
                            __half2 h1 = __floats2half2_rn(__uint_as_float(v[c][q * 8 + 2]), __uint_as_float(v[c][q * 8 + 3]));
                            __half2 h2 = __floats2half2_rn(__uint_as_float(v[c][q * 8 + 4]), __uint_as_float(v[c][q * 8 + 5]));
                            __half2 h3 = __floats2half2_rn(__uint_as_float(v[c][q * 8 + 6]), __uint_as_float(v[c][q * 8 + 7]));
                            pk.x = *reinterpret_cast<uint32_t *>(&h0);
                            pk.y = *reinterpret_cast<uint32_t *>(&h1);
                            pk.z = *reinterpret_cast<uint32_t *>(&h2);
                            pk.w = *reinterpret_cast<uint32_t *>(&h3);
                            *reinterpret_cast<uint4 *>(crow + col) = pk;
                        }
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------ scale stagers
        // Lane r of the warp for TMEM lane quarter q writes TMEM lane 32q + r. Word c of
        // k-block j goes to column 4j + c: the scales of row r + 32c, i.e. bytes
        // 4c..4c+3 of row r of the block. That is the layout tcgen05.cp .32x128b.warpx4
        // produces, repeated in all four quarters.
        const int quarter = warp % 4;  // warps 6,7,8,9 -> quarters 2,3,0,1
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (uint32_t it = item_begin; ok && it < item_end; ++it) {
            const WorkItem w = tab->item(it);
            const int kb64 = tab->group(w.group).kblocks64;
            const int nk = (kb64 + 3) / 4;
            for (int kb = 0; kb < nk; ++kb) {
                if (!warp_wait_phase(smem_addr(&full[stage]), phase, sh, args, kRoleScales, (int)it, kb)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = ring + stage * L::kStageBytes + L::kOffSfa + lane * 16;
                uint32_t ra[16], rb[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a = *reinterpret_cast<const uint4 *>(src + j * kScaleBlockBytes);
                    const uint4 b = *reinterpret_cast<const uint4 *>(src + L::kSfaBytes + j * kScaleBlockBytes);
                    ra[4 * j + 0] = a.x, ra[4 * j + 1] = a.y, ra[4 * j + 2] = a.z, ra[4 * j + 3] = a.w;
                    rb[4 * j + 0] = b.x, rb[4 * j + 1] = b.y, rb[4 * j + 2] = b.z, rb[4 * j + 3] = b.w;
                }
                const uint32_t col = tmem_base + lane_off + L::kSfCol0 + stage * L::kSfColsPerStage;
                tmem_store_16cols(col, ra);
                tmem_store_16cols(col + 16, rb);
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
