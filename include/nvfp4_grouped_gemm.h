/*
 * nvfp4_grouped_gemm.h -- C ABI of the grouped NVFP4 block-scaled GEMM library
 * (libnvfp4gg.so, built for sm_103a).
 *
 * The operation, for each group i < g (one kernel launch for all groups):
 *
 *   C_i[m][n] = fp16( sum_k e2m1(A_i[m][k]) * e4m3(SFA_i[m][k/16])
 *                          * e2m1(B_i[n][k]) * e4m3(SFB_i[n][k/16]) )
 *
 * Sources:
 *  - page 3 (kernelindex.com submission 444497), kernel header comment:
 *    C[i](M_i x N_i) = A[i](M_i x K_i) . B[i](N_i x K_i)^T, with E2M1 data,
 *    E4M3FN scales and fp16 output;
 *  - page 2 (submission 505431), python section, `custom_kernel_fallback`:
 *    dequantise, multiply each 16-element block by its scale, take the
 *    product in fp32 and cast to fp16.
 * The tensor cores add the products in fp32, so the result is one of the
 * fp16 values near the exact sum. It agrees with the exact result within
 * 1e-3 * sum_k |a*sa*b*sb| + 1 fp16 ulp.
 *
 * All pointers in Nvfp4Problem are DEVICE pointers on the current CUDA device.
 * The caller owns every buffer and the stream. Every call is stream-ordered and
 * asynchronous: it never synchronises the stream, and the inputs must stay
 * valid until the stream has run the launched work.
 *
 * Return codes: NVFP4_OK (0) or a negative NVFP4_ERR_* value. Arguments are
 * checked on the host before anything is queued. When a check fails, nothing
 * is launched.
 */
#ifndef NVFP4_GROUPED_GEMM_H
#define NVFP4_GROUPED_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t. NULL means the legacy default stream. */
typedef struct CUstream_st *nvfp4_stream_t;

enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = -1,        /* g < 0, NULL probs, negative sizes, NULL pointer of a non-empty operand, bad sf_layout, 0 < ldc < N, reserved != 0 */
    NVFP4_ERR_ALIGNMENT = -2,          /* a pointer not 16-byte aligned, K % 64 != 0, N % 8 != 0 or ldc % 8 != 0 */
    NVFP4_ERR_UNSUPPORTED_DEVICE = -3, /* current device is not compute capability 10.3 (sm_103a) */
    NVFP4_ERR_CUDA = -4,               /* a CUDA runtime or driver call failed; see nvfp4_last_cuda_error() */
    NVFP4_ERR_TIMEOUT = -5,            /* a kernel gave up a bounded wait; reported by nvfp4_device_status() */
    NVFP4_ERR_TOO_LARGE = -6,          /* a size beyond the library's limits (e.g. M, N or K >= 2^24, or 2^23 groups) */
    NVFP4_ERR_CAPTURE = -7             /* nvfp4_grouped_gemm_noalloc called on a stream being captured into a graph */
};

/* Scale-factor layouts of SFA/SFB. */
enum {
    /* The 128 x 4 blocked layout: see nvfp4_prepack_scales(). This is the layout
     * the kernel reads. */
    NVFP4_SF_PREPACKED = 0,
    /* Row-major [rows][K/16]. Where K % 256 == 0 (rows of K/16 bytes, a multiple of
     * 16) the GEMM kernel reads them directly: each K-stage's 16 scale bytes per row
     * arrive by TMA and the kernel rearranges them on their way into tensor memory,
     * so the call is one launch, as fast as with prepacked scales. Otherwise (or with
     * NVFP4_OPT_SF_DIRECT 0) the call first runs the prepack kernel into a
     * library-owned workspace (one extra launch), then the GEMM. */
    NVFP4_SF_ROWMAJOR = 1
};

/* One GEMM of the group.
 *  M, N, K  : sizes. M, N >= 0; K >= 0 with K % 64 == 0 (the MMA consumes K in
 *             steps of 64); N % 8 == 0 (16-byte rows of C); each < 2^24.
 *             M == 0 or N == 0 leaves the group out. K == 0 writes C = 0.
 *  A        : [M][K/2] bytes, row-major. Byte j of a row holds element 2j in its
 *             low nibble and element 2j+1 in its high nibble (page 2, python
 *             section, `dequantize_fp4`). E2M1 code: sign bit 3, magnitude
 *             0, .5, 1, 1.5, 2, 3, 4, 6 for codes 0..7.
 *  B        : [N][K/2] bytes, the same packing. B is N x K, and C = A . B^T.
 *  SFA, SFB : E4M3 scale bytes, one per 16 consecutive K of a row, in the layout
 *             sf_layout names. The scale type the tensor core reads is unsigned
 *             (UE4M3), so the sign bit must be 0. 0x7F is NaN and not allowed.
 *  C        : [M][N] fp16, row-major, rows ldc elements apart. Only m < M and n < N
 *             are written.
 *  ldc      : elements between consecutive rows of C. 0 means N (the pages' layout, a
 *             dense C). A library extension, for writing a column block of a wider
 *             matrix (e.g. one GPU's N-range of a call that is split across GPUs): then
 *             ldc >= N, ldc % 8 == 0 (16-byte rows), and C points at the block's first
 *             element.
 *  reserved : must be 0.
 *  A, B, SFA, SFB and C must be 16-byte aligned. */
typedef struct {
    int32_t M, N, K;
    int32_t sf_layout;
    const void *A;
    const void *B;
    const void *SFA;
    const void *SFB;
    void *C;
    int32_t ldc;
    int32_t reserved;
} Nvfp4Problem;

/* The grouped GEMM: one persistent kernel launch for all g problems (plus a
 * prepack launch when some row-major scales have K % 256 != 0, plus a memset per
 * K == 0 group).
 *
 * probs is read during the call only. The library keeps, per distinct problem
 * set, a device-side table: tensor maps, per-group pointers and the tile
 * schedule (and, where the schedule splits tiles along K, their fp32 workspace
 * and counters). The table is cached by a hash of probs, so a repeated call
 * uploads nothing. Calls on different streams may overlap on the GPU when their
 * problem sets differ; calls with the same problem set write the same C and
 * share its table, so they must not overlap.
 *
 * CUDA graphs: once a problem set has been called once outside a capture (its
 * table, and any prepack workspace of the stream, then exist), a call records
 * into a graph being captured on its stream: it allocates, uploads and
 * synchronises nothing.
 *
 * g == 0 is a no-op and returns NVFP4_OK. Errors: see the enum above. A
 * timeout inside the kernel is reported only by nvfp4_device_status(). */
int nvfp4_grouped_gemm(int g, const Nvfp4Problem *probs, nvfp4_stream_t stream);

/* Size in bytes of the blocked scale layout for a rows x K operand:
 * 128*ceil(rows/128) * 4*ceil(K/64). Returns 0 when rows <= 0 or K <= 0. */
size_t nvfp4_prepacked_scale_bytes(int rows, int K);

/* Scale prepack: row-major [rows][K/16] E4M3 bytes -> the 128 x 4 blocked layout
 * that the tensor core's scale copy reads. Page 4 (submission 482006),
 * `to_blocked_gpu`, defines the layout. Pad the rows to a multiple of 128 and
 * the scale columns to a multiple of 4 with zeros. Cut the result into 512-byte
 * blocks, one per (128-row tile, 4 scale columns). Blocks are ordered
 * row-tile major, with K blocks inner. Inside a block, row r = 32*i + j and
 * column c land at byte j*16 + i*4 + c.
 *  sf_rowmajor : device, rows*(K/16) bytes.
 *  sf_blocked  : device, nvfp4_prepacked_scale_bytes(rows, K) bytes, written
 *                in full, padding included.
 *  K % 16 == 0. Both pointers 16-byte aligned. One launch, stream-ordered.
 *  rows == 0 or K == 0 is a no-op. */
int nvfp4_prepack_scales(const void *sf_rowmajor, int rows, int K, void *sf_blocked, nvfp4_stream_t stream);

/* The same prepack for n operands at once (e.g. SFA and SFB of every group of a
 * call): operand i reads sf_rowmajor[i] ([rows[i]][K[i]/16] bytes, device) and
 * writes sf_blocked[i] (nvfp4_prepacked_scale_bytes(rows[i], K[i]) bytes,
 * device), with the rules of nvfp4_prepack_scales for each. The four arrays are
 * host arrays of n entries, read during the call only. One launch for up to 32
 * operands (more take one launch per 32). Operands with rows == 0 or K == 0 are
 * skipped; n == 0 is a no-op. Every operand is checked before anything is
 * launched. */
int nvfp4_prepack_scales_batch(int n, const void *const *sf_rowmajor, const int *rows, const int *K,
                               void *const *sf_blocked, nvfp4_stream_t stream);

/* Reads and clears the current device's error word, which kernels set when a
 * bounded wait runs out. Synchronises `stream` first.
 *  *status = NVFP4_OK, or NVFP4_ERR_TIMEOUT if any launch since the last read
 *  gave up a wait.
 *  detail (may be NULL) receives 4 words: the code, the role (0 producer,
 *  1 MMA issuer, 2 epilogue, 3 teardown, 4 scale stagers), the work item and
 *  the k-stage at which the first timeout happened.
 * Returns NVFP4_OK or an NVFP4_ERR_* code of its own. */
int nvfp4_device_status(nvfp4_stream_t stream, int *status, int32_t *detail);

/* A static, human-readable name for a return code. */
const char *nvfp4_status_string(int code);

/* The cudaError_t value of the last failed CUDA call (0 if none). */
int nvfp4_last_cuda_error(void);

/* The name of the kernel variant that the last successful GEMM call of this
 * process launched (for profiles and logs), e.g. "nvfp4_pair_gemm_kernel<5>" or
 * "nvfp4_grouped_gemm_kernel<128,5>"; "none" before the first launch. A static
 * string: the caller does not free it. */
const char *nvfp4_last_kernel(void);

/* How many kernels the last successful GEMM call of this process launched: 1
 * (the GEMM), or 2 when row-major scales first went through the prepack kernel;
 * 0 before the first launch. */
int nvfp4_last_launches(void);

/* How many A tensor maps the table of the last successful GEMM call holds: the
 * number of active groups, less one for every group that continues an M-fusion
 * run (NVFP4_OPT_M_FUSION); 0 before the first launch. */
int nvfp4_last_a_maps(void);

/* Options for tests and tuning. They apply to the calls that follow, are
 * process-wide, and take part in the table cache's key.
 *  NVFP4_OPT_CTA_PAIR      : the kernel kind. 0 = automatic, 1 = CTA pairs, 2 = single
 *                             CTAs, 3 = swapped operands on single CTAs, 4 = swapped
 *                             operands on CTA pairs.
 *                             CTA pairs: each cluster of two CTAs computes 256 x 256
 *                             output tiles with the pair form of the MMA (M = 256),
 *                             each SM loading its own 128 A rows and half of the B
 *                             tile. Swapped operands (swap-AB): the output tile is
 *                             computed transposed, 128 (single) or 256 (pairs) rows of
 *                             B on the MMA's M side and the group's rows of A, rounded
 *                             up to 16, on its N side (up to 2 x 128 per item on single
 *                             CTAs, 256 on pairs), so a group with few rows wastes no
 *                             MMA width and loads only the rows it has; their tile
 *                             lists are cut along K (stream-K) where that shortens the
 *                             busiest list (SPLIT_TAIL 0 turns that off).
 *                             Automatic (when BLOCK_N and STAGES are 0 too): swapped
 *                             operands on single CTAs when every group has at most 32
 *                             rows of A, else whichever of pairs and single CTAs
 *                             finishes its busiest tile list sooner by a measured
 *                             per-stage cost model (pairs for the MoE-sized sets,
 *                             single CTAs for small sets that would leave SMs idle).
 *                             BLOCK_N and STAGES apply to unswapped single CTAs only.
 *  NVFP4_OPT_BLOCK_N       : 0 = automatic (128), or 128 or 256: the width of
 *                             the single-CTA output tiles (and the MMA's N)
 *  NVFP4_OPT_STAGES        : 0 = automatic (the deepest shared-memory ring that
 *                             fits: 5 stages at BLOCK_N 128, 3 at 256, 5 for
 *                             pairs), or 2 (single CTAs)
 *  NVFP4_OPT_MAX_CTAS      : 0 = one CTA per SM, or an upper bound on the grid
 *                             (pairs: on twice the number of pairs)
 *  NVFP4_OPT_PREFETCH_STAGES: -1 = automatic (0), or 0..64: how many K-stages
 *                             ahead of its shared-memory ring each CTA prefetches
 *                             its operands into L2
 *  NVFP4_OPT_SPLIT_TAIL    : 1 = single CTAs only (default), 2 = single CTAs and
 *                             CTA pairs, 0 = off. When all tiles have the same K
 *                             and do not divide evenly among the CTAs, the last
 *                             partial wave of tiles is cut along K so that every CTA
 *                             does the same work (fp32 partials in a library-owned
 *                             workspace, summed in K order: results are deterministic).
 *                             It is applied only where it saves at least an eighth of
 *                             the busiest CTA's work. 3 = the small-grid fill on single
 *                             CTAs (pairs: off): the same, and where there are fewer
 *                             tiles than SMs the grid stays at one CTA per SM and every
 *                             tile is cut, so that all SMs share the K-stages; it
 *                             measured slower on the two-group shapes than whole tiles
 *                             on fewer SMs, hence opt-in.
 *  NVFP4_OPT_WAIT_TIMEOUT_US: the bound of every wait inside the kernel
 *                             (default 2,000,000 us)
 *  NVFP4_OPT_SF_DIRECT     : 1 = row-major scales are read directly by the GEMM
 *                             kernel where K % 256 == 0 (default), 0 = always
 *                             prepacked by an extra launch first
 *  NVFP4_OPT_PDL           : 0 = off (default), 1 = the GEMM kernel is launched
 *                             with programmatic stream serialization: it may begin
 *                             (barriers, TMEM, its tables) while the previous kernel
 *                             in the stream finishes, and waits for that kernel
 *                             (griddepcontrol.wait) before it reads or writes any of
 *                             the caller's memory. For callers that chain kernels.
 *  NVFP4_OPT_M_FUSION      : 1 = on (default), 0 = off. M-fusion (page 2 of the
 *                             sources, `_merge_groups`), on CTA pairs (the kernel for
 *                             the many-group sets): consecutive active groups
 *                             with the same K whose A rows follow one another in
 *                             memory (A of group i+1 starts where group i's M rows
 *                             end, as when the caller passes slices of one
 *                             concatenated A) share one A tensor map spanning the
 *                             run, and for row-major scales read by the kernel, one
 *                             SFA map (their SFA rows must follow one another too).
 *                             Results are the same bits either way; N may differ
 *                             within a run. A tile's rows past its group's M then
 *                             read the next group's rows, which only reach output
 *                             rows that are never written.
 *  NVFP4_OPT_FAULT_SKIP_LOAD: -1 = off (default). Otherwise the producer of
 *                             CTA 0 skips the copies of its k-stage with that
 *                             global index. The consumer's wait then runs out
 *                             and the kernel reports NVFP4_ERR_TIMEOUT instead
 *                             of hanging. Only for testing the timeout path.
 * Returns NVFP4_OK or NVFP4_ERR_INVALID_ARG. */
enum {
    NVFP4_OPT_BLOCK_N = 1,
    NVFP4_OPT_STAGES = 2,
    NVFP4_OPT_MAX_CTAS = 3,
    NVFP4_OPT_WAIT_TIMEOUT_US = 4,
    NVFP4_OPT_FAULT_SKIP_LOAD = 5,
    NVFP4_OPT_PREFETCH_STAGES = 6,
    NVFP4_OPT_SPLIT_TAIL = 7,
    NVFP4_OPT_CTA_PAIR = 8,
    NVFP4_OPT_SF_DIRECT = 9,
    NVFP4_OPT_PDL = 10,
    NVFP4_OPT_M_FUSION = 11
};
int nvfp4_set_option(int option, int64_t value);

/* Frees every cached table and workspace of every device. Synchronises each
 * device that holds one. Calls made afterwards start again from empty caches.
 * A CUDA graph that captured calls of this library reads their tables when it is
 * replayed: do not replay such a graph after nvfp4_release (capture it again). */
void nvfp4_release(void);

/* The grouped GEMM for callers that cannot allocate device memory. The pages
 * have no counterpart: this is a library convenience.
 *
 * Who needs it: code that must not call cudaMalloc/cudaFree, or anything that
 * allocates on the device. Examples: code running inside a custom device
 * allocator or an out-of-memory handler, or a runtime that owns every byte of
 * device memory and forbids libraries to take more. nvfp4_grouped_gemm
 * allocates its cached problem tables, its error word and (for row-major
 * scales) a workspace. This entry point allocates none of them. Its only
 * device memory beyond the caller's A, B, SFA, SFB and C is one fixed 256 KB
 * array built into the library. Every GPU that loads the library holds that
 * array until the process exits.
 *
 * Same arguments and results as nvfp4_grouped_gemm, with these limits:
 *  - Scales NVFP4_SF_PREPACKED, or NVFP4_SF_ROWMAJOR where K % 256 == 0 (read
 *    directly by the kernel). Row-major scales with another K: NVFP4_ERR_INVALID_ARG.
 *  - The problem table must fit the array:
 *      128 + 640*g' + 4*(grid+1) (rounded up to 16) + 64*tiles <= 262144 - 256 bytes,
 *    where g' counts the groups with M, N, K > 0,
 *    tiles = sum ceil(M/128)*ceil(N/128) and grid = min(tiles, SM count).
 *    In practice that is up to about 4,000 tiles of 128 x 128 for a few
 *    groups. A larger set returns NVFP4_ERR_TOO_LARGE and launches nothing.
 *  - Every call shares the one array. A call rewrites the table in stream
 *    order, and a kernel that is still running on another stream would read
 *    the new table: calls that can overlap on the GPU race and must not be made.
 *  - The first call on each device does a one-time set-up with that device
 *    current: it checks the device, looks up the array's device address
 *    (cudaGetSymbolAddress) and sets the kernel's shared-memory limit.
 *  - It must not be captured into a CUDA graph: each call copies its table from
 *    a static host buffer that the next call overwrites, so a replayed graph
 *    would launch with another call's table. On a stream that is capturing it
 *    returns NVFP4_ERR_CAPTURE and queues nothing.
 *  - The kernel's error words live in the same array and are sticky: a wait that
 *    runs out records NVFP4_ERR_TIMEOUT there (C may then be partly written).
 *    nvfp4_noalloc_status() reads and clears them; nvfp4_device_status() does not
 *    see them.
 * Each call encodes its tensor maps and copies the table (a few KB) from a
 * static host buffer before the launch. There is no cache. */
int nvfp4_grouped_gemm_noalloc(int g, const Nvfp4Problem *probs, nvfp4_stream_t stream);

/* The error words of nvfp4_grouped_gemm_noalloc's kernel on the current device,
 * read and cleared, like nvfp4_device_status() for the other entry point. The
 * pages have no counterpart. Synchronises `stream` first, then reads the fixed
 * array through its symbol (cudaMemcpyFromSymbol), so it allocates nothing.
 *  *status = NVFP4_OK, or NVFP4_ERR_TIMEOUT if a no-allocation launch since the
 *  last read gave up a wait; detail (may be NULL) receives the 4 words (code,
 *  role, work item, k-stage), as for nvfp4_device_status().
 * Returns NVFP4_OK or an NVFP4_ERR_* code of its own. */
int nvfp4_noalloc_status(nvfp4_stream_t stream, int *status, int32_t *detail);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_GROUPED_GEMM_H */
