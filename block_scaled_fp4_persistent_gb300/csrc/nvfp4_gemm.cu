// nvfp4_gemm.cu -- host side of the grouped NVFP4 GEMM library and its C ABI.
//
// One call runs through these steps:
//  1. Check every argument on the host. Nothing is queued when a check fails.
//  2. Clear C with cudaMemsetAsync for K == 0 groups (the empty sum).
//  3. For row-major scales, run the prepack kernel into a per-stream workspace.
//  4. Find the device table for this problem set: tensor maps, per-group
//     pointers and the per-CTA tile lists. It is cached under an FNV-1a hash of
//     the problem set. On a miss it is built on the host and uploaded with one
//     cudaMemcpyAsync.
//  5. Launch the persistent kernel: one launch for all groups.
//
// The pages cache their launch state the same way, because encoding tensor maps
// is a costly driver call (page 1, `group_gemm`, the FNV-1a keyed caches; page 2,
// `LaunchCache`).
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <list>
#include <map>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "nvfp4_grouped_gemm.h"
#include "gemm_kernel.cuh"
#include "pair_kernel.cuh"
#include "prepack.cuh"
#include "swapab_kernel.cuh"
#include "swapab_pair_kernel.cuh"
#include "table.h"

using namespace nvfp4;

namespace {

// ------------------------------------------------------------------ state --

std::atomic<int> g_last_cuda_error{0};
std::atomic<const char *> g_last_kernel{"none"};  // the variant the last call launched
std::atomic<int> g_last_launches{0};  // kernels the last GEMM call launched (prepack and GEMM)
std::atomic<int> g_last_a_maps{0};    // A tensor maps the last GEMM call's table holds (M-fusion runs)

struct Options {
    std::atomic<int64_t> block_n{0};
    std::atomic<int64_t> stages{0};
    std::atomic<int64_t> max_ctas{0};
    std::atomic<int64_t> timeout_us{2000000};
    std::atomic<int64_t> fault_skip_load{-1};
    std::atomic<int64_t> prefetch_stages{-1};  // -1 = automatic
    std::atomic<int64_t> split_tail{1};  // 0 off, 1 single CTAs only, 2 single CTAs and pairs, 3 fill (single CTAs)
    std::atomic<int64_t> cta_pair{0};  // 0 = automatic, 1 = CTA pairs, 2 = single CTAs
    std::atomic<int64_t> sf_direct{1};  // 1 = row-major scales read by the GEMM kernel where K % 256 == 0
    std::atomic<int64_t> pdl{0};  // 1 = GEMM launches with programmatic stream serialization
    std::atomic<int64_t> m_fusion{1};  // 1 = groups whose A rows follow one another share one A map
} g_opt;

// Launches one of the GEMM kernels. With the PDL option on, the launch allows
// programmatic stream serialization: the kernel may start (set up barriers and
// TMEM, read its own tables) while the previous kernel in the stream finishes;
// it waits for that kernel before it reads or writes the caller's memory.
template <class Kernel, class Args>
cudaError_t launch_kernel(Kernel kernel, unsigned grid, size_t smem, cudaStream_t stream, const Args &args)
{
    if (g_opt.pdl.load() == 0) {
        kernel<<<grid, kThreads, smem, stream>>>(args);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

constexpr int kMaxDevices = 64;
// Kernel variants: BLOCK_N 128 or 256, each with the deepest ring that fits in
// shared memory, or a 2-stage ring (for tests).
constexpr int kDefaultBlockN = 128;
constexpr int kDeepStages128 = 5;  // 5 x 36 KB, + 32 KB of epilogue staging
constexpr int kDeepStages256 = 3;  // 3 x 54 KB, + 32 KB of epilogue staging
constexpr int kDefaultStages = kDefaultBlockN == 256 ? kDeepStages256 : kDeepStages128;
// The CTA-pair kernel: 256 x 256 tiles, 5 x 38 KB ring (its TMEM holds 5 scale slots).
constexpr int kPairStages = 5;
constexpr int kVariantPair = 4;
// The swapped-operand kernel (swap-AB): 128 rows of B on the MMA's M side, a group's
// rows of A (up to 2 x 128 per item) on its N side, stream-K over all SMs.
constexpr int kVariantSwap = 5;
// The same on CTA pairs: 256 rows of B on the MMA's M side (128 per SM), up to 256 rows
// of A on its N side (half per SM), stream-K over the pairs.
constexpr int kVariantSwapPair = 6;
constexpr int kVariantAuto = -1;  // chosen per problem set
// How far ahead of the ring the producer prefetches into L2, in stages.
constexpr int kDefaultPrefetchStages = 0;
constexpr int kMaxDim = 1 << 24;
constexpr size_t kMaxCachedTables = 32;

struct DeviceState {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    int max_smem_optin = 0;
    int *status = nullptr;  // device: 4 words
    bool attr_set[8] = {};
    int pair_clusters = 0;  // CTA pairs of the pair kernel that fit on the device at once
};

std::mutex g_mu;  // guards everything below
DeviceState g_dev[kMaxDevices];

// The memory behind one cached table: the device table, its pinned host copy (the
// source of the asynchronous upload), and for split schedules the fp32 workspace
// and the counters. Blocks are recycled through a per-device pool rather than
// freed, and a block leaves a table only once the work that may read it has
// completed: each stream that launched with the table records an event after the
// launch, and an evicted table's blocks wait in a retiring list until all its
// events have completed. Nothing synchronises.
struct Buffers {
    int device = -1;
    void *dev = nullptr;
    size_t dev_cap = 0;
    void *host = nullptr;
    size_t host_cap = 0;
    float *ws = nullptr;
    size_t ws_cap = 0;
    int *cnt = nullptr;
    size_t cnt_cap = 0;
    std::vector<std::pair<cudaStream_t, cudaEvent_t>> uses;  // one event per stream that used the blocks
    bool untracked = false;  // more streams than tracked: retire only after a device synchronisation
};

struct CachedTable {
    uint64_t key = 0;
    std::vector<uint8_t> signature;  // exact inputs of the table, to rule out hash collisions
    void *dev = nullptr;
    float *workspace = nullptr;      // fp32 partials of split tiles
    int *counters = nullptr;         // one per split tile, 0 between launches
    int splits = 0;
    void *host = nullptr;  // pinned copy, kept alive for the asynchronous upload
    size_t bytes = 0;
    int device = 0;
    int grid = 0;
    int block_n = 0;
    int variant = 0;  // the kernel variant the table was built for
    int a_maps = 0;   // distinct A tensor maps: one per run of groups with consecutive A rows
    bool captured = false;  // used inside a stream capture: a graph may replay it, so it is never evicted
    std::vector<uint32_t> list_begin;  // the table's cta_begin, passed again with each launch
    Buffers buf;
};
// The device address of a cached table's work items.
const int4 *table_items(const CachedTable &t)
{
    const TableHeader *th = static_cast<const TableHeader *>(t.host);
    return reinterpret_cast<const int4 *>(static_cast<const uint8_t *>(t.dev) + th->off_items);
}

std::list<CachedTable> g_tables;  // most recently used first
std::unordered_map<uint64_t, std::list<CachedTable>::iterator> g_table_index;
struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::map<std::pair<int, uintptr_t>, Workspace> g_workspaces;  // key: (device, stream)

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cuda_fail(cudaError_t e)
{
    g_last_cuda_error.store((int)e);
    return NVFP4_ERR_CUDA;
}

#define CUDA_TRY(call)                          \
    do {                                        \
        cudaError_t e_ = (call);                \
        if (e_ != cudaSuccess)                  \
            return cuda_fail(e_);               \
    } while (0)

std::vector<Buffers> g_free_buffers;      // blocks that no queued work reads any more
std::vector<Buffers> g_retiring_buffers;  // blocks of evicted tables, waiting for their events
constexpr size_t kMaxFreeBuffers = 16;    // beyond this, idle blocks are returned to CUDA

size_t pool_round(size_t n) { return n == 0 ? 0 : std::max<size_t>(16384, size_t(1) << (64 - __builtin_clzll(n - 1))); }

void free_buffers(Buffers &b)
{
    for (auto &u : b.uses)
        cudaEventDestroy(u.second);
    b.uses.clear();
    cudaFree(b.dev);
    cudaFree(b.ws);
    cudaFree(b.cnt);
    cudaFreeHost(b.host);
    b = Buffers{};
}

// Whether every event of b has completed (nothing queued reads the blocks).
bool buffers_idle(const Buffers &b)
{
    if (b.untracked)
        return false;
    for (const auto &u : b.uses) {
        cudaError_t q = cudaEventQuery(u.second);
        if (q == cudaErrorNotReady)
            return false;
        if (q != cudaSuccess)
            cudaGetLastError();  // a failed event is not waited for: clear the sticky error
    }
    return true;
}

// Blocks of at least the given sizes on device dev: a free block of the pool that
// fits (the smallest), else new ones with sizes rounded up to powers of two.
int acquire_buffers(int dev, size_t table_bytes, size_t ws_bytes, size_t cnt_bytes, Buffers *out)
{
    for (size_t i = 0; i < g_retiring_buffers.size();) {
        if (buffers_idle(g_retiring_buffers[i])) {
            g_free_buffers.push_back(std::move(g_retiring_buffers[i]));
            g_retiring_buffers.erase(g_retiring_buffers.begin() + i);
        } else {
            ++i;
        }
    }
    int best = -1;
    size_t best_size = SIZE_MAX;
    for (size_t i = 0; i < g_free_buffers.size(); ++i) {
        const Buffers &b = g_free_buffers[i];
        if (b.device != dev || b.dev_cap < table_bytes || b.host_cap < table_bytes || b.ws_cap < ws_bytes ||
            b.cnt_cap < cnt_bytes)
            continue;
        const size_t sz = b.dev_cap + b.ws_cap + b.cnt_cap;
        if (sz < best_size) {
            best_size = sz;
            best = (int)i;
        }
    }
    if (best >= 0) {
        *out = std::move(g_free_buffers[best]);
        g_free_buffers.erase(g_free_buffers.begin() + best);
        return NVFP4_OK;
    }
    Buffers b;
    b.device = dev;
    b.dev_cap = b.host_cap = pool_round(table_bytes);
    b.ws_cap = pool_round(ws_bytes);
    b.cnt_cap = pool_round(cnt_bytes);
    cudaError_t e = cudaMalloc(&b.dev, b.dev_cap);
    if (e == cudaSuccess)
        e = cudaMallocHost(&b.host, b.host_cap);
    if (e == cudaSuccess && b.ws_cap)
        e = cudaMalloc(&b.ws, b.ws_cap);
    if (e == cudaSuccess && b.cnt_cap)
        e = cudaMalloc(&b.cnt, b.cnt_cap);
    if (e != cudaSuccess) {
        free_buffers(b);
        return cuda_fail(e);
    }
    *out = std::move(b);
    return NVFP4_OK;
}

// Blocks that no queued work has touched yet (the table was never uploaded) go
// straight back to the pool; the others wait for their events.
void return_buffers(Buffers &&b, bool used)
{
    if (used) {
        g_retiring_buffers.push_back(std::move(b));
    } else {
        g_free_buffers.push_back(std::move(b));
    }
    while (g_free_buffers.size() > kMaxFreeBuffers) {
        free_buffers(g_free_buffers.front());
        g_free_buffers.erase(g_free_buffers.begin());
    }
}

// After queuing work that reads t's blocks on `stream`: record (or re-record) the
// stream's event. Inside a stream capture the table is marked captured instead:
// a graph may replay the work at any later time, so the table stays cached.
int note_use(CachedTable &t, cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CUDA_TRY(cudaStreamIsCapturing(stream, &cs));
    if (cs != cudaStreamCaptureStatusNone) {
        t.captured = true;
        return NVFP4_OK;
    }
    for (auto &u : t.buf.uses)
        if (u.first == stream) {
            CUDA_TRY(cudaEventRecord(u.second, stream));
            return NVFP4_OK;
        }
    if (t.buf.uses.size() >= 16) {
        t.buf.untracked = true;
        return NVFP4_OK;
    }
    cudaEvent_t ev = nullptr;
    CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    t.buf.uses.push_back({stream, ev});
    CUDA_TRY(cudaEventRecord(ev, stream));
    return NVFP4_OK;
}

// Takes a table out of the cache; its blocks retire once their events complete.
void evict_table(std::list<CachedTable>::iterator it)
{
    auto idx = g_table_index.find(it->key);
    if (idx != g_table_index.end() && idx->second == it)
        g_table_index.erase(idx);
    if (it->buf.untracked) {
        // more streams used it than are tracked: wait for the device once
        cudaDeviceSynchronize();
        it->buf.untracked = false;
        for (auto &u : it->buf.uses)
            cudaEventDestroy(u.second);
        it->buf.uses.clear();
    }
    return_buffers(std::move(it->buf), true);
    g_tables.erase(it);
}


uint64_t fnv1a(const void *data, size_t n, uint64_t h = 1469598103934665603ull)
{
    const uint8_t *p = static_cast<const uint8_t *>(data);
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 1099511628211ull;
    }
    return h;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Caller holds g_mu.
int device_state(int dev, DeviceState **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
        CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
        CUDA_TRY(cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev));
        CUDA_TRY(cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        d.supported = (major == 10 && minor == 3);
        if (d.supported) {
            CUDA_TRY(cudaMalloc(&d.status, 4 * sizeof(int)));
            CUDA_TRY(cudaMemset(d.status, 0, 4 * sizeof(int)));
        }
        d.ready = true;
    }
    if (!d.supported)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return NVFP4_OK;
}

int get_encoder()
{
    if (g_encode)
        return NVFP4_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
    if (q != cudaDriverEntryPointSuccess || !fn)
        return cuda_fail(cudaErrorNotSupported);
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return NVFP4_OK;
}

// The tensor-map encoder is a driver call. Runtime calls bind the device's primary
// context to a host thread lazily, driver calls do not: in a thread that has made no
// context-binding runtime call yet (a worker thread whose first call to this library
// misses the table cache) the encoder fails with CUDA_ERROR_INVALID_CONTEXT. So before
// encoding, a thread with no current context gets the primary context of `dev` bound,
// as the runtime would have done; a context that the caller made current stays.
int ensure_context(int dev)
{
    using CtxGetCurrent = CUresult (*)(CUcontext *);
    static const CtxGetCurrent get_current = []() -> CtxGetCurrent {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<CtxGetCurrent>(fn);
    }();
    CUcontext ctx = nullptr;
    if (get_current && get_current(&ctx) == CUDA_SUCCESS && ctx)
        return NVFP4_OK;
    CUDA_TRY(cudaSetDevice(dev));
    return NVFP4_OK;
}

// A row-major uint8 matrix [rows][row_bytes] read as boxes of 128 bytes x box_rows,
// with the 128-byte swizzle the MMA's K-major operand layout expects.
int encode_operand_map(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows)
{
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error.store(10000 + (int)r);
        return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

// Row-major scales [rows][K/16] read as boxes of 16 bytes (one 256-K stage) x
// box_rows, unswizzled: a box lands as box_rows rows of 16 bytes. Rows past the
// matrix read as zero. Without scales to read (prepacked groups), a valid map of the
// buffer's first 16 bytes, which the kernel never copies through.
int encode_scale_map(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows)
{
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {16, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error.store(10000 + (int)r);
        return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}
int encode_unused_scale_map(CUtensorMap *map, const void *base) { return encode_scale_map(map, base, 16, 1, 1); }

// The fp16 output [M][N] as 32 x 32 boxes (64 bytes per box row) with the
// 64-byte swizzle, for TMA stores from the epilogue's staging buffers.
int encode_output_map(CUtensorMap *map, void *C, uint64_t M, uint64_t N, uint64_t ldc)
{
    cuuint64_t dims[2] = {N, M};
    cuuint64_t strides[1] = {ldc * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, C, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error.store(10000 + (int)r);
        return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

// The fp16 output [M][N] as boxes of 16 rows x 32 columns, unswizzled: the swapped
// kernel's transposed epilogue stores one such box per 16 rows of A and 32 of B.
int encode_output_map_t(CUtensorMap *map, void *C, uint64_t M, uint64_t N, uint64_t ldc)
{
    cuuint64_t dims[2] = {N, M};
    cuuint64_t strides[1] = {ldc * 2};
    cuuint32_t box[2] = {32, 16};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, C, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error.store(10000 + (int)r);
        return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

int check_problem(const Nvfp4Problem &p)
{
    if (p.M < 0 || p.N < 0 || p.K < 0 || p.ldc < 0 || p.reserved != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (p.ldc >= kMaxDim)
        return NVFP4_ERR_TOO_LARGE;
    if (p.sf_layout != NVFP4_SF_PREPACKED && p.sf_layout != NVFP4_SF_ROWMAJOR)
        return NVFP4_ERR_INVALID_ARG;
    if (p.M >= kMaxDim || p.N >= kMaxDim || p.K >= kMaxDim)
        return NVFP4_ERR_TOO_LARGE;
    if (p.M == 0 || p.N == 0)
        return NVFP4_OK;
    if (!p.C || (p.ldc != 0 && p.ldc < p.N))
        return NVFP4_ERR_INVALID_ARG;
    if (p.K % 64 != 0 || p.N % 8 != 0 || p.ldc % 8 != 0 || !aligned16(p.C))
        return NVFP4_ERR_ALIGNMENT;
    if (p.K == 0)
        return NVFP4_OK;
    if (!p.A || !p.B || !p.SFA || !p.SFB)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(p.A) || !aligned16(p.B) || !aligned16(p.SFA) || !aligned16(p.SFB))
        return NVFP4_ERR_ALIGNMENT;
    return NVFP4_OK;
}

// One active group as the table sees it (scale pointers already blocked).
struct ActiveGroup {
    int32_t M, N, K;
    int32_t sf_rowmajor;  // 1: the kernel reads row-major scales through tensor maps
    const void *A, *B, *SFA, *SFB;
    void *C;
    int32_t ldc = 0;      // elements between rows of C (0: N)
    int32_t pad = 0;
    int64_t c_stride() const { return ldc ? ldc : N; }
};

// C = 0 for a K == 0 group (the empty sum), rows ldc apart.
cudaError_t clear_output(const Nvfp4Problem &p, cudaStream_t stream)
{
    const size_t row = (size_t)p.N * sizeof(__half);
    if (p.ldc == 0 || p.ldc == p.N)
        return cudaMemsetAsync(p.C, 0, row * p.M, stream);
    return cudaMemset2DAsync(p.C, (size_t)p.ldc * sizeof(__half), 0, row, (size_t)p.M, stream);
}

// Tile lists. The kernel runs kPipes pipelines per CTA, and each pipeline walks
// its own list; list number c * kPipes + p belongs to pipeline p of CTA c.
// Tiles are numbered group by group, and inside a group B-strip by B-strip
// (tile_n outer, tile_m inner). Tile t goes to CTA t % grid, pipeline
// (t / grid) % kPipes. So the CTAs that run at the same moment hold
// consecutive tiles: the m-tiles that share one strip of B read it from HBM
// once and from L2 after that. Each SM's two pipelines take alternate waves.
inline int list_of_tile(size_t t, int grid) { return (int)(t % grid) * kPipes + (int)((t / grid) % kPipes); }

// A work item with the producer's fields filled in (see WorkItem): the scale
// blocks of the tile's first 128-row tiles of A and B, and whether the second
// 128-row halves (of a 256-row A tile, of a 256-wide B tile) hold any rows.
WorkItem make_item(const ActiveGroup &g, int group, int m, int n, int kb_begin, int kb_end, int split, int seg,
                   int nseg, int slot, int block_m, int block_n)
{
    WorkItem w{};
    w.group = group;
    w.tile_m = m;
    w.tile_n = n;
    w.kb_begin = kb_begin;
    w.kb_end = kb_end;
    w.split = split;
    w.seg = seg;
    w.nseg = nseg;
    w.ws_slot = slot;
    w.a_row = m * block_m;  // the group's own A map; M-fusion rebases it
    const int kb64 = g.K / 64;
    w.kblocks64 = kb64;
    const int row_tiles_a = (g.M + 127) / 128, row_tiles_b = (g.N + 127) / 128;
    const int ra = m * (block_m / 128), rb = n * (block_n / 128);
    w.flags = ((g.M + block_m - 1) / block_m > 1 ? kItemBShared : 0) |
              (block_m == 256 && ra + 1 < row_tiles_a ? kItemA2 : 0) |
              (block_n == 256 && rb + 1 < row_tiles_b ? kItemB2 : 0) | (g.sf_rowmajor ? kItemSfRowMajor : 0) |
              (group << kItemAMapShift);
    const size_t blocks = (size_t)kb64 * kScaleBlockBytes;
    w.sfa = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(g.SFA) + (size_t)ra * blocks);
    w.sfb = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(g.SFB) + (size_t)rb * blocks);
    return w;
}

struct Schedule {
    std::vector<WorkItem> items;
    std::vector<uint32_t> list_begin;
    int grid = 0;
    int splits = 0;    // split tiles (one counter each)
    int ws_slots = 0;  // fp32 partial slots (one per segment of a split tile)
};

// Tiles are numbered group by group, and inside a group B-strip by B-strip
// (tile_n outer, tile_m inner), so that the CTAs running at the same moment
// hold neighbouring tiles: the m-tiles that share one strip of B read it from
// HBM once and from L2 after that.
//
// Balance. When every tile has the same number of K-stages and there are more
// tiles than CTAs, the first floor(T/G)*G tiles go round-robin, whole. The
// remaining T mod G tiles (the tail) are cut along K so that every CTA gets the
// same number of tail stages: CTA c takes stages [c*W/G, (c+1)*W/G) of the
// tail's W stages. A tail tile that lands on several CTAs is a split tile: its
// segments write fp32 partials and the last to finish stores C. Otherwise (mixed
// K, T <= G, or split off) every tile goes whole to CTA t % G.
// split: kSplitNone, kSplitTail (the above), or kSplitFill: the same, and with fewer
// tiles than CTAs the grid stays at grid_cap and every tile joins the tail, so that
// the whole grid shares the K-stages (the small-grid fill).
constexpr int kSplitNone = 0, kSplitTail = 1, kSplitFill = 2;
Schedule build_schedule(const std::vector<ActiveGroup> &gs, int block_m, int block_n, int grid_cap, int split)
{
    struct Tile {
        int group, m, n, nk;
    };
    std::vector<Tile> tiles;
    for (int gi = 0; gi < (int)gs.size(); ++gi) {
        const int tm = (gs[gi].M + block_m - 1) / block_m, tn = (gs[gi].N + block_n - 1) / block_n;
        const int nk = (gs[gi].K / 64 + 3) / 4;
        for (int n = 0; n < tn; ++n)
            for (int m = 0; m < tm; ++m)
                tiles.push_back(Tile{gi, m, n, nk});
    }
    Schedule sc;
    const size_t T = tiles.size();
    bool uniform = true;
    for (const Tile &t : tiles)
        uniform = uniform && t.nk == tiles[0].nk;
    // Split only where it shortens the busiest CTA by at least an eighth (and two
    // stages): each split costs a partial write and a reduction. With fewer tiles than
    // CTAs only the fill mode splits: spreading every tile over the whole grid measured
    // slower on the two-group sets (K = 4096: 21.1 us against 15.3 whole), so it is opt-in.
    auto split_pays = [&](int G) {
        const int64_t nk = tiles[0].nk;
        const int64_t unbalanced = (int64_t)((T + G - 1) / G) * nk;
        const int64_t balanced = ((int64_t)T * nk + G - 1) / G;
        return unbalanced - balanced >= 2 && (unbalanced - balanced) * 8 >= unbalanced;
    };
    sc.grid = std::max(1, std::min<int>((int)T, grid_cap));
    if (split == kSplitFill && uniform && T > 0 && T < (size_t)grid_cap && split_pays(grid_cap))
        sc.grid = grid_cap;
    const int G = sc.grid, lists = G * kPipes;
    size_t whole = T;
    if (split != kSplitNone && uniform && T % G != 0 && (T > (size_t)G || split == kSplitFill) && split_pays(G))
        whole = (T / G) * G;
    // Split segments go at the head of their CTA's list: their partial writes and
    // reductions then overlap the whole tiles that follow instead of ending the launch.
    std::vector<std::vector<WorkItem>> head(lists), per(lists);
    for (size_t t = 0; t < whole; ++t) {
        const Tile &x = tiles[t];
        per[list_of_tile(t, G)].push_back(make_item(gs[x.group], x.group, x.m, x.n, 0, x.nk, -1, 0, 1, 0, block_m, block_n));
    }
    if (whole < T) {
        const int nk = tiles[0].nk;
        const int64_t W = (int64_t)(T - whole) * nk;
        auto cta_start = [&](int c) { return (int64_t)c * W / G; };
        for (size_t r = 0; r < T - whole; ++r) {
            const Tile &x = tiles[whole + r];
            const int64_t a = (int64_t)r * nk, b = a + nk;
            // CTAs whose tail ranges meet [a, b)
            int c0 = (int)std::min<int64_t>(G - 1, a * G / W);
            while (c0 > 0 && cta_start(c0) > a)
                --c0;
            while (cta_start(c0 + 1) <= a)
                ++c0;
            std::vector<std::pair<int, std::pair<int, int>>> segs;  // cta, [kb_begin, kb_end)
            for (int c = c0; c < G && cta_start(c) < b; ++c) {
                const int64_t lo = std::max(a, cta_start(c)), hi = std::min(b, cta_start(c + 1));
                if (hi > lo)
                    segs.push_back({c, {(int)(lo - a), (int)(hi - a)}});
            }
            const int nseg = (int)segs.size();
            const int split = nseg > 1 ? sc.splits++ : -1;
            for (int j = 0; j < nseg; ++j) {
                const int slot = nseg > 1 ? sc.ws_slots++ : 0;
                head[segs[j].first * kPipes].push_back(
                    make_item(gs[x.group], x.group, x.m, x.n, segs[j].second.first, segs[j].second.second, split, j, nseg,
                              slot, block_m, block_n));
            }
        }
    }
    sc.list_begin.assign(lists + 1, 0);
    for (int l = 0; l < lists; ++l) {
        sc.list_begin[l] = (uint32_t)sc.items.size();
        sc.items.insert(sc.items.end(), head[l].begin(), head[l].end());
        sc.items.insert(sc.items.end(), per[l].begin(), per[l].end());
    }
    sc.list_begin[lists] = (uint32_t)sc.items.size();
    return sc;
}

// ------------------------------------------------------ swap-AB schedule --
//
// Tiles of the swapped-operand kernel, numbered group by group, then by 128-row
// tile w of B, then by item p: item p of tile w covers the 128-row tiles 2p and
// 2p + 1 of A (one where the group has an odd number). An item's cost is its
// shared-memory stages: K-stages x token tiles. With stream-K the items are laid
// end to end and cut into grid-many equal spans at K-stage boundaries; a cut that
// would leave fewer than kSwapMinSeg K-stages on either side of a tile moves to
// the tile's edge. A tile cut into several segments is a split tile (fp32
// partials, summed in K order by the last segment to finish). Without stream-K
// (or where it would not shorten the busiest CTA) whole items go to the CTAs
// longest first, each to the least loaded.
constexpr int kSwapMinSeg = 2;

struct SwapTile {
    int group, w, t0, ntok, nk;
};

inline int round16(int x) { return (x + 15) / 16 * 16; }

WorkItem make_swap_item(const ActiveGroup &g, int gi, const SwapTile &t, int kb_begin, int kb_end, int split, int seg,
                        int nseg, int slot)
{
    WorkItem w{};
    w.group = gi;
    w.tile_m = t.t0;
    w.tile_n = t.w;
    w.kb_begin = kb_begin;
    w.kb_end = kb_end;
    w.split = split;
    w.seg = seg;
    w.nseg = nseg;
    w.ws_slot = slot;
    const int kb64 = g.K / 64;
    w.kblocks64 = kb64;
    const int ntt = (g.M + kSwapTileRows - 1) / kSwapTileRows;
    const int nt0 = round16(std::min(kSwapTileRows, g.M - kSwapTileRows * t.t0));
    const int nt1 = t.ntok == 2 ? round16(std::min(kSwapTileRows, g.M - kSwapTileRows * (t.t0 + 1))) : 0;
    const int box = g.M <= kSwapTileRows ? round16(g.M) : kSwapTileRows;
    w.flags = ((ntt + 1) / 2 > 1 ? kItemBShared : 0) | (g.sf_rowmajor ? kItemSfRowMajor : 0) |
              ((nt0 / 16) << kSwapNt0Shift) | ((nt1 / 16) << kSwapNt1Shift) | ((box / 16) << kSwapBoxShift);
    w.a_row = kSwapTileRows * t.t0;
    const size_t blocks = (size_t)kb64 * kScaleBlockBytes;
    w.sfa = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(g.SFA) + (size_t)t.t0 * blocks);
    w.sfb = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(g.SFB) + (size_t)t.w * blocks);
    return w;
}

// Lists for grid_cap CTAs (or CTA pairs) over `tiles` in their order, each tile
// costing nk * ntok stages: whole tiles longest first, each to the least loaded list,
// or stream-K spans (see above), whichever leaves the busiest list shorter (a split
// segment counted two stages dearer). make(tile, kb_begin, kb_end, split, seg, nseg,
// slot) builds an item; a split tile takes `ntok` split ids and each of its segments
// `ntok` slots. Lists that come out empty are dropped.
template <class Make>
Schedule stream_k_schedule(const std::vector<SwapTile> &tiles, int grid_cap, bool stream_k, Make make)
{
    Schedule sc;
    const size_t T = tiles.size();
    std::vector<int64_t> start(T + 1, 0);
    for (size_t t = 0; t < T; ++t)
        start[t + 1] = start[t] + (int64_t)tiles[t].nk * tiles[t].ntok;
    const int64_t U = start[T];

    // whole items, longest first, each to the least loaded CTA
    const int Gw = std::max(1, std::min<int>((int)T, grid_cap));
    std::vector<int> owner(T, 0);
    std::vector<int64_t> load(Gw, 0);
    {
        std::vector<size_t> order(T);
        for (size_t t = 0; t < T; ++t)
            order[t] = t;
        std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) {
            return start[a + 1] - start[a] > start[b + 1] - start[b];
        });
        for (size_t t : order) {
            int best = 0;
            for (int c = 1; c < Gw; ++c)
                if (load[c] < load[best])
                    best = c;
            owner[t] = best;
            load[best] += start[t + 1] - start[t];
        }
    }
    const int64_t makespan_whole = *std::max_element(load.begin(), load.end());

    // stream-K spans
    const int Gs = std::max(1, grid_cap);
    std::vector<int64_t> b(Gs + 1, 0);
    b[Gs] = U;
    for (int c = 1; c < Gs; ++c) {
        const int64_t x = ((int64_t)c * U + Gs / 2) / Gs;
        const size_t t = (size_t)(std::upper_bound(start.begin(), start.end(), x) - start.begin()) - 1;
        int64_t snapped = x;
        if (t < T) {
            const int ntok = tiles[t].ntok, nk = tiles[t].nk;
            int kb = (int)((x - start[t] + ntok / 2) / ntok);
            if (kb < kSwapMinSeg)
                kb = 0;
            else if (nk - kb < kSwapMinSeg)
                kb = nk;
            snapped = start[t] + (int64_t)kb * ntok;
            // nor a short segment after the previous cut inside the same tile
            if (b[c - 1] > start[t] && snapped > b[c - 1] && snapped - b[c - 1] < (int64_t)kSwapMinSeg * ntok)
                snapped = b[c - 1];
        }
        b[c] = std::max(snapped, b[c - 1]);
    }
    int64_t makespan_sk = 0;
    for (int c = 0; c < Gs; ++c) {
        int64_t cost = b[c + 1] - b[c];
        const size_t t_lo = (size_t)(std::upper_bound(start.begin(), start.end(), b[c]) - start.begin()) - 1;
        if (b[c + 1] > b[c] && t_lo < T && b[c] > start[t_lo])
            cost += 2;
        const size_t t_hi = (size_t)(std::upper_bound(start.begin(), start.end(), b[c + 1] - 1) - start.begin()) - 1;
        if (b[c + 1] > b[c] && t_hi < T && b[c + 1] < start[t_hi + 1])
            cost += 2;
        makespan_sk = std::max(makespan_sk, cost);
    }
    const bool use_sk = stream_k && T > 0 && makespan_sk < makespan_whole;

    const int G = use_sk ? Gs : Gw;
    std::vector<std::vector<WorkItem>> per(G);
    if (!use_sk) {
        for (size_t t = 0; t < T; ++t)
            per[owner[t]].push_back(make(tiles[t], 0, tiles[t].nk, -1, 0, 1, 0));
    } else {
        int c = 0;
        for (size_t t = 0; t < T; ++t) {
            const SwapTile &x = tiles[t];
            const int64_t s0 = start[t], s1 = start[t + 1];
            while (c < G && b[c + 1] <= s0)
                ++c;
            std::vector<std::pair<int, std::pair<int, int>>> segs;
            for (int cc = c; cc < G && b[cc] < s1; ++cc) {
                const int64_t lo = std::max(s0, b[cc]), hi = std::min(s1, b[cc + 1]);
                if (hi > lo)
                    segs.push_back({cc, {(int)((lo - s0) / x.ntok), (int)((hi - s0) / x.ntok)}});
            }
            const int nseg = (int)segs.size();
            const int split = nseg > 1 ? sc.splits : -1;
            if (nseg > 1)
                sc.splits += x.ntok;
            for (int j = 0; j < nseg; ++j) {
                const int slot = nseg > 1 ? sc.ws_slots : 0;
                if (nseg > 1)
                    sc.ws_slots += x.ntok;
                per[segs[j].first].push_back(make(x, segs[j].second.first, segs[j].second.second, split, j, nseg, slot));
            }
        }
    }
    // CTAs whose span came out empty (cuts moved to tile edges) are not launched
    per.erase(std::remove_if(per.begin(), per.end(), [](const std::vector<WorkItem> &l) { return l.empty(); }),
              per.end());
    if (per.empty())
        per.resize(1);
    sc.grid = (int)per.size();
    sc.list_begin.assign(sc.grid + 1, 0);
    for (int l = 0; l < sc.grid; ++l) {
        sc.list_begin[l] = (uint32_t)sc.items.size();
        sc.items.insert(sc.items.end(), per[l].begin(), per[l].end());
    }
    sc.list_begin[sc.grid] = (uint32_t)sc.items.size();
    return sc;
}

Schedule build_swap_schedule(const std::vector<ActiveGroup> &gs, int grid_cap, bool stream_k)
{
    std::vector<SwapTile> tiles;
    for (int gi = 0; gi < (int)gs.size(); ++gi) {
        const ActiveGroup &g = gs[gi];
        const int ntt = (g.M + kSwapTileRows - 1) / kSwapTileRows, tw = (g.N + kSwapTileRows - 1) / kSwapTileRows;
        const int nk = (g.K / 64 + 3) / 4;
        for (int w = 0; w < tw; ++w)
            for (int t0 = 0; t0 < ntt; t0 += 2)
                tiles.push_back(SwapTile{gi, w, t0, std::min(2, ntt - t0), nk});
    }
    return stream_k_schedule(tiles, grid_cap, stream_k,
                             [&](const SwapTile &t, int kb0, int kb1, int split, int seg, int nseg, int slot) {
                                 return make_swap_item(gs[t.group], t.group, t, kb0, kb1, split, seg, nseg, slot);
                             });
}

// The pair kernel's item: B rows 256w .. 256w + 255 (tile_n = w), A rows 256t .. (tile_m
// = t), the group's MMA width in the flags. The scale blocks of the first 128-row tiles
// of both; the second ones follow (kItemA2 / kItemB2 say whether they exist).
WorkItem make_swap_pair_item(const ActiveGroup &g, int gi, const SwapTile &t, int kb_begin, int kb_end, int split,
                             int seg, int nseg, int slot)
{
    WorkItem w{};
    w.group = gi;
    w.tile_m = t.t0;
    w.tile_n = t.w;
    w.kb_begin = kb_begin;
    w.kb_end = kb_end;
    w.split = split;
    w.seg = seg;
    w.nseg = nseg;
    w.ws_slot = slot;
    const int kb64 = g.K / 64;
    w.kblocks64 = kb64;
    const int nt = round16(std::min(g.M, kSwapPairRows));
    w.flags = (kSwapPairRows * t.w + 128 < g.N ? kItemA2 : 0) | (kSwapPairRows * t.t0 + 128 < g.M ? kItemB2 : 0) |
              (g.sf_rowmajor ? kItemSfRowMajor : 0) | ((nt / 16) << kSwapPairNtShift);
    w.a_row = kSwapPairRows * t.t0;
    const size_t blocks = (size_t)kb64 * kScaleBlockBytes;
    w.sfa = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(g.SFA) + (size_t)(2 * t.t0) * blocks);
    w.sfb = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(g.SFB) + (size_t)(2 * t.w) * blocks);
    return w;
}

Schedule build_swap_pair_schedule(const std::vector<ActiveGroup> &gs, int grid_cap, bool stream_k)
{
    std::vector<SwapTile> tiles;
    for (int gi = 0; gi < (int)gs.size(); ++gi) {
        const ActiveGroup &g = gs[gi];
        const int ntt = (g.M + kSwapPairRows - 1) / kSwapPairRows, tw = (g.N + kSwapPairRows - 1) / kSwapPairRows;
        const int nk = (g.K / 64 + 3) / 4;
        for (int w = 0; w < tw; ++w)
            for (int t = 0; t < ntt; ++t)
                tiles.push_back(SwapTile{gi, w, t, 1, nk});
    }
    return stream_k_schedule(tiles, grid_cap, stream_k,
                             [&](const SwapTile &t, int kb0, int kb1, int split, int seg, int nseg, int slot) {
                                 return make_swap_pair_item(gs[t.group], t.group, t, kb0, kb1, split, seg, nseg, slot);
                             });
}

// How one kernel variant tiles a problem set.
struct Plan {
    int variant;
    int block_m, block_n;
    int grid_cap;  // lists: CTAs, or CTA pairs
};

Plan plan_for(int variant, const DeviceState &ds, int64_t max_ctas)
{
    const bool pair = variant == kVariantPair || variant == kVariantSwapPair;
    Plan p;
    p.variant = variant;
    p.block_m = pair ? kPairBlockM : kBlockM;
    p.block_n = pair ? kPairBlockN : ((variant == 2 || variant == 3) ? 256 : 128);
    int cap = std::min(pair ? ds.pair_clusters : ds.sm_count, kMaxLists);
    if (max_ctas > 0)
        cap = (int)std::min<int64_t>(pair ? std::max<int64_t>(1, max_ctas / 2) : max_ctas, cap);
    p.grid_cap = cap;
    return p;
}

// Whether a variant's schedule cuts its last partial wave along K. On the pair
// kernel the fp32 partials of 256 x 256 tiles (their write, the reduction's
// reads) cost more than the balance gains: on the MoE-shaped set with K = 7168
// it measured 40.5 us split against 38.0 us whole. So pairs split only when
// asked to (split_mode 2). split_mode 3 asks for the small-grid fill on single CTAs.
int split_for(int variant, int split_mode)
{
    if (split_mode == 2)
        return kSplitTail;
    if (variant == kVariantPair)
        return kSplitNone;
    return split_mode == 1 ? kSplitTail : split_mode == 3 ? kSplitFill : kSplitNone;
}

// Estimated time of a schedule's busiest list, in microseconds: stage_us per
// K-stage, plus 1 us per item (the tile change: accumulator drain, epilogue,
// refilling the ring) and 1 us more per split segment (its fp32 partial).
double makespan_us(const Schedule &sc, double stage_us)
{
    double worst = 0;
    for (size_t l = 0; l + 1 < sc.list_begin.size(); ++l) {
        double t = 0;
        for (uint32_t i = sc.list_begin[l]; i < sc.list_begin[l + 1]; ++i)
            t += stage_us * (sc.items[i].kb_end - sc.items[i].kb_begin) + (sc.items[i].split >= 0 ? 2.0 : 1.0);
        worst = std::max(worst, t);
    }
    return worst;
}

// The automatic choice between CTA pairs and single CTAs with 128 x 128 tiles,
// from each schedule's busiest list. Measured on this GPU with every SM busy: a
// K-stage takes about 0.39 us on a single CTA (128 x 128 outputs) and 0.44 us on
// a CTA pair (256 x 256 outputs), and a pair reaches its first MMA about 1 us
// later. The MoE-shaped sets go to pairs (K = 7168: 38 us against 41.6 us; K =
// 2048: 25.4 against 31.9); the two-group sets, which leave SMs idle either way,
// stay on single CTAs (16.6 against about 18; 12.3 against about 14).
int choose_variant(const std::vector<ActiveGroup> &gs, const DeviceState &ds, int64_t max_ctas, int split_mode)
{
    // Every group with at most 32 rows of A (decode-sized MoE sets): the swapped-operand
    // kernel, whose MMA is only as wide as the rows there are. Measured on this GPU,
    // against the best of the others: M 1-8, N 7168, K 2048: 20.6 against 22.0 us;
    // M 4-32, N 4096, K 7168: 33.5 against 35.0; 32 groups of M 8, N 4096, K 7168: 104
    // against 109. With 48-96 rows per group the unswapped kernels are ahead again.
    int max_m = 0;
    for (const ActiveGroup &g : gs)
        max_m = std::max(max_m, g.M);
    if (max_m <= 32)
        return kVariantSwap;
    const Plan pp = plan_for(kVariantPair, ds, max_ctas), p1 = plan_for(0, ds, max_ctas);
    const double t_pair = 1.0 + makespan_us(build_schedule(gs, pp.block_m, pp.block_n, pp.grid_cap,
                                                           split_for(kVariantPair, split_mode)),
                                            0.44);
    const double t_single =
        makespan_us(build_schedule(gs, p1.block_m, p1.block_n, p1.grid_cap, split_for(0, split_mode)), 0.39);
    return t_pair < t_single ? kVariantPair : 0;
}

// M-fusion (page 2, `_merge_groups`). Active group i continues the run of group
// i - 1 when its A rows follow that group's in memory (the caller passed slices of
// one concatenated A) with the same K, and, where the kernel reads row-major scales,
// its SFA rows follow too. A run shares its first group's A (and SFA) tensor map,
// which spans the rows of the whole run; an item addresses its rows from the run's
// first row. A tile's rows past its group's M are then the next group's rows rather
// than TMA's zero fill: they reach only output rows that are never stored.
struct ARuns {
    std::vector<int> head;       // the run's first group
    std::vector<int32_t> row0;   // the group's first row in the run's map
    std::vector<int64_t> rows;   // at a run's first group: the rows of the run
    int maps = 0;
};

bool rows_follow(const void *prev, size_t bytes, const void *next)
{
    return reinterpret_cast<uintptr_t>(prev) + bytes == reinterpret_cast<uintptr_t>(next);
}

ARuns a_runs(const std::vector<ActiveGroup> &gs, bool fuse)
{
    ARuns r;
    const size_t n = gs.size();
    r.head.resize(n);
    r.row0.resize(n);
    r.rows.assign(n, 0);
    for (size_t i = 0; i < n; ++i) {
        const ActiveGroup &q = gs[i];
        bool join = fuse && i > 0;
        if (join) {
            const ActiveGroup &p = gs[i - 1];
            join = p.K == q.K && p.sf_rowmajor == q.sf_rowmajor && rows_follow(p.A, (size_t)p.M * (p.K / 2), q.A) &&
                   (!q.sf_rowmajor || rows_follow(p.SFA, (size_t)p.M * (p.K / 16), q.SFA)) &&
                   r.rows[r.head[i - 1]] + q.M <= INT32_MAX;  // TMA row coordinates are 32-bit
        }
        if (join) {
            r.head[i] = r.head[i - 1];
            r.row0[i] = r.row0[i - 1] + gs[i - 1].M;
        } else {
            r.head[i] = (int)i;
            r.row0[i] = 0;
            ++r.maps;
        }
        r.rows[r.head[i]] += q.M;
    }
    return r;
}

// Caller holds g_mu. variant_req is a kernel variant or kVariantAuto.
int get_table(int dev, const DeviceState &ds, const std::vector<ActiveGroup> &gs, int variant_req, int64_t max_ctas,
              int split_mode, int m_fusion, cudaStream_t stream, CachedTable **out)
{
    std::vector<uint8_t> sig(sizeof(int) * 5 + gs.size() * sizeof(ActiveGroup));
    int hdr[5] = {dev, variant_req, (int)std::min<int64_t>(max_ctas, 1 << 30), m_fusion, split_mode};
    memcpy(sig.data(), hdr, sizeof(hdr));
    if (!gs.empty())
        memcpy(sig.data() + sizeof(hdr), gs.data(), gs.size() * sizeof(ActiveGroup));
    const uint64_t key = fnv1a(sig.data(), sig.size());
    auto it = g_table_index.find(key);
    if (it != g_table_index.end() && it->second->signature == sig) {
        g_tables.splice(g_tables.begin(), g_tables, it->second);
        *out = &g_tables.front();
        return NVFP4_OK;
    }
    if (it != g_table_index.end() && !it->second->captured) {
        // a hash collision: the older table leaves the cache, the new one takes its key
        evict_table(it->second);
        it = g_table_index.end();
    }
    if (int rc = get_encoder())
        return rc;
    if (int rc = ensure_context(dev))
        return rc;

    // The pair kernel (variant kVariantPair) runs 256 x 256 tiles, one list per CTA pair.
    const int variant = variant_req == kVariantAuto ? choose_variant(gs, ds, max_ctas, split_mode) : variant_req;
    const Plan plan = plan_for(variant, ds, max_ctas);
    const bool swap_pair = variant == kVariantSwapPair;
    const bool pair = variant == kVariantPair || swap_pair;
    const bool swap = variant == kVariantSwap || swap_pair;
    const int block_m = plan.block_m, block_n = plan.block_n;
    const int halves = pair ? 2 : 1;  // workspace slots and counters per split segment / tile
    Schedule sc = swap_pair ? build_swap_pair_schedule(gs, plan.grid_cap, split_mode != 0)
                  : swap    ? build_swap_schedule(gs, plan.grid_cap, split_mode != 0)
                            : build_schedule(gs, block_m, block_n, plan.grid_cap, split_for(variant, split_mode));
    // M-fusion for the pair kernel only: the single-CTA kernel addressing A through
    // the item's row rather than its tile index measured ~1 us slower on the small
    // two-group sets it serves (which have no runs to fuse anyway). The swapped
    // kernel's item flags carry its MMA shapes instead of an A map.
    const ARuns runs = a_runs(gs, m_fusion != 0 && pair && !swap);
    if (!swap)
        for (WorkItem &w : sc.items) {
            w.a_row += runs.row0[w.group];
            w.flags = (w.flags & ((1 << kItemAMapShift) - 1)) | (runs.head[w.group] << kItemAMapShift);
        }
    const std::vector<WorkItem> &items = sc.items;
    const std::vector<uint32_t> &cta_begin = sc.list_begin;
    const int grid = sc.grid;  // lists: CTAs, or CTA pairs

    const size_t off_groups = sizeof(TableHeader);
    const size_t off_cta = off_groups + gs.size() * sizeof(GroupEntry);
    const size_t off_items = (off_cta + cta_begin.size() * sizeof(uint32_t) + 15) & ~size_t(15);
    const size_t total = off_items + items.size() * sizeof(WorkItem);

    CachedTable t;
    t.key = key;
    t.signature = std::move(sig);
    t.bytes = total;
    t.device = dev;
    t.grid = grid * halves;
    t.block_n = block_n;
    t.variant = variant;
    t.a_maps = runs.maps;
    t.list_begin = sc.list_begin;
    const size_t ws_bytes = sc.splits > 0 ? (size_t)sc.ws_slots * halves * kBlockM * block_n * sizeof(float) : 0;
    const size_t cnt_bytes = sc.splits > 0 ? (size_t)sc.splits * halves * sizeof(int) : 0;
    if (int rc = acquire_buffers(dev, total, ws_bytes, cnt_bytes, &t.buf))
        return rc;
    t.host = t.buf.host;
    t.dev = t.buf.dev;
    t.workspace = sc.splits > 0 ? t.buf.ws : nullptr;
    t.counters = sc.splits > 0 ? t.buf.cnt : nullptr;
    memset(t.host, 0, total);
    uint8_t *h = static_cast<uint8_t *>(t.host);
    TableHeader *th = reinterpret_cast<TableHeader *>(h);
    th->num_groups = (int32_t)gs.size();
    th->num_items = (int32_t)items.size();
    th->grid = grid;
    th->block_n = block_n;
    th->off_cta_begin = (uint32_t)off_cta;
    th->off_items = (uint32_t)off_items;
    th->total_bytes = (uint32_t)total;
    GroupEntry *ge = reinterpret_cast<GroupEntry *>(h + off_groups);
    for (size_t i = 0; i < gs.size(); ++i) {
        const ActiveGroup &a = gs[i];
        GroupEntry &e = ge[i];
        const int h = runs.head[i];
        const uint64_t run_rows = (uint64_t)runs.rows[h];
        // A run's later groups keep a copy of its map, so every group's maps stay
        // valid descriptors; the items read the first group's.
        int rc = 0;
        // the swapped kernels' A box: the group's rows (rounded up to 16) when they fit one
        // tile; on CTA pairs each CTA holds half of them
        const uint32_t a_box = swap_pair ? (uint32_t)(round16(std::min(a.M, kSwapPairRows)) / 2)
                               : swap    ? (uint32_t)(a.M <= kSwapTileRows ? round16(a.M) : kSwapTileRows)
                                         : (uint32_t)kBlockM;
        if (h == (int)i)
            rc = encode_operand_map(&e.tmap_a, a.A, (uint64_t)a.K / 2, run_rows, a_box);
        else
            e.tmap_a = ge[h].tmap_a;
        if (!rc)
            rc = encode_operand_map(&e.tmap_b, a.B, (uint64_t)a.K / 2, (uint64_t)a.N, pair ? 128u : (uint32_t)block_n);
        if (!rc)
            rc = swap ? encode_output_map_t(&e.tmap_c, a.C, (uint64_t)a.M, (uint64_t)a.N, (uint64_t)a.c_stride())
                      : encode_output_map(&e.tmap_c, a.C, (uint64_t)a.M, (uint64_t)a.N, (uint64_t)a.c_stride());
        if (!rc) {
            if (!a.sf_rowmajor)
                rc = encode_unused_scale_map(&e.tmap_sfa, a.SFA);
            else if (h == (int)i)
                rc = encode_scale_map(&e.tmap_sfa, a.SFA, (uint64_t)a.K / 16, run_rows,
                                      swap_pair ? (uint32_t)kSwapPairRows : (uint32_t)kBlockM);
            else
                e.tmap_sfa = ge[h].tmap_sfa;
        }
        if (!rc)
            rc = a.sf_rowmajor ? encode_scale_map(&e.tmap_sfb, a.SFB, (uint64_t)a.K / 16, (uint64_t)a.N,
                                                  swap ? 128u : pair ? (uint32_t)kPairBlockN : (uint32_t)block_n)
                               : encode_unused_scale_map(&e.tmap_sfb, a.SFB);
        if (rc) {
            return_buffers(std::move(t.buf), false);
            return rc;
        }
        e.sfa = static_cast<const uint8_t *>(a.SFA);
        e.sfb = static_cast<const uint8_t *>(a.SFB);
        e.C = static_cast<__half *>(a.C);
        e.M = a.M;
        e.N = a.N;
        e.K = a.K;
        e.kblocks64 = a.K / 64;
        e.tiles_m = (a.M + block_m - 1) / block_m;
        e.tiles_n = (a.N + block_n - 1) / block_n;
        e.sf_rowmajor = a.sf_rowmajor;
    }
    memcpy(h + off_cta, cta_begin.data(), cta_begin.size() * sizeof(uint32_t));
    if (!items.empty())
        memcpy(h + off_items, items.data(), items.size() * sizeof(WorkItem));

    cudaError_t e = cudaMemcpyAsync(t.dev, t.host, total, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && sc.splits > 0) {
        e = cudaMemsetAsync(t.counters, 0, cnt_bytes, stream);
        t.splits = sc.splits * halves;
    }
    if (e != cudaSuccess) {
        return_buffers(std::move(t.buf), true);
        return cuda_fail(e);
    }

    // The least recently used table leaves (tables a graph may replay stay); its
    // blocks retire once the work queued with them has completed.
    if (g_tables.size() >= kMaxCachedTables) {
        for (auto old = g_tables.end(); old != g_tables.begin();) {
            --old;
            if (!old->captured) {
                evict_table(old);
                break;
            }
        }
    }
    g_tables.push_front(std::move(t));
    if (it != g_table_index.end())
        g_table_index.erase(it);  // a collision with a captured table: the newer one takes the key
    g_table_index[key] = g_tables.begin();
    *out = &g_tables.front();
    // the upload reads the pinned copy: its blocks are in use from here on
    return note_use(g_tables.front(), stream);
}

// Each list's first item, copied from the host copy of the work items into the launch
// parameters (lists past the array's length read theirs from the table).
template <int N>
void fill_first_items(FirstItem (&first)[N], const WorkItem *items, const uint32_t *list_begin, int lists)
{
    for (int l = 0; l < std::min(lists, N); ++l)
        if (list_begin[l] < list_begin[l + 1])
            first[l] = first_item_of(items[list_begin[l]]);
}

template <int N>
void fill_first_items(FirstItem (&first)[N], const CachedTable &t)
{
    const TableHeader *th = static_cast<const TableHeader *>(t.host);
    const WorkItem *items = reinterpret_cast<const WorkItem *>(static_cast<const uint8_t *>(t.host) + th->off_items);
    fill_first_items(first, items, t.list_begin.data(), (int)t.list_begin.size() - 1);
}

// The A, B and C maps of the first kParamMapGroups groups, copied from the table's
// host copy into the launch parameters.
void fill_param_maps(KernelArgs &args, const void *host_table, int num_groups)
{
    const GroupEntry *ge = reinterpret_cast<const GroupEntry *>(static_cast<const uint8_t *>(host_table) +
                                                                sizeof(TableHeader));
    for (int g = 0; g < std::min(num_groups, kParamMapGroups); ++g) {
        args.pmaps[2 * g] = ge[g].tmap_a;
        args.pmaps[2 * g + 1] = ge[g].tmap_b;
        args.cmaps[g] = ge[g].tmap_c;
    }
}

// Sets the kernel's shared-memory limit once per device and checks that one CTA
// fits on an SM.
template <int BN, int STAGES>
int prepare_kernel(DeviceState &ds, int nslot)
{
    using L = Layout<BN, STAGES>;
    auto kern = nvfp4_grouped_gemm_kernel<BN, STAGES>;
    if (L::kSmemBytes > ds.max_smem_optin)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    if (!ds.attr_set[nslot]) {
        CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes));
        int n = 0;
        CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, L::kSmemBytes));
        if (n < 1)
            return NVFP4_ERR_UNSUPPORTED_DEVICE;
        ds.attr_set[nslot] = true;
    }
    return NVFP4_OK;
}

template <int BN, int STAGES>
int launch_gemm(DeviceState &ds, const CachedTable &t, cudaStream_t stream, int num_groups)
{
    using L = Layout<BN, STAGES>;
    SingleArgs args{};
    args.table = static_cast<const Table *>(t.dev);
    args.items = table_items(t);
    args.status = ds.status;
    args.timeout_ns = (uint64_t)std::max<int64_t>(1, g_opt.timeout_us.load()) * 1000ull;
    args.fault_skip_load = (int32_t)g_opt.fault_skip_load.load();
    args.num_groups = num_groups;
    args.prefetch_stages = (int32_t)(g_opt.prefetch_stages.load() < 0 ? kDefaultPrefetchStages
                                                                       : g_opt.prefetch_stages.load());
    args.workspace = t.workspace;
    args.counters = t.counters;
    fill_param_maps(args, t.host, num_groups);
    std::copy(t.list_begin.begin(), t.list_begin.end(), args.list_begin);
    fill_first_items(args.first, t);
    CUDA_TRY(launch_kernel(nvfp4_grouped_gemm_kernel<BN, STAGES>, (unsigned)t.grid, L::kSmemBytes, stream, args));
    static_assert(kDeepStages128 == 5 && kDeepStages256 == 3, "kernel names below");
    g_last_kernel.store(BN == 128 ? (STAGES == 2 ? "nvfp4_grouped_gemm_kernel<128,2>" : "nvfp4_grouped_gemm_kernel<128,5>")
                                  : (STAGES == 2 ? "nvfp4_grouped_gemm_kernel<256,2>" : "nvfp4_grouped_gemm_kernel<256,3>"));
    return NVFP4_OK;
}

// The pair kernel: shared-memory limit, and how many CTA pairs fit at once
// (clusters must sit inside one GPC, so this can be fewer than SMs / 2).
int prepare_pair_kernel(DeviceState &ds)
{
    using L = PairLayout<kPairStages>;
    auto kern = nvfp4_pair_gemm_kernel<kPairStages>;
    if (L::kSmemBytes > ds.max_smem_optin)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    if (!ds.attr_set[kVariantPair]) {
        CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes));
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (unsigned)std::max(1, ds.sm_count / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = L::kSmemBytes;
        int n = 0;
        CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
        if (n < 1)
            return NVFP4_ERR_UNSUPPORTED_DEVICE;
        ds.pair_clusters = n;
        ds.attr_set[kVariantPair] = true;
    }
    return NVFP4_OK;
}

int launch_pair(DeviceState &ds, const CachedTable &t, cudaStream_t stream, int num_groups)
{
    using L = PairLayout<kPairStages>;
    PairArgs args{};
    args.table = static_cast<const Table *>(t.dev);
    args.items = table_items(t);
    args.status = ds.status;
    args.timeout_ns = (uint64_t)std::max<int64_t>(1, g_opt.timeout_us.load()) * 1000ull;
    args.fault_skip_load = (int32_t)g_opt.fault_skip_load.load();
    args.num_groups = num_groups;
    args.prefetch_stages = 0;
    args.workspace = t.workspace;
    args.counters = t.counters;
    fill_param_maps(args, t.host, num_groups);
    std::copy(t.list_begin.begin(), t.list_begin.end(), args.list_begin);
    fill_first_items(args.first, t);
    CUDA_TRY(launch_kernel(nvfp4_pair_gemm_kernel<kPairStages>, (unsigned)t.grid, L::kSmemBytes, stream, args));
    g_last_kernel.store("nvfp4_pair_gemm_kernel<5>");
    return NVFP4_OK;
}

int prepare_swap_kernel(DeviceState &ds)
{
    using L = SwapLayout<kSwapStages>;
    auto kern = nvfp4_swapab_gemm_kernel<kSwapStages>;
    if (L::kSmemBytes > ds.max_smem_optin)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    if (!ds.attr_set[kVariantSwap]) {
        CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes));
        int n = 0;
        CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, L::kSmemBytes));
        if (n < 1)
            return NVFP4_ERR_UNSUPPORTED_DEVICE;
        ds.attr_set[kVariantSwap] = true;
    }
    return NVFP4_OK;
}

int launch_swap(DeviceState &ds, const CachedTable &t, cudaStream_t stream, int num_groups)
{
    using L = SwapLayout<kSwapStages>;
    KernelArgs args{};
    args.table = static_cast<const Table *>(t.dev);
    args.items = table_items(t);
    args.status = ds.status;
    args.timeout_ns = (uint64_t)std::max<int64_t>(1, g_opt.timeout_us.load()) * 1000ull;
    args.fault_skip_load = (int32_t)g_opt.fault_skip_load.load();
    args.num_groups = num_groups;
    args.prefetch_stages = 0;
    args.workspace = t.workspace;
    args.counters = t.counters;
    fill_param_maps(args, t.host, num_groups);
    std::copy(t.list_begin.begin(), t.list_begin.end(), args.list_begin);
    CUDA_TRY(launch_kernel(nvfp4_swapab_gemm_kernel<kSwapStages>, (unsigned)t.grid, L::kSmemBytes, stream, args));
    static_assert(kSwapStages == 5, "kernel name below");
    g_last_kernel.store("nvfp4_swapab_gemm_kernel<5>");
    return NVFP4_OK;
}

int prepare_swap_pair_kernel(DeviceState &ds)
{
    using L = SwapPairLayout<kSwapPairStages>;
    auto kern = nvfp4_swapab_pair_kernel<kSwapPairStages>;
    if (L::kSmemBytes > ds.max_smem_optin)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    if (!ds.attr_set[kVariantSwapPair]) {
        CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes));
        ds.attr_set[kVariantSwapPair] = true;
    }
    return NVFP4_OK;
}

int launch_swap_pair(DeviceState &ds, const CachedTable &t, cudaStream_t stream, int num_groups)
{
    using L = SwapPairLayout<kSwapPairStages>;
    PairArgs args{};
    args.table = static_cast<const Table *>(t.dev);
    args.items = table_items(t);
    args.status = ds.status;
    args.timeout_ns = (uint64_t)std::max<int64_t>(1, g_opt.timeout_us.load()) * 1000ull;
    args.fault_skip_load = (int32_t)g_opt.fault_skip_load.load();
    args.num_groups = num_groups;
    args.prefetch_stages = 0;
    args.workspace = t.workspace;
    args.counters = t.counters;
    fill_param_maps(args, t.host, num_groups);
    std::copy(t.list_begin.begin(), t.list_begin.end(), args.list_begin);
    fill_first_items(args.first, t);
    CUDA_TRY(launch_kernel(nvfp4_swapab_pair_kernel<kSwapPairStages>, (unsigned)t.grid, L::kSmemBytes, stream, args));
    static_assert(kSwapPairStages == 5, "kernel name below");
    g_last_kernel.store("nvfp4_swapab_pair_kernel<5>");
    return NVFP4_OK;
}

int workspace_for(int dev, cudaStream_t stream, size_t bytes, void **out)
{
    Workspace &w = g_workspaces[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (w.bytes < bytes) {
        const size_t want = std::max(bytes, w.bytes * 2);  // grow geometrically
        if (w.ptr) {
            CUDA_TRY(cudaStreamSynchronize(stream));
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
        }
        CUDA_TRY(cudaMalloc(&w.ptr, want));
        w.bytes = want;
    }
    *out = w.ptr;
    return NVFP4_OK;
}

}  // namespace

// =================================================================== C ABI ==

extern "C" int nvfp4_grouped_gemm(int g, const Nvfp4Problem *probs, nvfp4_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (g < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (g == 0)
        return NVFP4_OK;
    if (!probs)
        return NVFP4_ERR_INVALID_ARG;
    if (g >= kMaxGroups)
        return NVFP4_ERR_TOO_LARGE;
    for (int i = 0; i < g; ++i)
        if (int rc = check_problem(probs[i]))
            return rc;

    const int64_t opt_bn = g_opt.block_n.load(), opt_st = g_opt.stages.load();
    const int block_n = opt_bn == 0 ? kDefaultBlockN : (int)opt_bn;
    const bool shallow = opt_st == 2;

    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    DeviceState *ds = nullptr;
    if (int rc = device_state(dev, &ds))
        return rc;

    // K == 0: C is the empty sum.
    for (int i = 0; i < g; ++i) {
        const Nvfp4Problem &p = probs[i];
        if (p.M > 0 && p.N > 0 && p.K == 0)
            CUDA_TRY(clear_output(p, stream));
    }

    // Row-major scales are read directly by the kernel where their rows are whole
    // multiples of 16 bytes (K % 256 == 0); the others go through the prepack kernel
    // into this stream's workspace.
    std::vector<ActiveGroup> gs;
    std::vector<PrepackJob> jobs;
    size_t ws_bytes = 0;
    std::vector<std::pair<size_t, size_t>> ws_off;  // per active group: SFA, SFB offsets (or SIZE_MAX)
    for (int i = 0; i < g; ++i) {
        const Nvfp4Problem &p = probs[i];
        if (p.M == 0 || p.N == 0 || p.K == 0)
            continue;
        const bool direct = p.sf_layout == NVFP4_SF_ROWMAJOR && g_opt.sf_direct.load() != 0 && p.K % 256 == 0;
        gs.push_back(ActiveGroup{p.M, p.N, p.K, direct ? 1 : 0, p.A, p.B, p.SFA, p.SFB, p.C, p.ldc ? p.ldc : p.N});
        if (p.sf_layout == NVFP4_SF_ROWMAJOR && !direct) {
            const size_t oa = ws_bytes;
            ws_bytes += (blocked_scale_bytes(p.M, p.K / 16) + 255) & ~size_t(255);
            const size_t ob = ws_bytes;
            ws_bytes += (blocked_scale_bytes(p.N, p.K / 16) + 255) & ~size_t(255);
            ws_off.push_back({oa, ob});
        } else {
            ws_off.push_back({SIZE_MAX, SIZE_MAX});
        }
    }
    if (gs.empty())
        return NVFP4_OK;
    if (ws_bytes > 0) {
        void *ws = nullptr;
        if (int rc = workspace_for(dev, stream, ws_bytes, &ws))
            return rc;
        uint8_t *base = static_cast<uint8_t *>(ws);
        for (size_t i = 0; i < gs.size(); ++i) {
            if (ws_off[i].first == SIZE_MAX)
                continue;
            ActiveGroup &a = gs[i];
            jobs.push_back(PrepackJob{static_cast<const uint8_t *>(a.SFA), base + ws_off[i].first, a.M, a.K / 16, 0, 0, 0, 0});
            jobs.push_back(PrepackJob{static_cast<const uint8_t *>(a.SFB), base + ws_off[i].second, a.N, a.K / 16, 0, 0, 0, 0});
            a.SFA = base + ws_off[i].first;
            a.SFB = base + ws_off[i].second;
        }
        CUDA_TRY(launch_prepack(jobs.data(), (int)jobs.size(), stream));
    }
    const int prepack_launches = jobs.empty() ? 0 : 1;

    // BLOCK_N or STAGES select a single-CTA variant; CTA_PAIR forces either kind.
    const int64_t opt_pair = g_opt.cta_pair.load();
    const int single = (block_n == 256 ? 2 : 0) + (shallow ? 1 : 0);
    const int variant_req = opt_pair == 1 ? kVariantPair
                            : opt_pair == 3 ? kVariantSwap
                            : opt_pair == 4 ? kVariantSwapPair
                            : (opt_pair == 2 || opt_bn != 0 || shallow) ? single
                                                                        : kVariantAuto;
    if (variant_req == kVariantPair || variant_req == kVariantSwapPair || variant_req == kVariantAuto)
        if (int rc = prepare_pair_kernel(*ds))  // also learns how many CTA pairs fit at once
            return rc;
    CachedTable *t = nullptr;
    if (int rc2 = get_table(dev, *ds, gs, variant_req, g_opt.max_ctas.load(), (int)g_opt.split_tail.load(),
                            (int)g_opt.m_fusion.load(), stream, &t))
        return rc2;
    const int variant = t->variant;
    int rc = NVFP4_OK;
    switch (variant) {
    case 0: rc = prepare_kernel<128, kDeepStages128>(*ds, 0); break;
    case 1: rc = prepare_kernel<128, 2>(*ds, 1); break;
    case 2: rc = prepare_kernel<256, kDeepStages256>(*ds, 2); break;
    case 3: rc = prepare_kernel<256, 2>(*ds, 3); break;
    case kVariantSwap: rc = prepare_swap_kernel(*ds); break;
    case kVariantSwapPair: rc = prepare_swap_pair_kernel(*ds); break;
    default: rc = prepare_pair_kernel(*ds); break;
    }
    if (rc)
        return rc;
    switch (variant) {
    case 0: rc = launch_gemm<128, kDeepStages128>(*ds, *t, stream, (int)gs.size()); break;
    case 1: rc = launch_gemm<128, 2>(*ds, *t, stream, (int)gs.size()); break;
    case 2: rc = launch_gemm<256, kDeepStages256>(*ds, *t, stream, (int)gs.size()); break;
    case 3: rc = launch_gemm<256, 2>(*ds, *t, stream, (int)gs.size()); break;
    case kVariantSwap: rc = launch_swap(*ds, *t, stream, (int)gs.size()); break;
    case kVariantSwapPair: rc = launch_swap_pair(*ds, *t, stream, (int)gs.size()); break;
    default: rc = launch_pair(*ds, *t, stream, (int)gs.size()); break;
    }
    if (rc == NVFP4_OK) {
        g_last_launches.store(prepack_launches + 1);
        g_last_a_maps.store(t->a_maps);
        rc = note_use(*t, stream);
    }
    return rc;
}

extern "C" size_t nvfp4_prepacked_scale_bytes(int rows, int K)
{
    if (rows <= 0 || K <= 0)
        return 0;
    return (size_t)((rows + 127) / 128) * 128 * (size_t)((K + 63) / 64) * 4;
}

extern "C" int nvfp4_prepack_scales(const void *sf_rowmajor, int rows, int K, void *sf_blocked, nvfp4_stream_t stream)
{
    if (rows < 0 || K < 0 || K % 16 != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (rows >= kMaxDim || K >= kMaxDim)
        return NVFP4_ERR_TOO_LARGE;
    if (rows == 0 || K == 0)
        return NVFP4_OK;
    if (!sf_rowmajor || !sf_blocked)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(sf_rowmajor) || !aligned16(sf_blocked))
        return NVFP4_ERR_ALIGNMENT;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int dev = 0;
        CUDA_TRY(cudaGetDevice(&dev));
        DeviceState *ds = nullptr;
        if (int rc = device_state(dev, &ds))
            return rc;
    }
    PrepackJob j{static_cast<const uint8_t *>(sf_rowmajor), static_cast<uint8_t *>(sf_blocked), rows, K / 16, 0, 0, 0, 0};
    CUDA_TRY(launch_prepack(&j, 1, reinterpret_cast<cudaStream_t>(stream)));
    return NVFP4_OK;
}

extern "C" int nvfp4_prepack_scales_batch(int n, const void *const *sf_rowmajor, const int *rows, const int *K,
                                          void *const *sf_blocked, nvfp4_stream_t stream)
{
    if (n < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (n == 0)
        return NVFP4_OK;
    if (!sf_rowmajor || !rows || !K || !sf_blocked)
        return NVFP4_ERR_INVALID_ARG;
    std::vector<PrepackJob> jobs;
    jobs.reserve(n);
    for (int i = 0; i < n; ++i) {
        if (rows[i] < 0 || K[i] < 0 || K[i] % 16 != 0)
            return NVFP4_ERR_INVALID_ARG;
        if (rows[i] >= kMaxDim || K[i] >= kMaxDim)
            return NVFP4_ERR_TOO_LARGE;
        if (rows[i] == 0 || K[i] == 0)
            continue;
        if (!sf_rowmajor[i] || !sf_blocked[i])
            return NVFP4_ERR_INVALID_ARG;
        if (!aligned16(sf_rowmajor[i]) || !aligned16(sf_blocked[i]))
            return NVFP4_ERR_ALIGNMENT;
        jobs.push_back(PrepackJob{static_cast<const uint8_t *>(sf_rowmajor[i]), static_cast<uint8_t *>(sf_blocked[i]),
                                  rows[i], K[i] / 16, 0, 0, 0, 0});
    }
    if (jobs.empty())
        return NVFP4_OK;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int dev = 0;
        CUDA_TRY(cudaGetDevice(&dev));
        DeviceState *ds = nullptr;
        if (int rc = device_state(dev, &ds))
            return rc;
    }
    CUDA_TRY(launch_prepack(jobs.data(), (int)jobs.size(), reinterpret_cast<cudaStream_t>(stream)));
    return NVFP4_OK;
}

extern "C" int nvfp4_device_status(nvfp4_stream_t stream, int *status, int32_t *detail)
{
    if (!status)
        return NVFP4_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    DeviceState *ds = nullptr;
    if (int rc = device_state(dev, &ds))
        return rc;
    CUDA_TRY(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    int words[4] = {0, 0, 0, 0};
    CUDA_TRY(cudaMemcpy(words, ds->status, sizeof(words), cudaMemcpyDeviceToHost));
    if (words[0] != 0) {
        CUDA_TRY(cudaMemset(ds->status, 0, sizeof(words)));
        // A launch that gave up may have left split-tile counters part-way.
        for (const CachedTable &t : g_tables)
            if (t.device == dev && t.counters)
                CUDA_TRY(cudaMemset(t.counters, 0, (size_t)t.splits * sizeof(int)));
    }
    *status = words[0];
    if (detail)
        for (int i = 0; i < 4; ++i)
            detail[i] = words[i];
    return NVFP4_OK;
}

extern "C" const char *nvfp4_status_string(int code)
{
    switch (code) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_ALIGNMENT: return "misaligned pointer or size (16-byte pointers, K % 64 == 0, N % 8 == 0)";
    case NVFP4_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3, sm_103a)";
    case NVFP4_ERR_CUDA: return "CUDA error (see nvfp4_last_cuda_error)";
    case NVFP4_ERR_TIMEOUT: return "a kernel wait timed out";
    case NVFP4_ERR_TOO_LARGE: return "size beyond the library's limits";
    case NVFP4_ERR_CAPTURE: return "not allowed while the stream is being captured";
    default: return "unknown status";
    }
}

extern "C" int nvfp4_last_cuda_error(void) { return g_last_cuda_error.load(); }

extern "C" const char *nvfp4_last_kernel(void) { return g_last_kernel.load(); }

extern "C" int nvfp4_last_launches(void) { return g_last_launches.load(); }

extern "C" int nvfp4_last_a_maps(void) { return g_last_a_maps.load(); }

extern "C" int nvfp4_set_option(int option, int64_t value)
{
    switch (option) {
    case NVFP4_OPT_BLOCK_N:
        if (value != 0 && value != 128 && value != 256)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.block_n = value;
        return NVFP4_OK;
    case NVFP4_OPT_STAGES:
        if (value != 0 && value != 2)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.stages = value;
        return NVFP4_OK;
    case NVFP4_OPT_MAX_CTAS:
        if (value < 0)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.max_ctas = value;
        return NVFP4_OK;
    case NVFP4_OPT_WAIT_TIMEOUT_US:
        if (value < 1 || value > 60000000)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.timeout_us = value;
        return NVFP4_OK;
    case NVFP4_OPT_SPLIT_TAIL:
        if (value < 0 || value > 3)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.split_tail = value;
        return NVFP4_OK;
    case NVFP4_OPT_PDL:
        if (value < 0 || value > 1)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.pdl = value;
        return NVFP4_OK;
    case NVFP4_OPT_M_FUSION:
        if (value < 0 || value > 1)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.m_fusion = value;
        return NVFP4_OK;
    case NVFP4_OPT_SF_DIRECT:
        if (value < 0 || value > 1)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.sf_direct = value;
        return NVFP4_OK;
    case NVFP4_OPT_CTA_PAIR:
        if (value < 0 || value > 4)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.cta_pair = value;
        return NVFP4_OK;
    case NVFP4_OPT_PREFETCH_STAGES:
        if (value < -1 || value > 64)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.prefetch_stages = value;
        return NVFP4_OK;
    case NVFP4_OPT_FAULT_SKIP_LOAD:
        if (value < -1)
            return NVFP4_ERR_INVALID_ARG;
        g_opt.fault_skip_load = value;
        return NVFP4_OK;
    default:
        return NVFP4_ERR_INVALID_ARG;
    }
}

extern "C" void nvfp4_release(void)
{
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess)
        cur = -1;
    for (int d = 0; d < kMaxDevices; ++d) {
        if (!g_dev[d].ready)
            continue;
        cudaSetDevice(d);
        cudaDeviceSynchronize();
        for (auto it = g_tables.begin(); it != g_tables.end();) {
            if (it->device == d) {
                auto idx = g_table_index.find(it->key);
                if (idx != g_table_index.end() && idx->second == it)
                    g_table_index.erase(idx);
                free_buffers(it->buf);
                it = g_tables.erase(it);
            } else {
                ++it;
            }
        }
        for (std::vector<Buffers> *pool : {&g_free_buffers, &g_retiring_buffers})
            for (auto it = pool->begin(); it != pool->end();) {
                if (it->device == d) {
                    free_buffers(*it);
                    it = pool->erase(it);
                } else {
                    ++it;
                }
            }
        for (auto it = g_workspaces.begin(); it != g_workspaces.end();) {
            if (it->first.first == d) {
                cudaFree(it->second.ptr);
                it = g_workspaces.erase(it);
            } else {
                ++it;
            }
        }
        if (g_dev[d].status)
            cudaFree(g_dev[d].status);
        g_dev[d] = DeviceState{};
    }
    if (cur >= 0)
        cudaSetDevice(cur);
}

// ======================================================= no-allocation entry ==
//
// nvfp4_grouped_gemm_noalloc: the same grouped GEMM kernel for callers that
// cannot allocate device memory. Examples: code running inside a custom
// allocator or an out-of-memory handler, or a runtime that owns every byte of
// device memory and forbids cudaMalloc/cudaFree from libraries. The caller
// still passes A, B, SFA, SFB and C. The kernel's only other device memory (its
// problem table and its error words) lives in the fixed array below, which is
// part of the loaded module. Every GPU that loads this library holds this
// array until the process exits.
//
// Limits and rules (repeated in the header):
//  * Scratch size kNoAllocScratchBytes (256 KB). The first 256 bytes hold the
//    error words and the rest holds the table:
//    128 + sizeof(GroupEntry) * g + 4 * (grid + 1) (rounded up to 16) + 64 * tiles,
//    where tiles = sum over groups of ceil(M/128) * ceil(N/128). A larger
//    problem set returns NVFP4_ERR_TOO_LARGE and launches nothing.
//  * Row-major scales only where K % 256 == 0, read directly by the kernel: the
//    prepack pass would need a workspace.
//  * All calls share the one array. A call overwrites the previous call's table
//    in stream order. Calls that can overlap on the GPU (on different streams,
//    without ordering between them) race on it and must not be issued.
//  * The first call on a device does the set-up: the device checks, the
//    cudaGetSymbolAddress lookup of the array and the kernel's shared-memory
//    attribute.
//  * A call on a stream that is being captured returns NVFP4_ERR_CAPTURE and
//    queues nothing: the table copy would become a graph node that reads the
//    static host buffer when the graph is replayed, by then another call's table.
//  * The kernel's error words (the first 16 bytes of the array) are sticky: a
//    wait that runs out records NVFP4_ERR_TIMEOUT there and ends the launch
//    early. nvfp4_noalloc_status reads and clears them without allocating.

namespace {

constexpr size_t kNoAllocScratchBytes = 256 * 1024;
constexpr size_t kNoAllocStatusBytes = 256;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    uint8_t *scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
std::mutex g_noalloc_mu;  // guards the per-device set-up and the host staging buffer
NoAllocDevice g_noalloc_dev[kMaxDevices];
alignas(128) uint8_t g_noalloc_host[kNoAllocScratchBytes];  // host staging copy of the table

// Once per device, with that device current. The caller holds g_noalloc_mu.
int noalloc_setup(int dev, NoAllocDevice **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, smem = 0;
        CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
        CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
        CUDA_TRY(cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev));
        CUDA_TRY(cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        d.supported = (major == 10 && minor == 3) && smem >= Layout<kDefaultBlockN, kDefaultStages>::kSmemBytes;
        if (d.supported) {
            void *p = nullptr;
            CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
            d.scratch = static_cast<uint8_t *>(p);
            CUDA_TRY(cudaFuncSetAttribute(nvfp4_grouped_gemm_kernel<kDefaultBlockN, kDefaultStages>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<kDefaultBlockN, kDefaultStages>::kSmemBytes));

        }
        d.ready = true;
    }
    if (!d.supported)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return NVFP4_OK;
}

}  // namespace

extern "C" int nvfp4_grouped_gemm_noalloc(int g, const Nvfp4Problem *probs, nvfp4_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (g < 0)
        return NVFP4_ERR_INVALID_ARG;
    {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        CUDA_TRY(cudaStreamIsCapturing(stream, &cs));
        if (cs != cudaStreamCaptureStatusNone)
            return NVFP4_ERR_CAPTURE;
    }
    if (g == 0)
        return NVFP4_OK;
    if (!probs)
        return NVFP4_ERR_INVALID_ARG;
    if (g >= kMaxGroups)
        return NVFP4_ERR_TOO_LARGE;
    for (int i = 0; i < g; ++i) {
        if (int rc = check_problem(probs[i]))
            return rc;
        // row-major scales only where the kernel reads them directly (no workspace here)
        const Nvfp4Problem &p = probs[i];
        if (p.sf_layout == NVFP4_SF_ROWMAJOR && p.M > 0 && p.N > 0 && p.K > 0 && p.K % 256 != 0)
            return NVFP4_ERR_INVALID_ARG;
    }

    // Size the table before touching anything.
    constexpr int BN = kDefaultBlockN;
    size_t ngroups = 0, ntiles = 0;
    for (int i = 0; i < g; ++i) {
        const Nvfp4Problem &p = probs[i];
        if (p.M == 0 || p.N == 0 || p.K == 0)
            continue;
        ++ngroups;
        ntiles += (size_t)((p.M + kBlockM - 1) / kBlockM) * (size_t)((p.N + BN - 1) / BN);
    }

    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    NoAllocDevice *nd = nullptr;
    if (int rc = noalloc_setup(dev, &nd))
        return rc;
    const int cap = g_opt.max_ctas.load() > 0 ? (int)std::min<int64_t>(g_opt.max_ctas.load(), nd->sm_count)
                                              : nd->sm_count;
    const int grid = (int)std::max<size_t>(1, std::min<size_t>(ntiles, (size_t)std::min(cap, kMaxLists)));
    const size_t off_groups = sizeof(TableHeader);
    const size_t off_cta = off_groups + ngroups * sizeof(GroupEntry);
    const int lists = grid * kPipes;
    const size_t off_items = (off_cta + (size_t)(lists + 1) * sizeof(uint32_t) + 15) & ~size_t(15);
    const size_t total = off_items + ntiles * sizeof(WorkItem);
    if (total > kNoAllocScratchBytes - kNoAllocStatusBytes)
        return NVFP4_ERR_TOO_LARGE;

    // K == 0: C is the empty sum.
    for (int i = 0; i < g; ++i) {
        const Nvfp4Problem &p = probs[i];
        if (p.M > 0 && p.N > 0 && p.K == 0)
            CUDA_TRY(clear_output(p, stream));
    }
    if (ngroups == 0)
        return NVFP4_OK;
    if (int rc = get_encoder())
        return rc;
    if (int rc = ensure_context(dev))
        return rc;

    // Build the table in the static host buffer, with the same tile order and
    // CTA assignment as the cached path: group by group, tile_n outer and
    // tile_m inner, tile t to CTA t % grid.
    uint8_t *h = g_noalloc_host;
    memset(h, 0, total);
    TableHeader *th = reinterpret_cast<TableHeader *>(h);
    th->num_groups = (int32_t)ngroups;
    th->num_items = (int32_t)ntiles;
    th->grid = grid;
    th->block_n = BN;
    th->off_cta_begin = (uint32_t)off_cta;
    th->off_items = (uint32_t)off_items;
    th->total_bytes = (uint32_t)total;
    GroupEntry *ge = reinterpret_cast<GroupEntry *>(h + off_groups);
    uint32_t *cta_begin = reinterpret_cast<uint32_t *>(h + off_cta);
    WorkItem *items = reinterpret_cast<WorkItem *>(h + off_items);
    // Tile t goes to list l = (t % grid) * kPipes + (t / grid) % kPipes (the cached
    // path's rule). List l = c * kPipes + p holds t = c + grid * (kPipes * j + p) for
    // j = 0, 1, ..., so tile t sits at position t / (kPipes * grid) of its list.
    uint32_t run = 0;
    for (int l = 0; l < lists; ++l) {
        const size_t first = (size_t)(l / kPipes) + (size_t)grid * (l % kPipes);
        cta_begin[l] = run;
        run += (ntiles > first) ? (uint32_t)((ntiles - first + (size_t)kPipes * grid - 1) / ((size_t)kPipes * grid)) : 0u;
    }
    cta_begin[lists] = run;
    int gi = 0;
    size_t t = 0;
    for (int i = 0; i < g; ++i) {
        const Nvfp4Problem &p = probs[i];
        if (p.M == 0 || p.N == 0 || p.K == 0)
            continue;
        GroupEntry &e = ge[gi];
        int rc = encode_operand_map(&e.tmap_a, p.A, (uint64_t)p.K / 2, (uint64_t)p.M, kBlockM);
        if (!rc)
            rc = encode_operand_map(&e.tmap_b, p.B, (uint64_t)p.K / 2, (uint64_t)p.N, (uint32_t)BN);
        if (!rc)
            rc = encode_output_map(&e.tmap_c, p.C, (uint64_t)p.M, (uint64_t)p.N, (uint64_t)(p.ldc ? p.ldc : p.N));
        const bool rm = p.sf_layout == NVFP4_SF_ROWMAJOR;
        if (!rc)
            rc = rm ? encode_scale_map(&e.tmap_sfa, p.SFA, (uint64_t)p.K / 16, (uint64_t)p.M, kBlockM)
                    : encode_unused_scale_map(&e.tmap_sfa, p.SFA);
        if (!rc)
            rc = rm ? encode_scale_map(&e.tmap_sfb, p.SFB, (uint64_t)p.K / 16, (uint64_t)p.N, (uint32_t)BN)
                    : encode_unused_scale_map(&e.tmap_sfb, p.SFB);
        if (rc)
            return rc;
        e.sfa = static_cast<const uint8_t *>(p.SFA);
        e.sfb = static_cast<const uint8_t *>(p.SFB);
        e.C = static_cast<__half *>(p.C);
        e.M = p.M;
        e.N = p.N;
        e.K = p.K;
        e.kblocks64 = p.K / 64;
        e.tiles_m = (p.M + kBlockM - 1) / kBlockM;
        e.tiles_n = (p.N + BN - 1) / BN;
        e.sf_rowmajor = rm ? 1 : 0;
        const ActiveGroup a{p.M, p.N, p.K, rm ? 1 : 0, p.A, p.B, p.SFA, p.SFB, p.C, p.ldc ? p.ldc : p.N};
        for (int n = 0; n < e.tiles_n; ++n)
            for (int m = 0; m < e.tiles_m; ++m, ++t)
                items[cta_begin[list_of_tile(t, grid)] + t / ((size_t)kPipes * grid)] =
                    make_item(a, gi, m, n, 0, (p.K / 64 + 3) / 4, -1, 0, 1, 0, kBlockM, BN);
        ++gi;
    }

    uint8_t *dscratch = nd->scratch;
    int *dstatus = reinterpret_cast<int *>(dscratch);  // sticky: cleared by nvfp4_noalloc_status
    const Table *dtable = reinterpret_cast<const Table *>(dscratch + kNoAllocStatusBytes);
    // From pageable memory: returns once the bytes are staged, so the host
    // buffer may be reused by the next call.
    CUDA_TRY(cudaMemcpyAsync(dscratch + kNoAllocStatusBytes, h, total, cudaMemcpyHostToDevice, stream));

    SingleArgs args{};
    args.table = dtable;
    args.items = reinterpret_cast<const int4 *>(reinterpret_cast<const uint8_t *>(dtable) + off_items);
    args.status = dstatus;
    args.timeout_ns = (uint64_t)std::max<int64_t>(1, g_opt.timeout_us.load()) * 1000ull;
    args.fault_skip_load = (int32_t)g_opt.fault_skip_load.load();
    args.num_groups = (int32_t)ngroups;
    args.prefetch_stages = kDefaultPrefetchStages;
    args.workspace = nullptr;  // no split tiles here
    args.counters = nullptr;
    std::copy(cta_begin, cta_begin + lists + 1, args.list_begin);
    fill_param_maps(args, h, (int)ngroups);
    fill_first_items(args.first, items, cta_begin, (int)lists);
    CUDA_TRY(launch_kernel(nvfp4_grouped_gemm_kernel<kDefaultBlockN, kDefaultStages>, (unsigned)grid,
                           Layout<kDefaultBlockN, kDefaultStages>::kSmemBytes, stream, args));
    g_last_kernel.store("nvfp4_grouped_gemm_kernel<128,5>");
    g_last_launches.store(1);
    g_last_a_maps.store(ngroups);  // no M-fusion here: one A map per group
    return NVFP4_OK;
}

extern "C" int nvfp4_noalloc_status(nvfp4_stream_t stream, int *status, int32_t *detail)
{
    if (!status)
        return NVFP4_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    NoAllocDevice *nd = nullptr;
    if (int rc = noalloc_setup(dev, &nd))
        return rc;
    CUDA_TRY(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    int32_t words[4] = {0, 0, 0, 0};
    // Reads and writes the array through its symbol: no device allocation.
    CUDA_TRY(cudaMemcpyFromSymbol(words, g_noalloc_scratch, sizeof(words), 0, cudaMemcpyDeviceToHost));
    if (words[0] != 0) {
        const int32_t zero[4] = {0, 0, 0, 0};
        CUDA_TRY(cudaMemcpyToSymbol(g_noalloc_scratch, zero, sizeof(zero), 0, cudaMemcpyHostToDevice));
    }
    *status = words[0];
    if (detail)
        for (int i = 0; i < 4; ++i)
            detail[i] = words[i];
    return NVFP4_OK;
}
