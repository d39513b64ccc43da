// Host side of the C ABI declared in include/lora.h: argument validation,
// workspace carving, TMA tensor-map encoding and kernel dispatch.  Nothing
// here allocates device memory, synchronises or copies device->host except
// lora_get_status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "moe_pair.h"
#include "lora.h"

namespace lora {

// ---------------------------------------------------------------------------
// device queries and the tensor-map encoder (driver entry point, no -lcuda)
// ---------------------------------------------------------------------------
int num_sms_current_device()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 64 && cache[dev]) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    if (dev < 64) cache[dev] = n;
    return n;
}

static bool device_supported()
{
    static int cache[64] = {0};   // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (dev < 64 && cache[dev]) return cache[dev] == 1;
    int major = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    int minor = 0;
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    const bool ok = (major == 10 && minor == 3);
    if (dev < 64) cache[dev] = ok ? 1 : 2;
    return ok;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encoder()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 map: `inner` elements per row, `rows` rows, row pitch in bytes.
static bool encode_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t pitch,
                      uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw,
                      CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
{
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows < 1 ? 1 : rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map: dims {d0, d1, d2}, byte strides of dims 1 and 2.
static bool encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                      uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw,
                      CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
{
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1 < 1 ? 1 : d1, d2 < 1 ? 1 : d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

static int split_tpad(int64_t M) { return static_cast<int>(((M + 15) / 16) * 16); }

WsLayout make_ws_layout(int64_t M, int32_t N, int32_t A)
{
    WsLayout L;
    std::memset(&L, 0, sizeof L);
    L.M = M;
    L.N = N;
    L.A = A;
    L.num_mtiles = static_cast<int32_t>((M + kBM - 1) / kBM);
    constexpr int kMaxPanels = LORA_MAX_RANK / kChunk;   // rank panels of one adapter
    L.max_chunks = kMaxPanels * (A + L.num_mtiles) + kMaxPanels;
    L.max_sjobs = L.num_mtiles + L.max_chunks / kMaxShrinkChunks + 1;
    const int64_t present = std::min<int64_t>(A, M);
    L.max_dchunks = static_cast<int32_t>(kMaxPanels * present + kMaxPanels);
    const int NT = (N + kSplitBN - 1) / kSplitBN;
    const int RTmax = (L.max_dchunks + 7) / 8;
    L.split_tiles = NT + std::max<int>(RTmax, static_cast<int>(2 * present + 2));
    size_t split_s = 0;
    if (M <= kSplitMaxTokens) {
        const int T = split_tpad(M);
        L.acc_out_bytes = static_cast<size_t>(NT) * kSplitBN * T * 4;
        L.acc_shr_bytes = std::max<size_t>(static_cast<size_t>(RTmax) * kSplitBN,
                                           static_cast<size_t>(2 * present + 2) * 32) * T * 4;
        split_s = static_cast<size_t>(L.max_dchunks) * T * kChunk * 2;
    }
    // per (layer, token tile): the tiled schedule's S-ready and consumer
    // counters, for up to kMaxLayers layers of one launch; per split-K
    // tile: its arrival counter.  Sized for N >= 65536 so that
    // the regions after it (the segment table) sit at offsets that depend
    // on M and A only: one table then serves layers of any K and N.
    const int NT_cnt = (std::max<int32_t>(N, 65536) + kSplitBN - 1) / kSplitBN;
    const size_t split_cnt = static_cast<size_t>(NT_cnt) + std::max<int>(RTmax, static_cast<int>(2 * present + 2));
    L.n_counters = CNT_FIXED + std::max<size_t>(2 * static_cast<size_t>(kMaxLayers) * L.num_mtiles, split_cnt) + 8;
    // tiled schedule: S panels, one set per K piece of a shrink job (two for M > 128)
    const size_t tiled_s = static_cast<size_t>(L.max_chunks) * kBM * kChunk * 2 * tiled_s_sets(M);
    L.s_scratch_bytes = std::max(tiled_s, split_s);

    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    L.counters = take(L.n_counters * 4);
    L.perm = take(static_cast<size_t>(std::max<int64_t>(M, 1)) * 4);
    L.offsets = take(static_cast<size_t>(A + 2) * 4);
    L.seg_id = take(static_cast<size_t>(std::max(A, 1)) * 4);
    L.seg_start = take(static_cast<size_t>(std::max(A, 1)) * 4);
    L.seg_len = take(static_cast<size_t>(std::max(A, 1)) * 4);
    L.seg_rank = take(static_cast<size_t>(std::max(A, 1)) * 4);
    L.num_segments = take(4);
    L.hdr = take(HDR_WORDS * 4);
    L.tile_chunk_off = take((static_cast<size_t>(L.num_mtiles) * LORA_MAX_SLICES + 1) * 4);
    L.chunk_arow = take(static_cast<size_t>(L.max_chunks) * 4);
    L.chunk_bpanel = take(static_cast<size_t>(L.max_chunks) * 4);
    L.chunk_rng = take(static_cast<size_t>(L.max_chunks) * 4);
    L.sjob_tile = take(static_cast<size_t>(L.max_sjobs) * 4);
    L.sjob_c0 = take(static_cast<size_t>(L.max_sjobs) * 4);
    L.sjob_c1 = take(static_cast<size_t>(L.max_sjobs) * 4);
    L.tile_njobs = take(static_cast<size_t>(L.num_mtiles) * 4);
    L.dchunk_arow = take(static_cast<size_t>(L.max_dchunks) * 4);
    L.dchunk_bpanel = take(static_cast<size_t>(L.max_dchunks) * 4);
    L.dchunk_adapter = take(static_cast<size_t>(L.max_dchunks) * 4);
    // stream schedule: windows of 8 pool panels.  An adapter's <= 8 panels
    // span at most 2 windows, so a batch touches <= 2 * min(A, M) of them.
    L.max_win_str = M <= kStreamMaxTokens
                        ? static_cast<int32_t>(std::min<int64_t>((kMaxPanels * A + 7) / 8, 2 * present)) : 0;
    L.wcnt = take(static_cast<size_t>(std::max(L.max_win_str, 1)) * kWinCntStride * 4);
    L.acc_str_bytes = M <= kStreamMaxTokens
                          ? static_cast<size_t>(std::max(L.max_win_str, 1)) * split_tpad(M) * kSplitBN * 4 : 16;
    L.acc_str = take(L.acc_str_bytes);
    o = (o + 1023) & ~size_t(1023);
    L.s_scratch = take(L.s_scratch_bytes);
    L.acc_out = take(std::max<size_t>(L.acc_out_bytes, 16));
    L.acc_shr = take(std::max<size_t>(L.acc_shr_bytes, 16));
    L.fac = take(static_cast<size_t>(kMaxLayers) * std::max(A, 1) * 4);
    L.total_min = o;
    // stream-K scratch of the tiled schedule: partial sums and counters of
    // the split tiles (used only when the workspace is this large)
    if (M > kSplitMaxTokens) {
        L.sk_part = take(static_cast<size_t>(kStreamKMaxTiles) * kBM * kBN * 4);
        L.sk_cnt = take(static_cast<size_t>(kStreamKMaxTiles) * kWinCntStride * 4);
    }
    L.total = o;
    return L;
}

template <typename T>
static T *at(void *ws, size_t off)
{
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_pool(const lora_pool_t *pool)
{
    if (!pool) return LORA_ERR_NULL;
    if (pool->K <= 0 || pool->N <= 0 || (pool->K % 8) || (pool->N % 8)) return LORA_ERR_SHAPE;
    if (pool->num_adapters < 0 || pool->num_adapters > LORA_MAX_ADAPTERS) return LORA_ERR_SHAPE;
    if (pool->num_slices < 0 || pool->num_slices > LORA_MAX_SLICES) return LORA_ERR_SHAPE;
    const int S = pool->num_slices;
    if (S > 1) {
        // a merged output: ordered slices covering [0, N), inner boundaries
        // on output-tile edges
        if (pool->slice_start[0] != 0 || pool->slice_start[S] != pool->N) return LORA_ERR_SHAPE;
        for (int s = 1; s <= S; ++s)
            if (pool->slice_start[s] <= pool->slice_start[s - 1] || (s < S && pool->slice_start[s] % LORA_SLICE_ALIGN))
                return LORA_ERR_SHAPE;
    }
    if (pool->num_adapters > 0) {
        if (!pool->a_pool || !pool->b_pool || !pool->a_offset || !pool->b_offset || !pool->rank) return LORA_ERR_NULL;
        if (!aligned16(pool->a_pool) || !aligned16(pool->b_pool)) return LORA_ERR_ALIGN;
        if (reinterpret_cast<uintptr_t>(pool->adapter_scale) & 3) return LORA_ERR_ALIGN;
        if (pool->adapter_type != LORA_ADAPTER_BF16 && pool->adapter_type != LORA_ADAPTER_E4M3) return LORA_ERR_SHAPE;
        if (pool->adapter_type == LORA_ADAPTER_E4M3) {
            if (!pool->dequant) return LORA_ERR_NULL;
            if ((reinterpret_cast<uintptr_t>(pool->dequant) & 3) || !aligned16(pool->widened)) return LORA_ERR_ALIGN;
        }
        if (pool->max_rank < LORA_RANK_ALIGN || pool->max_rank > LORA_MAX_RANK || (pool->max_rank % LORA_RANK_ALIGN))
            return LORA_ERR_RANK;
        if (S > 1 && pool->max_rank % (LORA_RANK_ALIGN * S)) return LORA_ERR_RANK;   // whole panels per slice
        if (pool->a_elems <= 0 || pool->b_elems <= 0 || (pool->a_elems % pool->K) || (pool->b_elems % kChunk))
            return LORA_ERR_SHAPE;
    }
    return LORA_OK;
}

struct Carve {
    WsLayout L;
    int32_t *counters;
};

static void fill_segments(void *ws, const WsLayout &L, int64_t M, const lora_pool_t *pool, lora_segments_t *out)
{
    out->perm = at<int32_t>(ws, L.perm);
    out->bucket_offsets = at<int32_t>(ws, L.offsets);
    out->seg_id = at<int32_t>(ws, L.seg_id);
    out->seg_start = at<int32_t>(ws, L.seg_start);
    out->seg_len = at<int32_t>(ws, L.seg_len);
    out->seg_rank = at<int32_t>(ws, L.seg_rank);
    out->num_segments = at<int32_t>(ws, L.num_segments);
    out->plan = ws;
    out->M = M;
    out->num_adapters = pool->num_adapters;
    out->num_slices = pool->num_slices > 1 ? pool->num_slices : 1;
}

static void fill_seg_params(SegParams &p, const int32_t *ids, int64_t M, const lora_pool_t *pool, const WsLayout &L,
                            void *ws)
{
    p.ids = ids;
    p.M = M;
    p.A = pool->num_adapters;
    p.K = pool->K;
    p.N = pool->N;
    p.num_mtiles = L.num_mtiles;
    p.rank = pool->rank;
    p.a_offset = pool->a_offset;
    p.b_offset = pool->b_offset;
    p.perm = at<int32_t>(ws, L.perm);
    p.offsets = at<int32_t>(ws, L.offsets);
    p.seg_id = at<int32_t>(ws, L.seg_id);
    p.seg_start = at<int32_t>(ws, L.seg_start);
    p.seg_len = at<int32_t>(ws, L.seg_len);
    p.seg_rank = at<int32_t>(ws, L.seg_rank);
    p.num_segments = at<int32_t>(ws, L.num_segments);
    p.hdr = at<int32_t>(ws, L.hdr);
    p.tile_chunk_off = at<int32_t>(ws, L.tile_chunk_off);
    p.chunk_arow = at<int32_t>(ws, L.chunk_arow);
    p.chunk_bpanel = at<int32_t>(ws, L.chunk_bpanel);
    p.chunk_rng = at<int32_t>(ws, L.chunk_rng);
    p.sjob_tile = at<int32_t>(ws, L.sjob_tile);
    p.sjob_c0 = at<int32_t>(ws, L.sjob_c0);
    p.sjob_c1 = at<int32_t>(ws, L.sjob_c1);
    p.tile_njobs = at<int32_t>(ws, L.tile_njobs);
    p.dchunk_arow = at<int32_t>(ws, L.dchunk_arow);
    p.dchunk_bpanel = at<int32_t>(ws, L.dchunk_bpanel);
    p.dchunk_adapter = at<int32_t>(ws, L.dchunk_adapter);
    p.counters = at<int32_t>(ws, L.counters);
    p.n_counters = static_cast<int32_t>(L.n_counters);
    p.num_slices = pool->num_slices > 1 ? pool->num_slices : 1;
}

// The table checker over the table in ws (lora_check_segments; after every
// table build in the LORA_DEBUG build).
static int enqueue_check(const int32_t *ids, int64_t M, const lora_pool_t *pool, const WsLayout &L, void *ws,
                         cudaStream_t stream)
{
    SegCheckParams q;
    fill_seg_params(q.s, ids, M, pool, L, ws);
    q.max_chunks = L.max_chunks;
    q.max_sjobs = L.max_sjobs;
    q.max_dchunks = L.max_dchunks;
    q.a_rows = pool->num_adapters ? pool->a_elems / pool->K : 0;
    q.b_panels = pool->num_adapters ? pool->b_elems / (static_cast<int64_t>(kChunk) * pool->N) : 0;
    return launch_seg_check(q, stream) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

static int enqueue_segments(const int32_t *ids, int64_t M, const lora_pool_t *pool, const WsLayout &L, void *ws,
                            cudaStream_t stream, bool pdl = false)
{
    SegParams p;
    fill_seg_params(p, ids, M, pool, L, ws);
    if (launch_seg_build(p, pdl, stream) != cudaSuccess) return LORA_ERR_CUDA;
    return kDebugChecks ? enqueue_check(ids, M, pool, L, ws, stream) : LORA_OK;
}

// Validate the common arguments and make sure a segment table exists in ws
// (unless build is false: the caller enqueues it itself).
static int prepare(const int32_t *ids, int64_t M, const lora_pool_t *pool, const lora_segments_t *segs, void *ws,
                   size_t ws_bytes, cudaStream_t stream, WsLayout *L, bool build = true)
{
    int rc = check_pool(pool);
    if (rc) return rc;
    if (M < 0) return LORA_ERR_SHAPE;
    if (M > kMaxTokens) return LORA_ERR_SHAPE;
    if (!ws) return LORA_ERR_WORKSPACE;
    if (!device_supported()) return LORA_ERR_UNSUPPORTED;
    *L = make_ws_layout(M, pool->N, pool->num_adapters);
    if (ws_bytes < L->total_min) return LORA_ERR_WORKSPACE;
    if (segs) {
        if (segs->plan != ws || segs->M != M || segs->num_adapters != pool->num_adapters ||
            segs->num_slices != (pool->num_slices > 1 ? pool->num_slices : 1) || segs->perm != at<int32_t>(ws, L->perm))
            return LORA_ERR_SEGMENTS;
        // the LORA_DEBUG build checks a prebuilt table before it is used
        return kDebugChecks && ids ? enqueue_check(ids, M, pool, *L, ws, stream) : LORA_OK;
    }
    if (!ids) return LORA_ERR_NULL;
    return build ? enqueue_segments(ids, M, pool, *L, ws, stream) : LORA_OK;
}

static std::atomic<int64_t> g_wait_cycles{kDefaultWaitCycles};

int64_t tc_wait_cycles() { return g_wait_cycles.load(std::memory_order_relaxed); }

// The shared part of a tiled launch's parameters (the table, the workspace,
// the S panel scratch at s_panels); the layers are filled by run_tiled.
static void fill_tc_params(TcParams &p, const WsLayout &L, void *ws, const lora_pool_t *pool, int64_t M,
                           uint16_t *s_panels)
{
    std::memset(&p, 0, sizeof p);
    p.M = M;
    p.out_rows = M;
    p.num_adapters = pool->num_adapters;
    p.num_slices = pool->num_slices > 1 ? pool->num_slices : 1;
    p.num_layers = 1;
    p.num_mtiles = L.num_mtiles;
    p.group_m = 8;
    p.s_panels = s_panels;
    p.perm = at<int32_t>(ws, L.perm);
    p.offsets = at<int32_t>(ws, L.offsets);
    p.hdr = at<int32_t>(ws, L.hdr);
    p.tile_chunk_off = at<int32_t>(ws, L.tile_chunk_off);
    p.chunk_arow = at<int32_t>(ws, L.chunk_arow);
    p.chunk_bpanel = at<int32_t>(ws, L.chunk_bpanel);
    p.chunk_rng = at<int32_t>(ws, L.chunk_rng);
    p.sjob_tile = at<int32_t>(ws, L.sjob_tile);
    p.sjob_c0 = at<int32_t>(ws, L.sjob_c0);
    p.sjob_c1 = at<int32_t>(ws, L.sjob_c1);
    p.tile_njobs = at<int32_t>(ws, L.tile_njobs);
    p.counters = at<int32_t>(ws, L.counters);
    p.shrink_split = 1;
    p.wait_cycles = tc_wait_cycles();
    p.s_sets = 1;
    p.s_set_rows = L.max_chunks * kBM;
}

// Layer l of a tiled launch.
static void fill_tc_layer(TcLayer &Ly, const lora_pool_t *pool, const lora_bf16_t *x, const lora_bf16_t *bias,
                          float scale, lora_bf16_t *y)
{
    std::memset(&Ly, 0, sizeof Ly);
    Ly.N = pool->N;
    Ly.K = pool->K;
    Ly.kblocks = (pool->K + kBK - 1) / kBK;
    Ly.num_ntiles = (pool->N + kBN - 1) / kBN;
    const int S = pool->num_slices > 1 ? pool->num_slices : 1;
    for (int s = 0; s <= LORA_MAX_SLICES; ++s) Ly.slice_start[s] = s <= S && S > 1 ? pool->slice_start[s] : 0;
    Ly.scale = scale;
    Ly.adapter_scale = pool->num_adapters ? pool->adapter_scale : nullptr;
    Ly.bias = bias;
    Ly.x = x;
    Ly.y = y;
}

// Maps shared by the schedules: A pool (16-row boxes), B pool (16-col panels).
template <typename Maps>
static bool encode_pool_maps(Maps &m, const lora_pool_t *pool, const void *dummy, uint32_t b_rows_box)
{
    const uint64_t K = pool->K;
    if (pool->num_adapters > 0) {
        if (!encode_2d(&m.a, pool->a_pool, K, pool->a_elems / K, K * 2, kBK, kChunk, CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
        if (!encode_2d(&m.a32, pool->a_pool, K, pool->a_elems / K, K * 2, kBK, 2 * kChunk, CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
        if (!encode_2d(&m.a48, pool->a_pool, K, pool->a_elems / K, K * 2, kBK, 3 * kChunk, CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
        if (!encode_2d(&m.a64, pool->a_pool, K, pool->a_elems / K, K * 2, kBK, 4 * kChunk, CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
        if (!encode_2d(&m.b, pool->b_pool, kChunk, pool->b_elems / kChunk, kChunk * 2, kChunk, b_rows_box,
                       CU_TENSOR_MAP_SWIZZLE_32B))
            return false;
    } else {
        if (!encode_2d(&m.a, dummy, K, 1, K * 2, kBK, kChunk, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
        m.a32 = m.a48 = m.a64 = m.a;
        if (!encode_2d(&m.b, dummy, kChunk, 1, kChunk * 2, kChunk, b_rows_box, CU_TENSOR_MAP_SWIZZLE_32B))
            return false;
    }
    return true;
}

// e4m3 pools: enqueue the widening of the adapters the table in ws names
// into the pool's bf16 scratch, with this call's per-adapter factors
// (mode: kWiden*) in factor row `slot` of the workspace, and describe the
// widened pool in *out.  bf16 pools: *out is the pool itself.
static int widen_pool(const lora_pool_t *pool, const WsLayout &L, void *ws, int mode, int slot, cudaStream_t stream,
                      lora_pool_t *out)
{
    *out = *pool;
    if (pool->adapter_type != LORA_ADAPTER_E4M3 || pool->num_adapters == 0) return LORA_OK;
    if (!pool->widened) return LORA_ERR_NULL;
    WidenParams w;
    std::memset(&w, 0, sizeof w);
    w.a8 = reinterpret_cast<const uint8_t *>(pool->a_pool);
    w.b8 = reinterpret_cast<const uint8_t *>(pool->b_pool);
    w.aw = pool->widened;
    w.bw = pool->widened + pool->a_elems;
    w.a_off = pool->a_offset;
    w.b_off = pool->b_offset;
    w.rank = pool->rank;
    w.K = pool->K;
    w.N = pool->N;
    w.A = pool->num_adapters;
    const int max_seg = static_cast<int>(std::min<int64_t>(pool->num_adapters, std::max<int64_t>(L.M, 1)));
    w.parts = std::max(1, 2 * num_sms_current_device() / std::max(1, max_seg));
    w.mode = mode;
    w.seg_id = at<int32_t>(ws, L.seg_id);
    w.num_segments = at<int32_t>(ws, L.num_segments);
    w.dequant = pool->dequant;
    w.adapter_scale = pool->adapter_scale;
    w.fac = at<float>(ws, L.fac) + static_cast<size_t>(slot) * std::max(pool->num_adapters, 1);
    if (launch_widen(w, max_seg, stream) != cudaSuccess) return LORA_ERR_CUDA;
    out->a_pool = pool->widened;
    out->b_pool = pool->widened + pool->a_elems;
    out->adapter_type = LORA_ADAPTER_BF16;
    out->adapter_scale = w.fac;
    out->dequant = nullptr;
    out->widened = nullptr;
    return LORA_OK;
}

// One layer of a tiled launch as the caller gives it.
struct LayerCall {
    const lora_bf16_t *x, *W, *bias;
    const lora_pool_t *pool;
    float scale;
    lora_bf16_t *y;
};

// The tiled schedule over nl layers that share the segment table in ws:
// one launch whose work list runs every layer's shrink items, then every
// layer's output tiles.  The layers' S panel sets start at s_panels
// (nl x tiled_s_sets(M) sets).  Stream-K (splitting a partial last wave
// along K) is used by one-layer fused calls only.
static int run_tiled(const LayerCall *lc, int nl, int64_t M, const int32_t *ids, void *ws, size_t ws_bytes,
                     const WsLayout &L, int mode, float *s_out, int32_t s_cols, const float *s_in, uint16_t *s_panels,
                     cudaStream_t stream)
{
    TcArgs a;
    std::memset(&a, 0, sizeof a);
    TcParams &p = a.p;
    fill_tc_params(p, L, ws, lc[0].pool, M, s_panels);
    p.num_layers = nl;
    const int sms = num_sms_current_device();
    int64_t n_out = 0;
    bool long_k = true;
    for (int l = 0; l < nl; ++l) {
        fill_tc_layer(p.layer[l], lc[l].pool, lc[l].x, lc[l].bias, lc[l].scale, lc[l].y);
        p.layer[l].tile0 = static_cast<int32_t>(n_out);
        n_out += static_cast<int64_t>(p.num_mtiles) * p.layer[l].num_ntiles;
        long_k = long_k && p.layer[l].kblocks >= 16;
    }
    // two K halves per shrink job when each half keeps 8 K blocks or more
    // and the output tiles fill at most four waves of the grid: the first
    // wave of output tiles then finds S ready when its own K loops end (a
    // wait that matters only while there are few waves).  Each half writes
    // its own S panel set; the expand steps add both, (S_a + S_b) B^T =
    // S_a B^T + S_b B^T, in the fp32 accumulator.
    p.shrink_split = (tiled_s_sets(M) == 2 && long_k && n_out <= 4 * sms) ? 2 : 1;
    p.s_sets = p.shrink_split;
    // stream-K for the last partial wave: the fused layer only, when the
    // workspace holds the partial-sum scratch and the grid fits its tiles
    if (mode == kModeLinear && nl == 1 && L.sk_part && ws_bytes >= L.total && sms <= kStreamKMaxTiles) {
        p.streamk = 1;
        p.sk_part = at<float>(ws, L.sk_part);
        p.sk_cnt = at<int32_t>(ws, L.sk_cnt);
    }
    p.mode = mode;
    p.ids = ids;
    // shrink mode: the pool's factor is what S is multiplied by (the caller
    // passes none for a bf16 pool: S leaves unscaled; an e4m3 pool's A factor)
    if (mode == kModeExpand) p.s_sets = 1;   // the caller's S, prepared as one panel set
    p.s_out = s_out;
    p.s_cols = s_cols;
    for (int l = 0; l < nl; ++l) {
        const lora_pool_t *pool = lc[l].pool;
        const uint64_t K = pool->K, N = pool->N;
        TcLayerMaps &m = a.maps[l];
        const void *xsrc = lc[l].x ? static_cast<const void *>(lc[l].x) : static_cast<const void *>(s_panels);
        const uint64_t xrows = lc[l].x ? static_cast<uint64_t>(M) : 1;
        if (!encode_2d(&m.x, xsrc, K, xrows, K * 2, kBK, 1, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ERR_CUDA;
        const void *wsrc = lc[l].W ? static_cast<const void *>(lc[l].W) : xsrc;
        if (!encode_2d(&m.w, wsrc, K, lc[l].W ? N : 1, K * 2, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B))
            return LORA_ERR_CUDA;
        if (!encode_pool_maps(m, pool, s_panels, kBN)) return LORA_ERR_CUDA;
    }
    const uint64_t s_rows = static_cast<uint64_t>(nl) * tiled_s_sets(M) * L.max_chunks * kBM;
    if (!encode_2d(&a.s, s_panels, kChunk, s_rows, kChunk * 2, kChunk, kBM, CU_TENSOR_MAP_SWIZZLE_32B))
        return LORA_ERR_CUDA;
    if (mode == kModeExpand) {
        if (launch_s_prep(s_in, s_cols, lc[0].scale, p, stream) != cudaSuccess) return LORA_ERR_CUDA;
    }
    int64_t jobs = 0;
    if (mode != kModeShrink) jobs += n_out;
    if (mode != kModeExpand) jobs += static_cast<int64_t>(L.max_sjobs) * p.shrink_split * nl;
    // with stream-K the last partial wave is shared out over every SM
    const int grid = p.streamk ? sms : static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms, jobs)));
    return launch_tc(a, grid, stream) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

// One layer (lora_linear, lora_shrink, lora_expand), S panels in the
// workspace's own scratch.
static int run_tiled(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                     const int32_t *ids, const lora_pool_t *pool, float scale, lora_bf16_t *y, void *ws,
                     size_t ws_bytes, const WsLayout &L, int mode, float *s_out, int32_t s_cols, const float *s_in,
                     cudaStream_t stream)
{
    const LayerCall lc = {x, W, bias, pool, scale, y};
    return run_tiled(&lc, 1, M, ids, ws, ws_bytes, L, mode, s_out, s_cols, s_in, at<uint16_t>(ws, L.s_scratch),
                     stream);
}

static int run_splitk(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                      const int32_t *ids, const lora_pool_t *pool, float scale, lora_bf16_t *y, void *ws,
                      const WsLayout &L, cudaStream_t stream)
{
    SplitParams p;
    std::memset(&p, 0, sizeof p);
    const int G = num_sms_current_device();
    const int T = split_tpad(M);
    p.M = M;
    p.N = pool->N;
    p.K = pool->K;
    p.T_pad = T;
    p.kblocks = (pool->K + kBK - 1) / kBK;
    p.NT = (pool->N + kSplitBN - 1) / kSplitBN;
    p.stages = splitk_stages(T);
    int tc = 32;
    while (tc < 2 * T) tc <<= 1;
    p.tmem_cols = tc;
    const int RTmax = (L.max_dchunks + 7) / 8;
    if ((RTmax + G - 1) / G + 2 + (p.NT + G - 1) / G + 2 > splitk_max_runs()) return LORA_ERR_SHAPE;
    p.A = pool->num_adapters;
    p.scale = scale;
    p.adapter_scale = pool->num_adapters ? pool->adapter_scale : nullptr;
    p.bias = bias;
    p.y = y;
    p.ids = ids;
    p.hdr = at<int32_t>(ws, L.hdr);
    p.dchunk_arow = at<int32_t>(ws, L.dchunk_arow);
    p.dchunk_bpanel = at<int32_t>(ws, L.dchunk_bpanel);
    p.dchunk_adapter = at<int32_t>(ws, L.dchunk_adapter);
    p.s_panels = at<uint16_t>(ws, L.s_scratch);
    p.acc_out = at<float>(ws, L.acc_out);
    p.acc_shr = at<float>(ws, L.acc_shr);
    p.counters = at<int32_t>(ws, L.counters);
    p.wait_cycles = tc_wait_cycles();
    const uint64_t K = pool->K, N = pool->N;
    TcMaps m;
    if (!encode_2d(&m.x, x, K, static_cast<uint64_t>(M), K * 2, kBK, T, CU_TENSOR_MAP_SWIZZLE_128B))
        return LORA_ERR_CUDA;
    if (!encode_2d(&m.w, W, K, N, K * 2, kBK, kSplitBN, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ERR_CUDA;
    if (!encode_pool_maps(m, pool, p.s_panels, kSplitBN)) return LORA_ERR_CUDA;
    if (!encode_2d(&m.s, p.s_panels, kChunk, static_cast<uint64_t>(L.max_dchunks) * T, kChunk * 2, kChunk, T,
                   CU_TENSOR_MAP_SWIZZLE_32B))
        return LORA_ERR_CUDA;
    return launch_splitk(m, p, G, stream) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

// Weight-streaming schedule (M <= 64, K a multiple of 64): one cluster of C
// CTAs per 128-feature output tile.  Returns -1 when this device / shape
// cannot host it, so the caller falls back to split-K.  pdl: launch it as a
// programmatic dependent of whatever kernel precedes it on the stream; it
// then streams its first weight boxes before that kernel has finished
// (LORA_FLAG_STATIC_WEIGHTS).  build: one more cluster, whose first CTA
// builds the call's segment table in ws beside the weight stream (the
// kernel itself reads no table).
static int run_cluster(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                       const int32_t *ids, const lora_pool_t *pool, float scale, lora_bf16_t *y, void *ws,
                       const WsLayout &L, bool pdl, bool build, cudaStream_t stream)
{
    if (M > kStreamMaxTokens || (pool->K % kBK) != 0) return -1;
    const int T = split_tpad(M);
    const int NT = (pool->N + kSplitBN - 1) / kSplitBN;
    const int sms = num_sms_current_device();
    // one cached choice of C per (device, NT, T)
    struct Pick {
        int dev, NT, T, C;
    };
    static Pick cache[32];
    static int ncache = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    int C = -1;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < ncache; ++i)
            if (cache[i].dev == dev && cache[i].NT == NT && cache[i].T == T) C = cache[i].C;
        if (C < 0) {
            C = cluster_pick_size(NT, T, sms);
            cache[ncache % 32] = {dev, NT, T, C};
            ncache = ncache < 32 ? ncache + 1 : 32;
        }
    }
    if (C <= 0) return -1;
    const int grid = C * NT;
    const int kblocks = pool->K / kBK;
    const int64_t KU2 = (kblocks + 1) / 2;
    const int max_regions = std::min(cluster_max_regions(), 512 / T);
    const uint64_t panels =
        pool->num_adapters ? static_cast<uint64_t>(pool->b_elems / (static_cast<int64_t>(kChunk) * pool->N)) : 1;
    if ((panels + cluster_win() - 1) / cluster_win() > 512) return -1;   // the kernel's window bitmap
    // windows the kernel can shrink: those a batch touches, at most all of the pool's
    const int64_t wins = std::min<int64_t>(L.max_win_str, (panels + cluster_win() - 1) / cluster_win());
    // the shrink runs and expand windows of one CTA fit its on-chip tables
    const int64_t u_cta = (wins * KU2 + grid - 1) / grid;
    const int64_t runs = (u_cta + KU2 - 1) / KU2 + 1;
    if (runs > cluster_max_runs() || runs + 1 > max_regions) return -1;
    if ((wins + C - 1) / C > cluster_max_win_cta()) return -1;
    if (std::max<int64_t>(wins, 1) * KU2 * grid >= (int64_t(1) << 31)) return -1;   // 32-bit slicing
    ClusterParams p;
    std::memset(&p, 0, sizeof p);
    p.M = M;
    p.N = pool->N;
    p.K = pool->K;
    p.T_pad = T;
    p.C = C;
    p.NT = NT;
    p.kblocks = kblocks;
    p.stages = cluster_stages(T);
    p.s_ring = cluster_s_ring(T, p.stages);
    p.max_regions = max_regions;
    p.max_win_str = L.max_win_str;
    p.A = pool->num_adapters;
    p.a_offset = pool->a_offset;
    p.rank = pool->rank;
    p.windows_all = pool->num_adapters ? static_cast<int32_t>((panels + cluster_win() - 1) / cluster_win()) : 0;
    // a pool no larger than what one batch could touch is processed whole:
    // the unit list is then known at launch and the shrink can go first
    p.all_windows = p.windows_all <= L.max_win_str ? 1 : 0;
    p.early_weights = pdl ? 1 : 0;
    if (build) {
        if (cluster_build_smem_bytes(pool->num_adapters) + 1024 > cluster_smem_bytes(T, p.stages, p.s_ring)) return -1;
        p.build = 1;
        fill_seg_params(p.seg, ids, M, pool, L, ws);
    }
    p.scale = scale;
    p.adapter_scale = pool->num_adapters ? pool->adapter_scale : nullptr;
    p.fp8 = pool->num_adapters && pool->adapter_type == LORA_ADAPTER_E4M3 ? 1 : 0;
    p.dequant = p.fp8 ? pool->dequant : nullptr;
    p.bias = bias;
    p.x = x;
    p.y = y;
    p.ids = ids;
    p.acc = at<float>(ws, L.acc_str);
    p.wcnt = at<int32_t>(ws, L.wcnt);
    p.counters = at<int32_t>(ws, L.counters);
    const uint64_t K = pool->K, N = pool->N, KB = kblocks;
    ClusterMaps m;
    const CUtensorMapSwizzle s128 = CU_TENSOR_MAP_SWIZZLE_128B, s32 = CU_TENSOR_MAP_SWIZZLE_32B;
    if (!encode_3d(&m.w3, W, kBK, N, KB, K * 2, kBK * 2, kBK, kSplitBN, 2, s128)) return LORA_ERR_CUDA;
    if (!encode_3d(&m.x3, x, kBK, static_cast<uint64_t>(M), KB, K * 2, kBK * 2, kBK, static_cast<uint32_t>(T), 2, s128))
        return LORA_ERR_CUDA;
    const void *apool = pool->num_adapters ? static_cast<const void *>(pool->a_pool) : static_cast<const void *>(W);
    const uint64_t arows = pool->num_adapters ? static_cast<uint64_t>(pool->a_elems / pool->K) : 1;
    const void *bpool = pool->num_adapters ? static_cast<const void *>(pool->b_pool) : static_cast<const void *>(W);
    if (p.fp8) {
        // e4m3 pools, one byte per element: a shrink unit's A box is 128
        // rows x 128 K codes, an expand window's B box 8 panels x 128 rows x
        // 16 codes (16 KB each, unswizzled); the kernel widens them in place
        const CUtensorMapSwizzle s0 = CU_TENSOR_MAP_SWIZZLE_NONE;
        const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        if (!encode_2d(&m.a3, apool, K, arows, K, 2 * kBK, kSplitBN, s0, u8)) return LORA_ERR_CUDA;
        if (!encode_3d(&m.b3, bpool, kChunk, N, panels, kChunk, N * kChunk, kChunk, kSplitBN, cluster_win(), s0, u8))
            return LORA_ERR_CUDA;
    } else {
        if (!encode_3d(&m.a3, apool, kBK, arows, KB, K * 2, kBK * 2, kBK, kSplitBN, 2, s128)) return LORA_ERR_CUDA;
        if (!encode_3d(&m.b3, bpool, kChunk, N, panels, kChunk * 2, N * kChunk * 2, kChunk, kSplitBN, cluster_win(),
                       s32))
            return LORA_ERR_CUDA;
    }
    if (launch_cluster(m, p, pdl, stream) != cudaSuccess) return LORA_ERR_CUDA;
    // the table this launch built, checked once the launch is complete
    return kDebugChecks && build ? enqueue_check(ids, M, pool, L, ws, stream) : LORA_OK;
}

}  // namespace lora

using namespace lora;

// ---- mixture of experts ----------------------------------------------------
// Workspace of the routing and the grouped GEMM: the status / counter block,
// the routing's perm, bucket offsets and segment table over the M * topk
// (token, slot) pairs, then the padded expert order (each expert's pairs
// from a fresh 128-row tile, -1 in the gaps), each tile's expert and the
// routing's per-chunk bucket counts.
struct MoeLayout {
    int64_t P;                 // pairs
    int32_t E, max_mtiles;
    size_t counters, n_counters, perm, offsets, seg_id, seg_start, seg_len, seg_rank, num_segments, hdr;
    size_t perm_pad, mt_expert, route_cnt, total;
    int32_t chunk, nchunks;    // the routing's pairs per CTA and CTAs
};

static MoeLayout make_moe_layout(int64_t M, int32_t topk, int32_t E)
{
    MoeLayout L;
    std::memset(&L, 0, sizeof L);
    L.P = M * topk;
    L.E = E;
    L.max_mtiles = static_cast<int32_t>((L.P + kBM - 1) / kBM + E);
    L.n_counters = CNT_FIXED + 8;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    L.counters = take(L.n_counters * 4);
    L.perm = take(static_cast<size_t>(std::max<int64_t>(L.P, 1)) * 4);
    L.offsets = take(static_cast<size_t>(E + 2) * 4);
    L.seg_id = take(static_cast<size_t>(std::max(E, 1)) * 4);
    L.seg_start = take(static_cast<size_t>(std::max(E, 1)) * 4);
    L.seg_len = take(static_cast<size_t>(std::max(E, 1)) * 4);
    L.seg_rank = take(static_cast<size_t>(std::max(E, 1)) * 4);
    L.num_segments = take(4);
    L.hdr = take(HDR_WORDS * 4);
    L.perm_pad = take(static_cast<size_t>(L.max_mtiles) * kBM * 4);
    L.mt_expert = take(static_cast<size_t>(L.max_mtiles) * 4);
    // the routing's chunks: 1024 pairs or more per CTA (a multiple of 256),
    // at most kRouteMaxChunks of them, and their bucket counts
    const int64_t per = (L.P + kRouteMaxChunks - 1) / kRouteMaxChunks;
    L.chunk = static_cast<int32_t>(std::max<int64_t>(1024, (per + 255) / 256 * 256));
    L.nchunks = static_cast<int32_t>(std::max<int64_t>(1, (L.P + L.chunk - 1) / L.chunk));
    L.route_cnt = take(static_cast<size_t>(L.nchunks) * (E + 1) * 4);
    L.total = o;
    return L;
}

static int check_moe(int64_t M, int32_t K, int32_t N, int32_t E, int32_t topk)
{
    if (M < 0 || K <= 0 || N <= 0 || (K % 8) || (N % 8)) return LORA_ERR_SHAPE;
    if (E <= 0 || E > LORA_MAX_ADAPTERS || topk <= 0 || topk > E) return LORA_ERR_SHAPE;
    if (M * topk > (int64_t(1) << 31) - 2 * kBM * static_cast<int64_t>(E)) return LORA_ERR_SHAPE;
    if (static_cast<int64_t>(E) * N >= (int64_t(1) << 31)) return LORA_ERR_SHAPE;   // stacked weight rows
    return LORA_OK;
}

extern "C" {

size_t lora_moe_workspace_size(int64_t M, int32_t topk, int32_t num_experts)
{
    if (M < 0 || topk <= 0 || num_experts <= 0) return 0;
    return make_moe_layout(M, topk, num_experts).total;
}

// The routing's parameters over the workspace ws of layout L.
static RouteParams route_params(const int32_t *expert, const MoeLayout &L, void *ws)
{
    RouteParams p;
    std::memset(&p, 0, sizeof p);
    p.expert = expert;
    p.P = L.P;
    p.E = L.E;
    p.nb = L.E + 1;
    p.chunk = L.chunk;
    p.nchunks = L.nchunks;
    p.max_mtiles = L.max_mtiles;
    p.n_counters = static_cast<int32_t>(L.n_counters);
    p.cnt = at<int32_t>(ws, L.route_cnt);
    p.perm = at<int32_t>(ws, L.perm);
    p.offsets = at<int32_t>(ws, L.offsets);
    p.seg_id = at<int32_t>(ws, L.seg_id);
    p.seg_start = at<int32_t>(ws, L.seg_start);
    p.seg_len = at<int32_t>(ws, L.seg_len);
    p.seg_rank = at<int32_t>(ws, L.seg_rank);
    p.num_segments = at<int32_t>(ws, L.num_segments);
    p.hdr = at<int32_t>(ws, L.hdr);
    p.counters = at<int32_t>(ws, L.counters);
    p.perm_pad = at<int32_t>(ws, L.perm_pad);
    p.mt_expert = at<int32_t>(ws, L.mt_expert);
    return p;
}

// Shared validation of the routing calls; *L receives the layout.
static int route_prepare(const int32_t *expert, int64_t M, int32_t topk, int32_t num_experts, void *ws,
                         size_t ws_bytes, MoeLayout *L)
{
    int rc = check_moe(M, 8, 8, num_experts, topk);
    if (rc) return rc;
    if (M == 0) return LORA_OK;
    if (!expert) return LORA_ERR_NULL;
    *L = make_moe_layout(M, topk, num_experts);
    if (!ws || ws_bytes < L->total) return LORA_ERR_WORKSPACE;
    if (!device_supported()) return LORA_ERR_UNSUPPORTED;
    return LORA_OK;
}

int lora_moe_route(const int32_t *expert, int64_t M, int32_t topk, int32_t num_experts, void *ws, size_t ws_bytes,
                   lora_stream_t stream)
{
    MoeLayout L;
    const int rc = route_prepare(expert, M, topk, num_experts, ws, ws_bytes, &L);
    if (rc || M == 0) return rc;
    const RouteParams p = route_params(expert, L, ws);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_moe_route(p, s) != cudaSuccess) return LORA_ERR_CUDA;
    // the LORA_DEBUG build checks every routing it makes
    return kDebugChecks && launch_moe_route_check(p, s) != cudaSuccess ? LORA_ERR_CUDA : LORA_OK;
}

int lora_moe_check_route(const int32_t *expert, int64_t M, int32_t topk, int32_t num_experts, void *ws,
                         size_t ws_bytes, lora_stream_t stream)
{
    MoeLayout L;
    const int rc = route_prepare(expert, M, topk, num_experts, ws, ws_bytes, &L);
    if (rc || M == 0) return rc;
    return launch_moe_route_check(route_params(expert, L, ws), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? LORA_OK
               : LORA_ERR_CUDA;
}

int lora_moe_gemm(const lora_bf16_t *x, int64_t M, int32_t K, const lora_bf16_t *W, int32_t N, int32_t num_experts,
                  int32_t topk, lora_bf16_t *out, void *ws, size_t ws_bytes, lora_stream_t stream)
{
    int rc = check_moe(M, K, N, num_experts, topk);
    if (rc) return rc;
    if (M == 0) return LORA_OK;
    if (!x || !W || !out) return LORA_ERR_NULL;
    if (!aligned16(x) || !aligned16(W) || !aligned16(out)) return LORA_ERR_ALIGN;
    const MoeLayout L = make_moe_layout(M, topk, num_experts);
    if (!ws || ws_bytes < L.total) return LORA_ERR_WORKSPACE;
    if (!device_supported()) return LORA_ERR_UNSUPPORTED;
    const uint64_t Kq = K;
    if (L.max_mtiles <= kMoePairMaxTiles) {
        // two token tiles of an expert per work item (moe_pair.cu)
        CUtensorMap w;
        if (!encode_2d(&w, W, Kq, static_cast<uint64_t>(num_experts) * N, Kq * 2, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B))
            return LORA_ERR_CUDA;
        MoePairParams mp;
        mp.x = x;
        mp.out = out;
        mp.perm_pad = at<int32_t>(ws, L.perm_pad);
        mp.mt_expert = at<int32_t>(ws, L.mt_expert);
        mp.hdr = at<int32_t>(ws, L.hdr);
        mp.status = at<int32_t>(ws, L.counters) + CNT_STATUS;
        mp.out_rows = M * static_cast<int64_t>(topk);
        mp.K = K;
        mp.N = N;
        mp.topk = topk;
        mp.kblocks = (K + kBK - 1) / kBK;
        mp.num_ntiles = (N + kBN - 1) / kBN;
        mp.max_mtiles = L.max_mtiles;
        mp.wait_cycles = tc_wait_cycles();
        return launch_moe_pair(w, mp, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
    }
    TcArgs a;
    std::memset(&a, 0, sizeof a);
    TcParams &p = a.p;
    p.M = static_cast<int64_t>(L.max_mtiles) * kBM;   // positions of the padded order
    p.num_mtiles = L.max_mtiles;                      // an upper bound: the kernel reads the routing's count
    p.num_layers = 1;
    p.layer[0].N = N;
    p.layer[0].K = K;
    p.layer[0].kblocks = (K + kBK - 1) / kBK;
    p.layer[0].num_ntiles = (N + kBN - 1) / kBN;
    p.layer[0].scale = 1.f;
    p.layer[0].x = x;
    p.layer[0].y = out;
    // one group of every token tile: the tiles that use one expert's weight
    // tile (its token tiles, for one column tile) are consecutive in the work
    // list and run in the same wave, so each weight tile is read from HBM
    // once (groups of 8 measured 168 us per grouped GEMM, one group 157 us)
    p.group_m = L.max_mtiles;
    p.mode = kModeMoe;
    p.num_slices = 1;
    p.topk = topk;
    p.out_rows = M * static_cast<int64_t>(topk);   // perm_pad names pairs (or -1)
    p.perm = at<int32_t>(ws, L.perm_pad);
    p.hdr = at<int32_t>(ws, L.hdr);
    p.counters = at<int32_t>(ws, L.counters);
    p.mt_expert = at<int32_t>(ws, L.mt_expert);
    p.shrink_split = 1;
    p.wait_cycles = tc_wait_cycles();
    p.s_sets = 1;
    TcLayerMaps &m = a.maps[0];
    if (!encode_2d(&m.x, x, Kq, static_cast<uint64_t>(M), Kq * 2, kBK, 1, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ERR_CUDA;
    // the experts' weights stacked: [E * N, K]
    if (!encode_2d(&m.w, W, Kq, static_cast<uint64_t>(num_experts) * N, Kq * 2, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B))
        return LORA_ERR_CUDA;
    lora_pool_t none;
    std::memset(&none, 0, sizeof none);
    none.K = K;
    none.N = N;
    if (!encode_pool_maps(m, &none, W, kBN)) return LORA_ERR_CUDA;
    if (!encode_2d(&a.s, W, kChunk, 1, kChunk * 2, kChunk, kBM, CU_TENSOR_MAP_SWIZZLE_32B)) return LORA_ERR_CUDA;
    return launch_tc(a, num_sms_current_device(), static_cast<cudaStream_t>(stream)) == cudaSuccess ? LORA_OK
                                                                                                    : LORA_ERR_CUDA;
}

int lora_moe_finalize(const lora_bf16_t *out, const int32_t *expert, const float *weight, int64_t M, int32_t topk,
                      int32_t num_experts, int32_t N, lora_bf16_t *y, lora_stream_t stream)
{
    int rc = check_moe(M, 8, N, num_experts, topk);
    if (rc) return rc;
    if (M == 0) return LORA_OK;
    if (!out || !expert || !weight || !y) return LORA_ERR_NULL;
    if (!aligned16(out) || !aligned16(y)) return LORA_ERR_ALIGN;
    if (!device_supported()) return LORA_ERR_UNSUPPORTED;
    return launch_moe_finalize(out, expert, weight, M, topk, num_experts, N, y, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? LORA_OK
               : LORA_ERR_CUDA;
}

int lora_moe(const lora_bf16_t *x, int64_t M, int32_t K, const lora_bf16_t *W, int32_t N, const int32_t *expert,
             const float *weight, int32_t num_experts, int32_t topk, lora_bf16_t *out, lora_bf16_t *y, void *ws,
             size_t ws_bytes, lora_stream_t stream)
{
    int rc = check_moe(M, K, N, num_experts, topk);
    if (rc) return rc;
    if (M == 0) return LORA_OK;
    if (!x || !W || !out || !y || !expert || !weight) return LORA_ERR_NULL;
    if ((rc = lora_moe_route(expert, M, topk, num_experts, ws, ws_bytes, stream))) return rc;
    if ((rc = lora_moe_gemm(x, M, K, W, N, num_experts, topk, out, ws, ws_bytes, stream))) return rc;
    return lora_moe_finalize(out, expert, weight, M, topk, num_experts, N, y, stream);
}

int lora_pool_layout(int32_t num_adapters, const int32_t *true_rank, int32_t K, int32_t N, int64_t *a_offset,
                     int64_t *b_offset, int32_t *rank_padded, int64_t *a_elems, int64_t *b_elems)
{
    if (num_adapters < 0 || num_adapters > LORA_MAX_ADAPTERS) return LORA_ERR_SHAPE;
    if (K <= 0 || N <= 0 || (K % 8) || (N % 8)) return LORA_ERR_SHAPE;
    if (!a_elems || !b_elems) return LORA_ERR_NULL;
    if (num_adapters > 0 && (!true_rank || !a_offset || !b_offset || !rank_padded)) return LORA_ERR_NULL;
    for (int i = 0; i < num_adapters; ++i)
        if (true_rank[i] < 1 || true_rank[i] > LORA_MAX_RANK) return LORA_ERR_RANK;
    // rank-grouped: padded rank 16, 32, ..., 128 in that order, id order inside
    std::vector<int> order(num_adapters);
    for (int i = 0; i < num_adapters; ++i) order[i] = i;
    auto rp = [&](int i) { return ((true_rank[i] + LORA_RANK_ALIGN - 1) / LORA_RANK_ALIGN) * LORA_RANK_ALIGN; };
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return rp(a) < rp(b); });
    int64_t a = 0, b = 0;
    for (int i : order) {
        rank_padded[i] = rp(i);
        a_offset[i] = a;
        b_offset[i] = b;
        a += static_cast<int64_t>(rp(i)) * K;
        b += static_cast<int64_t>(rp(i)) * N;
    }
    *a_elems = a;
    *b_elems = b;
    return LORA_OK;
}

size_t lora_workspace_size(int64_t M, int32_t N, int32_t num_adapters)
{
    if (M < 0 || M > kMaxTokens || N <= 0 || num_adapters < 0 || num_adapters > LORA_MAX_ADAPTERS) return 0;
    return make_ws_layout(M, N, num_adapters).total;
}

int lora_workspace_init(void *ws, size_t ws_bytes, lora_stream_t stream)
{
    if (!ws) return LORA_ERR_WORKSPACE;
    return cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LORA_OK
                                                                                                : LORA_ERR_CUDA;
}

int lora_build_segments(const int32_t *lora_id_map, int64_t M, const lora_pool_t *pool, lora_segments_t *out,
                        void *ws, size_t ws_bytes, lora_stream_t stream)
{
    if (!out) return LORA_ERR_NULL;
    WsLayout L;
    if (M == 0) {
        int rc = check_pool(pool);
        if (rc) return rc;
        L = make_ws_layout(0, pool->N, pool->num_adapters);
        if (!ws || ws_bytes < L.total_min) return LORA_ERR_WORKSPACE;
        fill_segments(ws, L, 0, pool, out);
        return LORA_OK;
    }
    int rc = prepare(lora_id_map, M, pool, nullptr, ws, ws_bytes, static_cast<cudaStream_t>(stream), &L);
    if (rc) return rc;
    fill_segments(ws, L, M, pool, out);
    return LORA_OK;
}

int lora_check_segments(const int32_t *lora_id_map, int64_t M, const lora_pool_t *pool, const lora_segments_t *segs,
                        void *ws, size_t ws_bytes, lora_stream_t stream)
{
    if (!segs) return LORA_ERR_NULL;
    if (M < 0) return LORA_ERR_SHAPE;
    if (M == 0) return check_pool(pool);
    if (!lora_id_map) return LORA_ERR_NULL;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsLayout L;
    const int rc = prepare(lora_id_map, M, pool, segs, ws, ws_bytes, s, &L);
    if (rc) return rc;
    return enqueue_check(lora_id_map, M, pool, L, ws, s);
}

int lora_linear_ex(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                   const int32_t *lora_id_map, const lora_pool_t *pool, float scale, const lora_segments_t *segs,
                   lora_bf16_t *y, void *ws, size_t ws_bytes, lora_stream_t stream, int32_t path)
{
    if (M < 0) return LORA_ERR_SHAPE;
    if (M == 0) return check_pool(pool);
    if (!x || !W || !y) return LORA_ERR_NULL;
    if (!aligned16(x) || !aligned16(W) || !aligned16(y) || (bias && !aligned16(bias))) return LORA_ERR_ALIGN;
    const int32_t flags = path & ~0xFF;
    path &= 0xFF;
    if (flags & ~LORA_FLAG_STATIC_WEIGHTS) return LORA_ERR_SHAPE;
    const bool static_weights = (flags & LORA_FLAG_STATIC_WEIGHTS) != 0;
    if (path < LORA_PATH_AUTO || path > LORA_PATH_STREAM) return LORA_ERR_SHAPE;
    if (path == LORA_PATH_SPLITK && M > kSplitMaxTokens) return LORA_ERR_SHAPE;
    if (path == LORA_PATH_STREAM && (M > kStreamMaxTokens || (pool && (pool->K % kBK)))) return LORA_ERR_SHAPE;
    if ((path == LORA_PATH_SPLITK || path == LORA_PATH_STREAM) && !lora_id_map) return LORA_ERR_NULL;
    if (pool && pool->adapter_scale && !lora_id_map) return LORA_ERR_NULL;   // the factors are looked up by id
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsLayout L;
    // The decode-sized schedule reads no segment table: a table this call
    // builds is enqueued after it, as a programmatic dependent that runs on a
    // free SM beside it.
    const bool stream_path = path == LORA_PATH_STREAM || (path == LORA_PATH_AUTO && M <= kStreamMaxTokens && lora_id_map);
    int rc = prepare(lora_id_map, M, pool, segs, ws, ws_bytes, s, &L, !stream_path);
    if (rc) return rc;
    if (stream_path) {
        const int rc2 = run_cluster(x, M, W, bias, lora_id_map, pool, scale, y, ws, L, static_weights, !segs, s);
        if (rc2 >= 0) return rc2;
        if (path == LORA_PATH_STREAM) return LORA_ERR_UNSUPPORTED;
        if (!segs && (rc = enqueue_segments(lora_id_map, M, pool, L, ws, s))) return rc;
    }
    lora_pool_t wpool;   // e4m3: the widened pool
    if ((rc = widen_pool(pool, L, ws, kWidenFused, 0, s, &wpool))) return rc;
    const bool splitk = path == LORA_PATH_SPLITK || (path == LORA_PATH_AUTO && M <= kSplitMaxTokens && lora_id_map);
    if (splitk) return run_splitk(x, M, W, bias, lora_id_map, &wpool, scale, y, ws, L, s);
    return run_tiled(x, M, W, bias, lora_id_map, &wpool, scale, y, ws, ws_bytes, L, kModeLinear, nullptr, 0, nullptr, s);
}

int lora_linear(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                const int32_t *lora_id_map, const lora_pool_t *pool, float scale, const lora_segments_t *segs,
                lora_bf16_t *y, void *ws, size_t ws_bytes, lora_stream_t stream)
{
    return lora_linear_ex(x, M, W, bias, lora_id_map, pool, scale, segs, y, ws, ws_bytes, stream, LORA_PATH_AUTO);
}

// ---- several layers in one launch -------------------------------------------
// Workspace of lora_linear_layers: the one-layer layout for the largest N
// (everything but the stream-K scratch), then the S panel sets of every layer.
static size_t layers_s_offset(const WsLayout &L) { return (L.total_min + 1023) & ~size_t(1023); }
static size_t layers_s_bytes(const WsLayout &L, int nl)
{
    return static_cast<size_t>(nl) * tiled_s_sets(L.M) * L.max_chunks * kBM * kChunk * 2;
}

size_t lora_layers_workspace_size(int64_t M, int32_t max_N, int32_t num_adapters, int32_t num_layers)
{
    if (M < 0 || M > kMaxTokens || max_N <= 0 || num_adapters < 0 || num_adapters > LORA_MAX_ADAPTERS) return 0;
    if (num_layers < 1 || num_layers > LORA_MAX_LAYERS) return 0;
    const WsLayout L = make_ws_layout(M, max_N, num_adapters);
    return layers_s_offset(L) + layers_s_bytes(L, num_layers);
}

int lora_linear_layers(const lora_layer_t *layers, int32_t num_layers, int64_t M, const int32_t *lora_id_map,
                       const lora_segments_t *segs, void *ws, size_t ws_bytes, lora_stream_t stream)
{
    if (!layers) return LORA_ERR_NULL;
    if (num_layers < 1 || num_layers > LORA_MAX_LAYERS || M < 0 || M > kMaxTokens) return LORA_ERR_SHAPE;
    // every layer: a valid pool holding the same adapters with the same
    // ranks and slicing as layer 0's (what one segment table can describe)
    const lora_pool_t *p0 = layers[0].pool;
    int32_t max_N = 0;
    bool factors = false;
    for (int l = 0; l < num_layers; ++l) {
        const lora_pool_t *pl = layers[l].pool;
        int rc = check_pool(pl);
        if (rc) return rc;
        if (pl->num_adapters != p0->num_adapters || pl->max_rank != p0->max_rank ||
            (pl->num_slices > 1 ? pl->num_slices : 1) != (p0->num_slices > 1 ? p0->num_slices : 1))
            return LORA_ERR_SHAPE;
        if (pl->num_adapters &&
            (pl->a_elems / pl->K != p0->a_elems / p0->K || pl->b_elems / pl->N != p0->b_elems / p0->N))
            return LORA_ERR_SHAPE;
        max_N = std::max(max_N, pl->N);
        factors = factors || (pl->num_adapters && pl->adapter_scale);
    }
    if (M == 0) return LORA_OK;
    for (int l = 0; l < num_layers; ++l) {
        const lora_layer_t &ly = layers[l];
        if (!ly.x || !ly.W || !ly.y) return LORA_ERR_NULL;
        if (!aligned16(ly.x) || !aligned16(ly.W) || !aligned16(ly.y) || (ly.bias && !aligned16(ly.bias)))
            return LORA_ERR_ALIGN;
    }
    if ((!segs || factors) && !lora_id_map) return LORA_ERR_NULL;   // the table is built from it; factors look it up
    if (!ws) return LORA_ERR_WORKSPACE;
    if (!device_supported()) return LORA_ERR_UNSUPPORTED;
    const WsLayout L = make_ws_layout(M, max_N, p0->num_adapters);
    if (ws_bytes < layers_s_offset(L) + layers_s_bytes(L, num_layers)) return LORA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (segs) {
        if (segs->plan != ws || segs->M != M || segs->num_adapters != p0->num_adapters ||
            segs->num_slices != (p0->num_slices > 1 ? p0->num_slices : 1) || segs->perm != at<int32_t>(ws, L.perm))
            return LORA_ERR_SEGMENTS;
        // the LORA_DEBUG build checks a prebuilt table before it is used
        if (kDebugChecks && lora_id_map) {
            int rc = enqueue_check(lora_id_map, M, p0, L, ws, s);
            if (rc) return rc;
        }
    } else {
        int rc = enqueue_segments(lora_id_map, M, p0, L, ws, s);
        if (rc) return rc;
    }
    LayerCall lc[LORA_MAX_LAYERS];
    lora_pool_t wpool[LORA_MAX_LAYERS];   // e4m3 layers: their widened pools
    for (int l = 0; l < num_layers; ++l) {
        int rc = widen_pool(layers[l].pool, L, ws, kWidenFused, l, s, &wpool[l]);
        if (rc) return rc;
        lc[l] = {layers[l].x, layers[l].W, layers[l].bias, &wpool[l], layers[l].scale, layers[l].y};
    }
    return run_tiled(lc, num_layers, M, lora_id_map, ws, ws_bytes, L, kModeLinear, nullptr, 0, nullptr,
                     at<uint16_t>(ws, layers_s_offset(L)), s);
}

int lora_shrink(const lora_bf16_t *x, int64_t M, const int32_t *lora_id_map, const lora_pool_t *pool,
                const lora_segments_t *segs, float *S, int32_t s_cols, void *ws, size_t ws_bytes,
                lora_stream_t stream)
{
    if (M < 0) return LORA_ERR_SHAPE;
    if (M == 0) return check_pool(pool);
    if (!x || !S) return LORA_ERR_NULL;
    if (!pool) return LORA_ERR_NULL;
    if (!aligned16(x) || !aligned16(S)) return LORA_ERR_ALIGN;
    if (s_cols < std::max(pool->max_rank, 1) || (s_cols % 4)) return LORA_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsLayout L;
    int rc = prepare(lora_id_map, M, pool, segs, ws, ws_bytes, s, &L);
    if (rc) return rc;
    if (cudaMemsetAsync(S, 0, static_cast<size_t>(M) * s_cols * sizeof(float), s) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (pool->num_adapters == 0) return LORA_OK;
    lora_pool_t wpool;   // bf16: S unscaled; e4m3: the widened pool, S times A's factor
    if ((rc = widen_pool(pool, L, ws, kWidenShrink, 0, s, &wpool))) return rc;
    if (pool->adapter_type != LORA_ADAPTER_E4M3) wpool.adapter_scale = nullptr;
    return run_tiled(x, M, nullptr, nullptr, lora_id_map, &wpool, 1.0f, nullptr, ws, ws_bytes, L, kModeShrink, S, s_cols, nullptr, s);
}

int lora_expand(const float *S, int32_t s_cols, int64_t M, const int32_t *lora_id_map, const lora_pool_t *pool,
                const lora_segments_t *segs, float scale, lora_bf16_t *y, void *ws, size_t ws_bytes,
                lora_stream_t stream)
{
    if (M < 0) return LORA_ERR_SHAPE;
    if (M == 0) return check_pool(pool);
    if (!S || !y || !pool) return LORA_ERR_NULL;
    if (pool->adapter_scale && !lora_id_map) return LORA_ERR_NULL;   // the factors are looked up by id
    if (!aligned16(S) || !aligned16(y)) return LORA_ERR_ALIGN;
    if (s_cols < std::max(pool->max_rank, 1)) return LORA_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsLayout L;
    int rc = prepare(lora_id_map, M, pool, segs, ws, ws_bytes, s, &L);
    if (rc) return rc;
    if (pool->num_adapters == 0) return LORA_OK;
    lora_pool_t wpool;   // e4m3: the widened pool, the factor times B's factor
    if ((rc = widen_pool(pool, L, ws, kWidenExpand, 0, s, &wpool))) return rc;
    return run_tiled(nullptr, M, nullptr, nullptr, lora_id_map, &wpool, scale, y, ws, ws_bytes, L, kModeExpand, nullptr, s_cols, S, s);
}

int lora_set_wait_budget(int64_t cycles)
{
    if (cycles < 0) return LORA_ERR_SHAPE;
    g_wait_cycles.store(cycles ? cycles : kDefaultWaitCycles, std::memory_order_relaxed);
    return LORA_OK;
}

int lora_get_status(void *ws, lora_stream_t stream, int32_t *status)
{
    if (!ws || !status) return LORA_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LORA_ERR_CUDA;
    int32_t v = 0;
    int32_t *word = at<int32_t>(ws, 0) + CNT_STATUS;
    if (cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return LORA_ERR_CUDA;
    if (cudaMemset(word, 0, sizeof v) != cudaSuccess) return LORA_ERR_CUDA;
    *status = v;
    return LORA_OK;
}

const char *lora_status_string(int code)
{
    switch (code) {
    case LORA_OK: return "ok";
    case LORA_ERR_NULL: return "a required pointer is NULL";
    case LORA_ERR_SHAPE: return "invalid shape (M < 0, K or N not a positive multiple of 8, too many adapters)";
    case LORA_ERR_ALIGN: return "a tensor base address is not 16-byte aligned";
    case LORA_ERR_RANK: return "a rank outside [1, 128] or max_rank not a multiple of 16";
    case LORA_ERR_WORKSPACE: return "workspace missing or smaller than lora_workspace_size()";
    case LORA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case LORA_ERR_UNSUPPORTED: return "the current device is not an sm_103 (GB300-class) GPU";
    case LORA_ERR_SEGMENTS: return "the segment table was built for another call (M, pool or workspace differ)";
    case LORA_ERR_CAPACITY: return "the problem needs more scratch than lora_linear_noalloc holds (LORA_NOALLOC_SCRATCH_BYTES)";
    case LORA_ERR_ACCESS: return "memory the current device cannot access (pageable host memory or another device's)";
    default: return "unknown status";
    }
}

}  // extern "C"
