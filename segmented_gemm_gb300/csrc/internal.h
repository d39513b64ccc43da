// Internal declarations shared by the host API and the kernels of liblora.
//
// Workspace layout (all offsets 256-byte aligned), for M tokens, N outputs and
// A adapters:
//   counters   status word, grid counters, per-token-tile S-ready flags,
//              per-output-tile split-K arrival counters   (zero at rest)
//   segments   perm[M], bucket_offsets[A+2], seg_{id,start,len,rank}[A],
//              num_segments[1]                             (the §2.3 table)
//   plan       header, per-tile chunk lists, shrink-job list, split-K chunk
//              list                                        (kernel work lists)
//   windows    stream schedule: window list, per-window arrival and consumer
//              counters (zero at rest), fp32 window sums of S (zero at rest)
//   s_scratch  bf16 S panels (scaled, masked), [chunks][rows][16]
//   acc        fp32 split-K tile accumulators (zero at rest)
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "lora.h"

namespace lora {

// ---- tiled (token-tile x output-tile) schedule -----------------------------
constexpr int kBM = 128;          // permuted tokens per tile (UMMA M)
constexpr int kBN = 256;          // output features per tile (UMMA N)
constexpr int kBK = 64;           // K per stage (one 128-byte swizzle row)
constexpr int kChunk = 16;        // rank columns per chunk (one UMMA K step)
constexpr int kMaxShrinkChunks = 16;   // chunks per shrink job -> N <= 256

// ---- split-K (weight streaming) schedule ----------------------------------
constexpr int kSplitMaxTokens = 128;   // largest M served by the split-K path
constexpr int kSplitBN = 128;          // output features per tile (UMMA M)
constexpr int kSplitMaxCtas = 1024;    // upper bound on the persistent grid
constexpr int kStreamMaxTokens = 64;    // largest M served by the weight-streaming schedule
constexpr int kWinCntStride = 32;       // ints per window counter pair (one 128-byte line)
constexpr int kStreamKMaxTiles = 160;   // output tiles the tiled schedule may split along K in one call
constexpr int64_t kMaxTokens = (int64_t(1) << 31) - kBM;   // largest M of one call (32-bit row indices)

// plan header entries
enum PlanHdr {
    HDR_NCHUNKS = 0,      // chunks of the tiled schedule (all tiles)
    HDR_NSJOBS = 1,       // shrink jobs of the tiled schedule
    HDR_DCHUNKS = 2,      // chunks of the split-K schedule (adapters present)
    HDR_NSEG = 3,         // number of segments
    HDR_MOE_TILES = 4,    // routing: 128-row tiles of the padded expert order
    HDR_CHECK = 5,        // the table checker's verdict on this table: 0 consistent, 1 not
    HDR_WORDS = 16
};

// counter block entries (int32), zero between calls
enum Counters {
    CNT_STATUS = 0,       // LORA_DEV_* bits
    CNT_SPLIT_DONE = 2,   // split-K: CTAs finished
    CNT_SPLIT_SREADY = 3, // split-K: shrink row tiles reduced
    CNT_FIXED = 8         // first per-tile counter
};

// long budget of the tiled and split-K kernels' bounded waits (SM clock
// cycles), set by lora_set_wait_budget; read when a launch is enqueued
constexpr int64_t kDefaultWaitCycles = 2000000000ll;
int64_t tc_wait_cycles();

// Checks compiled into the LORA_DEBUG build only: an index that a kernel
// derives from the segment table is tested before it is used; a bad one
// sets LORA_DEV_CHECK and the access is skipped.  In the normal build the
// condition is not evaluated.
#ifdef LORA_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
__device__ __forceinline__ bool debug_index_ok(bool ok, int32_t *status)
{
    if (!ok) atomicOr(status, LORA_DEV_CHECK);
    return ok;
}

struct WsLayout {
    int64_t M;
    int32_t N, A;
    int32_t num_mtiles;       // ceil(M / kBM)
    int32_t max_chunks;       // tiled-schedule chunk capacity
    int32_t max_sjobs;        // shrink-job capacity
    int32_t max_dchunks;      // split-K chunk capacity
    int32_t split_tiles;      // split-K output + shrink tiles (counter slots)
    size_t counters, n_counters;
    size_t perm, offsets, seg_id, seg_start, seg_len, seg_rank, num_segments;
    size_t hdr, tile_chunk_off, chunk_arow, chunk_bpanel, chunk_rng;
    size_t sjob_tile, sjob_c0, sjob_c1, tile_njobs;
    size_t dchunk_arow, dchunk_bpanel, dchunk_adapter;
    size_t wcnt, acc_str, acc_str_bytes;
    int32_t max_win_str;      // windows the stream schedule's sums and counters can hold (M <= 64)
    size_t s_scratch, s_scratch_bytes;
    size_t acc_out, acc_out_bytes, acc_shr, acc_shr_bytes;
    size_t fac;               // e4m3 pools: each layer's per-adapter factors for a call, fp32 [kMaxLayers][A]
    size_t total_min;         // everything but the stream-K scratch
    size_t sk_part, sk_cnt;   // stream-K partial sums / counters of the tiled schedule (M > 128)
    size_t total;
};

// Host: compute the layout for (M, N, A); M <= kMaxTokens and
// A <= LORA_MAX_ADAPTERS (callers check both first).
WsLayout make_ws_layout(int64_t M, int32_t N, int32_t A);
// Host: validate a pool descriptor (LORA_OK or a LORA_ERR_* code).
int check_pool(const lora_pool_t *pool);

// chunk_rng packing: rows [lo, hi) of the tile, rank panel p of the segment
__host__ __device__ inline int32_t pack_rng(int lo, int hi, int p) { return lo | (hi << 8) | (p << 16); }
// S panel sets the workspace holds for the tiled schedule: a shrink job is
// split into two K halves (one set each) only for M > 128
inline int tiled_s_sets(int64_t M) { return M > kSplitMaxTokens ? 2 : 1; }
__host__ __device__ inline int rng_lo(int32_t v) { return v & 0xFF; }
__host__ __device__ inline int rng_hi(int32_t v) { return (v >> 8) & 0xFF; }
__host__ __device__ inline int rng_panel(int32_t v) { return (v >> 16) & 0xFF; }

// ---- kernel parameter blocks ----------------------------------------------
// kModeMoe: grouped expert GEMMs of a mixture-of-experts layer, over the
// routing's padded expert order (perm = perm_pad; output rows are pairs)
enum TcMode { kModeLinear = 0, kModeShrink = 1, kModeExpand = 2, kModeMoe = 3 };

struct TcMaps {
    CUtensorMap x, w, a, b, s;
    CUtensorMap a32, a48, a64;   // A pool with 32 / 48 / 64-row boxes (a: 16 rows)
};

// One layer of a tiled launch.  A launch covers up to kMaxLayers layers that
// share one segment table (the same M, ids, adapters, ranks and slicing;
// each its own K, N, weights and output); its work list runs every layer's
// shrink items, then every layer's output tiles.
constexpr int kMaxLayers = LORA_MAX_LAYERS;
struct TcLayer {
    int32_t N, K, kblocks, num_ntiles;
    int32_t slice_start[LORA_MAX_SLICES + 1];   // first output column of each slice
    float scale;
    const float *adapter_scale;   // per-adapter factor on top of scale, or null (all 1)
    const uint16_t *bias;      // bf16 [N] or null
    const uint16_t *x;         // bf16 [M, K] (rows gathered by the loader warps)
    uint16_t *y;               // bf16 [M, N]
    int32_t tile0;             // the layer's first output tile in the launch's list of output tiles
};

struct TcLayerMaps {
    CUtensorMap x, w, a, b;
    CUtensorMap a32, a48, a64;   // A pool with 32 / 48 / 64-row boxes (a: 16 rows)
};

struct TcParams {
    int64_t M;
    int32_t num_mtiles, group_m, mode, s_cols;
    int32_t num_adapters;
    int32_t num_slices;        // output slices (>= 1); tile_chunk_off holds [tiles][slices] + 1 offsets
    int32_t num_layers;        // layers of this launch (1..kMaxLayers)
    const int32_t *ids;        // lora_id_map (original token order); read when adapter_scale is set
    int32_t topk;              // kModeMoe: pairs per token (a pair's token is pair / topk)
    int64_t out_rows;          // rows a perm entry may name: M (kModeMoe: the pairs, M * topk)
    const int32_t *mt_expert;  // kModeMoe: the expert of each 128-row tile of the padded order
    uint16_t *s_panels;        // bf16 [layers][sets][chunks][128][16]
    float *s_out;              // fp32 [M, s_cols] (shrink mode)
    const int32_t *perm, *offsets, *hdr;
    const int32_t *tile_chunk_off, *chunk_arow, *chunk_bpanel, *chunk_rng;
    const int32_t *sjob_tile, *sjob_c0, *sjob_c1, *tile_njobs;
    int32_t *counters;         // S-ready counters [layers][tiles] at CNT_FIXED, their consumers after them
    int32_t streamk;           // split the last partial wave of output tiles along K (one layer only)
    int32_t shrink_split;      // K pieces per shrink job; piece h writes S panel set h
    int32_t s_sets;            // S panel sets the expand steps add up (shrink_split, or 1 for expand)
    int32_t s_set_rows;        // rows of one S panel set (chunks x 128)
    float *sk_part;            // fp32 [CTAs][256/4][128][4]: each tail piece's partial sums, in its CTA's slot
    int32_t *sk_cnt;           // [tiles][kWinCntStride]: tail pieces stored per split tile (zero at rest)
    int64_t wait_cycles;       // long budget of the kernel's bounded waits, in SM clock cycles
    TcLayer layer[kMaxLayers];
};

// Everything a tiled launch takes: each layer's tensor maps, the map of the
// S panel scratch and the parameters (one __grid_constant__ argument).
struct TcArgs {
    TcLayerMaps maps[kMaxLayers];
    CUtensorMap s;
    TcParams p;
};

struct SplitParams {
    int64_t M;
    int32_t N, K, T_pad, kblocks, NT, stages, tmem_cols, A;
    float scale;
    const float *adapter_scale;   // per-adapter factor on top of scale, or null (all 1)
    const uint16_t *bias;
    uint16_t *y;
    const int32_t *ids, *hdr, *dchunk_arow, *dchunk_bpanel, *dchunk_adapter;
    uint16_t *s_panels;        // bf16 [chunks][T_pad][16]
    float *acc_out;            // fp32 [NT][128][T_pad], zero at rest
    float *acc_shr;            // fp32 [shrink tiles][128][T_pad], zero at rest
    int32_t *counters;
    int64_t wait_cycles;       // long budget of the kernel's bounded waits, in SM clock cycles
};

struct SegParams {
    const int32_t *ids;
    int64_t M;
    int32_t A, K, N, num_mtiles;
    const int32_t *rank;
    const int64_t *a_offset;
    const int64_t *b_offset;
    int32_t *perm, *offsets, *seg_id, *seg_start, *seg_len, *seg_rank, *num_segments;
    int32_t *hdr, *tile_chunk_off, *chunk_arow, *chunk_bpanel, *chunk_rng;
    int32_t *sjob_tile, *sjob_c0, *sjob_c1, *tile_njobs;
    int32_t *dchunk_arow, *dchunk_bpanel, *dchunk_adapter;
    int32_t *counters;
    int32_t n_counters;
    int32_t num_slices;        // output slices of a merged projection (>= 1): tile chunk lists are slice-major
};

// The table checker (seg_check.cu): the builder's parameters plus the
// workspace's capacities and the pool's extent.
struct SegCheckParams {
    SegParams s;
    int32_t max_chunks, max_sjobs, max_dchunks;
    int64_t a_rows;            // rows of the A pool (a_elems / K)
    int64_t b_panels;          // [N, 16] panels of the B pool (b_elems / (16 N))
};

// Mixture-of-experts routing: the (token, slot) pairs sorted stably by
// expert (bucket 0: invalid ids, bucket e + 1: expert e), and each expert's
// pairs laid out from a fresh 128-row tile of the padded order.
constexpr int kRouteMaxChunks = 256;   // pair chunks (CTAs) of the routing, at most
struct RouteParams {
    const int32_t *expert;     // [P] each pair's expert
    int64_t P;                 // pairs
    int32_t E, nb;             // experts, buckets (E + 1)
    int32_t chunk, nchunks;    // pairs per CTA (a multiple of 256), CTAs
    int32_t max_mtiles;        // 128-row tiles the padded order has room for
    int32_t n_counters;
    int32_t *cnt;              // [nchunks][nb] bucket counts of each chunk
    int32_t *perm, *offsets, *seg_id, *seg_start, *seg_len, *seg_rank, *num_segments, *hdr, *counters;
    int32_t *perm_pad;         // [max_mtiles * 128] pair of each padded row, -1 in the gaps
    int32_t *mt_expert;        // [max_mtiles] expert of each tile, -1 past the last
};

struct ClusterMaps {
    CUtensorMap w3, a3, b3;    // W, A pool: {64, 128 rows, 2 K blocks}; B pool: {16, 128 rows, 8 panels}
    CUtensorMap x3;            // x: {64, T rows, 2 K blocks} (rows past M read as zeros)
};

struct ClusterParams {
    int64_t M;
    int32_t N, K, T_pad, C, NT, kblocks, stages, max_regions, max_win_str;
    int32_t s_ring;            // S operand slots of the expand windows (2..4)
    int32_t fp8;               // e4m3 pool: A and B boxes arrive as 8-bit codes and are widened in the kernel
    const float *dequant;      // e4m3 pool: [A][2] dequant factors of A and B
    float scale;
    const float *adapter_scale;   // per-adapter factor on top of scale, or null (all 1)
    const uint16_t *bias;
    const uint16_t *x;         // bf16 [M, K] (read through the x tensor map)
    uint16_t *y;
    const int32_t *ids;
    const int64_t *a_offset;   // the pool table (device): first A pool element of each adapter
    const int32_t *rank;       // padded rank of each adapter
    int32_t A, windows_all;    // adapters; 128-row windows in the pool
    int32_t all_windows;       // process every window (known at launch) instead of the ones the batch touches
    int32_t early_weights;     // launched as a programmatic dependent: weights are read before griddepcontrol.wait
    int32_t build;             // one extra cluster, whose first CTA builds the segment table (seg)
    SegParams seg;
    float *acc;                // fp32 [windows][T_pad][128]: per-window sums of S (zero at rest)
    int32_t *wcnt;             // [windows][kWinCntStride]: shrink arrivals at 0, consumer CTAs at 16 (zero at rest)
    int32_t *counters;
};


// e4m3 pools: widening the adapters a batch uses into the pool's bf16
// scratch (same offsets) and the call's per-adapter factors
enum WidenMode { kWidenFused = 0, kWidenShrink = 1, kWidenExpand = 2 };
struct WidenParams {
    const uint8_t *a8, *b8;    // the e4m3 pools
    uint16_t *aw, *bw;         // their bf16 twins in the scratch
    const int64_t *a_off, *b_off;
    const int32_t *rank;
    int32_t K, N, A, parts, mode;
    const int32_t *seg_id, *num_segments;   // the batch's segment table
    const float *dequant, *adapter_scale;
    float *fac;                // fused: s_i da_i db_i; shrink: da_i; expand: s_i db_i
};

// ---- launchers (enqueue only; return the launch status) --------------------
cudaError_t launch_widen(const WidenParams &p, int max_segments, cudaStream_t stream);
cudaError_t launch_seg_build(const SegParams &p, bool pdl, cudaStream_t stream);
cudaError_t launch_seg_check(const SegCheckParams &q, cudaStream_t stream);
cudaError_t launch_moe_route_check(const RouteParams &p, cudaStream_t stream);
cudaError_t launch_moe_route(const RouteParams &p, cudaStream_t stream);
cudaError_t launch_tc(const TcArgs &args, int grid, cudaStream_t stream);
cudaError_t launch_moe_finalize(const uint16_t *out, const int32_t *expert, const float *weight, int64_t M, int topk,
                                int E, int N, uint16_t *y, cudaStream_t stream);
cudaError_t launch_s_prep(const float *S, int32_t s_cols, float scale, const TcParams &p, cudaStream_t stream);
cudaError_t launch_splitk(const TcMaps &maps, const SplitParams &p, int grid, cudaStream_t stream);
int splitk_stages(int T_pad);
cudaError_t launch_cluster(const ClusterMaps &m, const ClusterParams &p, bool pdl, cudaStream_t stream);
int cluster_pick_size(int NT, int T_pad, int sms);
int cluster_stages(int T_pad);
size_t cluster_smem_bytes(int T_pad, int stages, int s_ring);
int cluster_s_ring(int T_pad, int stages);
size_t cluster_build_smem_bytes(int32_t A);   // the segment build inside the decode kernel
int cluster_max_regions();
int cluster_max_runs();
int cluster_max_win_cta();
int cluster_win();
int splitk_max_runs();
int num_sms_current_device();

}  // namespace lora
