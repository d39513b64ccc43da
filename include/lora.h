/*
 * lora.h — C ABI of the GB300 (sm_103a) fused dynamic multi-LoRA linear layer.
 *
 * The layer (page "vLLM-Ascend dynamic LoRA", pptc.cn/news/149022, §1.1, §2.1):
 *
 *     y[t,:] = x[t,:] W^T + bias + (id[t] >= 0 ? scale * (x[t,:] A_id^T) B_id^T : 0)
 *
 * x is hidden_states [M, K], W the base weight [N, K] (nn.Linear layout), bias [N]
 * or none, lora_id_map [M] int32 with -1 meaning "base only" (§2.1), A_i [r_i, K]
 * and B_i [N, r_i] the adapter factors (§1.1), and the result is [M, N].
 * `scale` is one fp32 scalar per call (the page's formula has scale 1).  A
 * pool may also carry one fp32 factor s_i per adapter (for instance the usual
 * alpha_i / r_i); adapter i's delta is then multiplied by scale * s_i.  This
 * per-adapter factor is an extension of this library: the page applies one
 * scale to every adapter, which is the case of a pool without factors.
 *
 * Conventions for every entry point
 *   - Pointers named "device" are CUDA device pointers; "host" ones are host
 *     memory.  Every buffer is owned by the caller; the library never
 *     allocates, frees, synchronises (except lora_get_status) or copies
 *     device->host on the compute entry points.
 *   - bf16 tensors are passed as raw 16-bit patterns (lora_bf16_t), row-major,
 *     16-byte aligned, with K and N multiples of 8 (rows are TMA-addressable).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). All device
 *     work of a call is enqueued on it, in order.
 *   - Return value: LORA_OK, or one of the LORA_ERR_* codes for problems that
 *     are visible on the host (checked before anything is enqueued, so nothing
 *     runs).  Problems found on the device (an id outside [-1, num_adapters),
 *     a bounded wait that gave up) never trap: the kernels finish, treat the
 *     offending token as base-only, and set bits of a status word inside the
 *     workspace that lora_get_status returns.
 *   - Concurrency: two calls that share a workspace must not run at the same
 *     time on the GPU; weights and the pool must not change while a call that
 *     reads them is in flight (§4.3, concurrent adapter replacement).
 */
#ifndef LORA_GB300_LORA_H
#define LORA_GB300_LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lora_bf16_t;   /* raw bfloat16 bits */
typedef void *lora_stream_t;    /* cudaStream_t */

/* Host-side status codes (return values). */
enum {
    LORA_OK = 0,
    LORA_ERR_NULL = 1,          /* a required pointer is NULL */
    LORA_ERR_SHAPE = 2,         /* negative M, K or N not positive multiples of 8, too many adapters */
    LORA_ERR_ALIGN = 3,         /* a tensor base address is not 16-byte aligned (4 for adapter_scale) */
    LORA_ERR_RANK = 4,          /* a rank outside [1, LORA_MAX_RANK], or max_rank not a padded rank */
    LORA_ERR_WORKSPACE = 5,     /* workspace NULL or smaller than lora_workspace_size() */
    LORA_ERR_CUDA = 6,          /* a CUDA runtime call failed (launch error, bad device) */
    LORA_ERR_UNSUPPORTED = 7,   /* device is not sm_103 / sm_100 family or similar */
    LORA_ERR_SEGMENTS = 8,      /* a prebuilt segment table does not match this call */
    LORA_ERR_CAPACITY = 9,      /* the problem needs more scratch than lora_linear_noalloc holds */
    LORA_ERR_ACCESS = 10        /* memory the current device cannot access (pageable host memory,
                                   another device's memory) */
};

/* Device-side status bits (returned through lora_get_status). */
enum {
    LORA_DEV_BAD_ID = 1 << 0,   /* some id was < -1 or >= num_adapters (treated as -1) */
    LORA_DEV_TIMEOUT = 1 << 1,  /* a bounded wait gave up; that call's output is invalid */
    LORA_DEV_BAD_POOL = 1 << 2, /* pool layout the tables cannot describe: a rank not whole panels per
                                   output slice, or a b_offset not whole [N, 16] panels */
    LORA_DEV_CHECK = 1 << 3     /* a segment table failed lora_check_segments, or (library built with
                                   LORA_DEBUG) a kernel met a table-derived index out of range and
                                   skipped that access; the call's output is invalid */
};

#define LORA_MAX_RANK 128       /* largest padded rank */
#define LORA_RANK_ALIGN 16      /* ranks are padded to a multiple of this (§4.3) */
#define LORA_MAX_ADAPTERS 1024  /* largest num_adapters in one pool */
#define LORA_MAX_SLICES 4       /* most output slices of a merged projection */
#define LORA_SLICE_ALIGN 256    /* output slice boundaries are multiples of this */

/*
 * Rank-grouped adapter pool (§2.1: all adapters of one rank stored in one
 * contiguous region, each adapter's start found by a table lookup on its id;
 * §2.2: B arranged at load time in the form the second product consumes;
 * §4.3: ranks padded to a multiple of 16 with zero rows of A / columns of B).
 *
 *   A_i  at a_pool + a_offset[i]: [rank[i], K] row-major bf16
 *        (rows >= true rank are zero).  a_offset[i] is a multiple of K.
 *   B_i  at b_pool + b_offset[i]: rank[i]/16 column panels, panel p being the
 *        [N, 16] row-major block B_i[:, 16p : 16p+16]; element (n, j) of B_i
 *        sits at b_offset[i] + (j/16)*N*16 + n*16 + j%16 (columns >= true rank
 *        are zero).  b_offset[i] is a whole number of [N, 16] panels (a
 *        multiple of 16 N), as lora_pool_layout lays them out.
 * a_pool, b_pool, a_offset, b_offset, rank: DEVICE pointers, caller-owned.
 * adapter_scale: DEVICE fp32 [num_adapters], adapter i's factor s_i on top of
 *        the call's scale (4-byte aligned), or NULL for s_i = 1 everywhere.
 *        Read by lora_linear and lora_expand (lora_shrink returns unscaled
 *        S); a call that reads it needs its lora_id_map even when it is
 *        given a prebuilt segment table.
 * num_slices, slice_start (host values): a merged projection (Q|K|V,
 *        gate|up) whose output columns are cut into num_slices slices
 *        [slice_start[s], slice_start[s+1]), slice_start[0] = 0 and
 *        slice_start[num_slices] = N, inner boundaries multiples of
 *        LORA_SLICE_ALIGN; each adapter then has one A / B pair per slice
 *        with one rank r_i.  The pool holds adapter i as one adapter of
 *        rank num_slices * r_i (r_i padded to 16): A rows [s r_i, (s+1) r_i)
 *        are slice s's A, and B is block-diagonal, B[n, j] = slice s's
 *        B[n - slice_start[s], j - s r_i] for n in slice s and j in
 *        [s r_i, (s+1) r_i), zero elsewhere.  The tiled schedule skips the
 *        zero blocks; the decode-sized schedules read them.  num_slices 0 or
 *        1: one output (slice_start unused).  lora_shrink returns the
 *        stacked S (slice s in columns [s r_i, (s+1) r_i)); lora_expand takes
 *        it in the same form.
 * adapter_type (host value): LORA_ADAPTER_BF16 (0, the layout above) or
 *        LORA_ADAPTER_E4M3: a_pool and b_pool then hold one byte per element,
 *        the 8-bit float e4m3 (1 sign, 4 exponent bits with bias 7, 3
 *        mantissa bits; largest finite 448), in the same layout and at the
 *        same element offsets, and adapter i is A_i = dequant[2i] * A8_i,
 *        B_i = dequant[2i+1] * B8_i.  The 8-bit codes are widened to bf16
 *        exactly (every e4m3 value is a bf16 value); the factors join the
 *        per-adapter factor that scales S before its one bf16 rounding
 *        (lora_shrink applies A's factor, lora_expand B's).  This storage is
 *        an extension of this library; the page stores adapters in the
 *        model's precision.
 * dequant: e4m3 pools: DEVICE fp32 [num_adapters][2] (A factor, B factor).
 * widened: e4m3 pools: DEVICE bf16 scratch of a_elems + b_elems elements
 *        (16-byte aligned).  The decode-sized schedule (M <= 64) reads the
 *        8-bit pool directly; the others (and lora_shrink / lora_expand)
 *        first widen the adapters a batch uses into this scratch, at the
 *        same offsets.  One scratch can serve every pool of a step (sized
 *        for the largest) when the calls run one after another on a
 *        stream.  NULL: those calls return LORA_ERR_NULL.
 * a_elems / b_elems (host values) are the total element counts of the pools;
 * num_adapters, max_rank (largest rank[i]), K and N are host values.
 * lora_pool_layout() computes offsets, padded ranks and sizes for a set of
 * true ranks; filling the pool is the caller's (adapter loader's) job.
 */
typedef struct {
    const lora_bf16_t *a_pool;
    const lora_bf16_t *b_pool;
    const int64_t *a_offset;
    const int64_t *b_offset;
    const int32_t *rank;
    int64_t a_elems;
    int64_t b_elems;
    int32_t num_adapters;
    int32_t max_rank;
    int32_t K;
    int32_t N;
    const float *adapter_scale;
    int32_t num_slices;
    int32_t slice_start[LORA_MAX_SLICES + 1];
    int32_t adapter_type;
    const float *dequant;
    lora_bf16_t *widened;
} lora_pool_t;

#define LORA_ADAPTER_BF16 0
#define LORA_ADAPTER_E4M3 1

/*
 * Segment table (§2.3): a stable bucket sort of the tokens by lora_id.
 * Filled by lora_build_segments with DEVICE pointers into the workspace.
 *   perm[M]            permuted position p -> original token index
 *                      (bucket order: id -1 first, then ascending id; within a
 *                      bucket, ascending token index)
 *   bucket_offsets[A+2] exclusive scan of the bucket counts (bucket 0 = id -1,
 *                      bucket i+1 = adapter i); bucket_offsets[A+1] = M
 *   seg_id/seg_start/seg_len/seg_rank[A]: one entry per adapter present, in
 *                      ascending id: its id, first permuted position, token
 *                      count and padded rank.  Only the first *num_segments
 *                      entries are defined.  Id -1 tokens form no segment.
 *   num_segments[1]
 * The remaining fields are the library's own bookkeeping (the tile work lists
 * that the fused kernels consume); callers pass the struct back unchanged.
 */
typedef struct {
    int32_t *perm;
    int32_t *bucket_offsets;
    int32_t *seg_id;
    int32_t *seg_start;
    int32_t *seg_len;
    int32_t *seg_rank;
    int32_t *num_segments;
    void *plan;                 /* internal: tile / chunk work lists */
    int64_t M;
    int32_t num_adapters;
    int32_t num_slices;         /* output slices of the pool it was built for (>= 1) */
} lora_segments_t;

/*
 * Host helper: rank-grouped pool layout for `num_adapters` adapters with true
 * ranks `true_rank[i]` (host array, each in [1, LORA_MAX_RANK]).  Adapters are
 * grouped by padded rank (16, 32, ..., 128) in that order, keeping id order inside a
 * group.  Writes (host arrays of num_adapters entries) a_offset, b_offset,
 * rank_padded, and *a_elems / *b_elems.  Returns LORA_ERR_RANK / _SHAPE / _NULL.
 */
int lora_pool_layout(int32_t num_adapters, const int32_t *true_rank, int32_t K, int32_t N,
                     int64_t *a_offset, int64_t *b_offset, int32_t *rank_padded,
                     int64_t *a_elems, int64_t *b_elems);

/*
 * Bytes of device workspace needed by every call below for M tokens, output
 * width N and a pool of num_adapters adapters.  The workspace holds the
 * segment table, the tile work lists, the bf16 S scratch, split-K partial sums
 * and a status / counter block; for M > 128 its last 20 MiB hold the partial
 * sums the tiled schedule uses when it splits a mostly empty last wave of
 * tiles along K (with less workspace than this, a call of that size still
 * runs, without the split).  It must be zero-filled once before its first
 * use (lora_workspace_init does that); every call leaves the parts that must
 * start at zero zeroed again.
 */
size_t lora_workspace_size(int64_t M, int32_t N, int32_t num_adapters);

/* Zero-fill a fresh workspace (enqueued on `stream`). ws: DEVICE pointer. */
int lora_workspace_init(void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * §2.3 / §3.2: build the segment table for one step's lora_id_map (DEVICE
 * int32 [M]) against `pool` (its ranks).  One small kernel; *out (HOST
 * struct) receives device pointers into ws.  The table names pool rows in
 * rank rows and whole [N, 16] B panels, so it serves every LoRA layer of the
 * step whose pool holds the same adapters with the same ranks, laid out alike
 * (lora_pool_layout of the same ranks) and sliced alike, whatever the
 * layer's K and N (N <= 65536): pass it with the same workspace, sized with
 * lora_workspace_size for the largest N.  A table that does not fit a call
 * (another M, workspace, adapter count, slicing or workspace layout) is
 * refused with LORA_ERR_SEGMENTS.
 */
int lora_build_segments(const int32_t *lora_id_map, int64_t M, const lora_pool_t *pool,
                        lora_segments_t *out, void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * §2.3 / §2.4: check, on the device, a segment table held in ws against the
 * lora_id_map (DEVICE int32 [M]) and pool it was built for.  One small
 * kernel that writes nothing but the status word: LORA_DEV_CHECK (read with
 * lora_get_status) when the bucket widths differ from the counts of the ids
 * (the segment sums), perm is not the stable order of the tokens by bucket,
 * the segment list is not the adapters present with their starts, lengths
 * and padded ranks, or a tile / chunk work list is out of range.  segs: the
 * table, as lora_build_segments returned it (checked against ws, M and the
 * pool like a prebuilt table: LORA_ERR_SEGMENTS).  M = 0 is a no-op.
 *
 * Debug build: the library compiled with LORA_DEBUG (liblora_debug.so, the
 * same exports) runs this check after every table it builds, and its fused
 * kernels test each table-derived row index before they use it (a bad one
 * sets LORA_DEV_CHECK and the access is skipped).  The normal build has
 * neither cost.
 */
int lora_check_segments(const int32_t *lora_id_map, int64_t M, const lora_pool_t *pool,
                        const lora_segments_t *segs, void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * §2.2 first product alone: S[t, j] = sum_k x[t,k] A_{id[t]}[j,k] for
 * j < rank[id[t]]; S[t, j] = 0 for j >= rank[id[t]] and for id -1 rows.
 * x: DEVICE bf16 [M, pool->K].  S: DEVICE fp32 [M, s_cols], original token
 * order, s_cols >= pool->max_rank (extra columns are zeroed).  segs: a table
 * built for lora_id_map, or NULL to build one in ws first.
 */
int lora_shrink(const lora_bf16_t *x, int64_t M, const int32_t *lora_id_map,
                const lora_pool_t *pool, const lora_segments_t *segs, float *S, int32_t s_cols,
                void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * §2.2 second product alone, added into the output rows (§2.3):
 * y[t, :] += scale * s_id * S[t, :rank] B_{id[t]}^T for id >= 0 (s_id: the
 * pool's per-adapter factor, 1 without one); id -1 rows untouched.
 * S: DEVICE fp32 [M, s_cols] (s_cols >= pool->max_rank), original order.
 * y: DEVICE bf16 [M, pool->N], read and written (rounded once to bf16).
 */
int lora_expand(const float *S, int32_t s_cols, int64_t M, const int32_t *lora_id_map,
                const lora_pool_t *pool, const lora_segments_t *segs, float scale,
                lora_bf16_t *y, void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * The fused layer (§2.1 operator contract, §2.3 one dispatch for all
 * segments): y = x W^T + bias + scale * s_id * (x A_id^T) B_id^T per token
 * (s_id: the pool's per-adapter factor, 1 without one).
 * x: DEVICE bf16 [M, K]; W: DEVICE bf16 [N, K]; bias: DEVICE bf16 [N] or NULL;
 * lora_id_map: DEVICE int32 [M]; y: bf16 [M, N] (written, never read) in
 * device memory or in pinned host memory through its device address
 * (lora_device_pointer): the kernels write y with plain 16-byte stores, which
 * reach host memory over the board's host link.  K and N are taken from the
 * pool.  segs: a table built for lora_id_map and
 * this pool's ranks, or NULL to build one in ws first.  Accumulation is fp32;
 * S is rounded to bf16 once after scaling, the output once at the end.
 * M == 0 is a no-op.  A call whose ids are all -1 runs the base GEMM only.
 */
int lora_linear(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                const int32_t *lora_id_map, const lora_pool_t *pool, float scale,
                const lora_segments_t *segs, lora_bf16_t *y, void *ws, size_t ws_bytes,
                lora_stream_t stream);

/*
 * Several LoRA layers of one step in ONE launch (page "vLLM-Ascend dynamic
 * LoRA", §1.2 end: a model runs many LoRA linears per layer and the
 * per-operator dispatch multiplies; §3.2: one lora_id_map and one segment
 * table per step serve every LoRA layer).  Each layer is
 *     y_l = x_l W_l^T + bias_l + scale_l * s_{l,id} * (x_l A_{l,id}^T) B_{l,id}^T
 * with the step's one lora_id_map; the layers may differ in K, N, weights,
 * inputs, outputs, scale, factors and slice boundaries, but their pools must
 * hold the same adapters with the same ranks, laid out alike (lora_pool_layout
 * of the same true ranks, each for its own K and N) and cut into the same
 * number of output slices.  The host checks what it can see of that (adapter
 * count, max_rank, pool row and panel counts, slice count) and returns
 * LORA_ERR_SHAPE otherwise.
 *
 * The tiled tensor-core schedule runs all layers in one persistent launch:
 * its work list holds every layer's shrink jobs, then every layer's output
 * tiles, so one layer's last partial wave overlaps the next layer's tiles.
 * Without a prebuilt table a segment build launch goes first, as for
 * lora_linear.
 *
 * layers: HOST array of num_layers (1..LORA_MAX_LAYERS) descriptors.
 * lora_id_map: DEVICE int32 [M] (needed unless segs is given and no pool
 * has per-adapter factors).  segs: a table built by lora_build_segments
 * for layer 0's pool in this ws, or NULL.  ws: DEVICE, at least
 * lora_layers_workspace_size(M, largest N, num_adapters, num_layers) bytes,
 * zero-filled once (lora_workspace_init); it also holds the table.
 * Accumulation and rounding as for lora_linear; M == 0 is a no-op.
 */
#define LORA_MAX_LAYERS 8
typedef struct {
    const lora_bf16_t *x;       /* DEVICE bf16 [M, pool->K] */
    const lora_bf16_t *W;       /* DEVICE bf16 [pool->N, pool->K] */
    const lora_bf16_t *bias;    /* DEVICE bf16 [pool->N] or NULL */
    const lora_pool_t *pool;    /* HOST descriptor of the layer's adapter pool */
    float scale;                /* the layer's LoRA scale */
    lora_bf16_t *y;             /* DEVICE bf16 [M, pool->N], written */
} lora_layer_t;

size_t lora_layers_workspace_size(int64_t M, int32_t max_N, int32_t num_adapters, int32_t num_layers);
int lora_linear_layers(const lora_layer_t *layers, int32_t num_layers, int64_t M, const int32_t *lora_id_map,
                       const lora_segments_t *segs, void *ws, size_t ws_bytes, lora_stream_t stream);

/* Schedules of lora_linear_ex (the automatic choice picks by M). */
enum {
    LORA_PATH_AUTO = 0,
    LORA_PATH_TILED = 1,        /* token-tile x output-tile persistent schedule */
    LORA_PATH_SPLITK = 2,       /* weight-streaming split-K schedule, M <= 128 */
    LORA_PATH_STREAM = 3        /* weight-streaming cluster schedule, M <= 64, K % 64 == 0 */
};

/*
 * Flags OR-ed into lora_linear_ex's `path` argument.
 *
 * LORA_FLAG_STATIC_WEIGHTS: W, bias and the adapter pool (A, B, offsets,
 * ranks, factors) are not written by any kernel that can still be running
 * when the call starts, i.e. by no kernel enqueued on `stream` since its last
 * operation that is not a kernel launch (a copy, a memset, an event wait).
 * Weights loaded once by copies and left alone during the steps qualify.
 * The call may then start streaming weights before the kernel ahead of it on
 * the stream has finished (a programmatic dependent launch); x, the ids, the
 * workspace and y are still touched only after that kernel completes.  Today
 * the decode-sized schedule (M <= 64) uses it; the others ignore it.
 */
#define LORA_FLAG_STATIC_WEIGHTS 0x100

/* lora_linear with an explicit schedule (for tests and tuning); `path` is a
 * LORA_PATH_* value, optionally OR-ed with LORA_FLAG_* bits. */
int lora_linear_ex(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                   const int32_t *lora_id_map, const lora_pool_t *pool, float scale,
                   const lora_segments_t *segs, lora_bf16_t *y, void *ws, size_t ws_bytes,
                   lora_stream_t stream, int32_t path);

/*
 * lora_linear without a workspace, for callers that cannot allocate device
 * memory: an inference-engine hook or plugin that is handed no workspace and
 * may not call cudaMalloc while it runs, for example.  The paper this library
 * follows (the page "vLLM-Ascend dynamic LoRA") has no counterpart to this
 * entry point; it is a convenience of this library.
 *
 * Same arguments, layouts and result as lora_linear (segments are always
 * built internally).  The scratch is a file-scope device array of
 * LORA_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits; nothing is allocated or
 * freed.  The call returns LORA_ERR_CAPACITY and enqueues nothing when the
 * minimal workspace layout of (M, pool->N, pool->num_adapters) is larger
 * than the array.  That minimal layout is lora_workspace_size() without the
 * tiled schedule's optional 20 MiB split-tile scratch, which never fits: a
 * call with M > 128 therefore runs the tiled schedule without splitting a
 * partial last wave along K.  Every workload of up to 8192 tokens, N = 4096
 * and 32 adapters fits (about 3 MiB).
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array, which keeps the previous call's
 * contents: each call first clears (with cudaMemsetAsync on `stream`) the
 * parts that must start at zero, the status word included.  Calls whose
 * execution overlaps on the GPU (other streams, other host threads) race on
 * the array and must be avoided.  Device-detected problems (bad ids) are
 * handled as in lora_linear, but the status word is cleared by the next call
 * and cannot be read through this entry point.
 */
#define LORA_NOALLOC_SCRATCH_BYTES (8u << 20)   /* 8 MiB */
int lora_linear_noalloc(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                        const int32_t *lora_id_map, const lora_pool_t *pool, float scale, lora_bf16_t *y,
                        lora_stream_t stream);

/*
 * Mixture of experts (the page "Qwen3-MoE low-latency inference on Atlas A3",
 * mokono.cn/news/2297686, its MoE section: route the tokens to their
 * experts, one grouped matmul over all experts, then put the rows back and
 * sum them with the routing weights).  Not a LoRA layer: a stable bucket sort
 * of the pairs like the segment build (two launches over chunks of the
 * pairs) and the tiled tensor-core kernel serve it.
 *
 *   y[t, :] = sum_{j < topk, e = expert[t, j] in [0, E)} weight[t, j] * x[t, :] W_e^T
 *
 * x: DEVICE bf16 [M, K]; W: DEVICE bf16 [E, N, K] (each expert's weight in
 * nn.Linear layout, stacked); expert: DEVICE int32 [M, topk] (ids outside
 * [0, E) contribute nothing); weight: DEVICE fp32 [M, topk]; out: DEVICE
 * bf16 [M * topk, N], each (token, slot) pair's expert row x[t] W_e^T in pair
 * order (rows of invalid pairs are not written); y: DEVICE bf16 [M, N].
 * K and N multiples of 8, 1 <= topk <= E <= LORA_MAX_ADAPTERS.  ws: DEVICE,
 * at least lora_moe_workspace_size(M, topk, E) bytes, zero-filled once before
 * its first use (lora_workspace_init) so that its status word starts clear;
 * the routing resets everything else it needs on every call.
 *   lora_moe_route:    the stable sort of the pairs by expert (segment
 *                      table over the pairs) and the padded expert order
 *   lora_moe_gemm:     the grouped GEMM over the routed pairs (needs the
 *                      routing of the same expert ids in ws)
 *   lora_moe_finalize: the weighted sum of each token's rows
 *   lora_moe:          the three in order
 *   lora_moe_check_route: a device check of the routing in ws against the
 *                      expert ids it was made from (bucket widths, perm
 *                      stable and complete, the segment table, the padded
 *                      order and each tile's expert): LORA_DEV_CHECK when
 *                      they disagree.  The LORA_DEBUG build runs it after
 *                      every routing, and its grouped GEMM leaves its work
 *                      list empty on a routing that failed.
 * Errors as for the other entry points.
 */
size_t lora_moe_workspace_size(int64_t M, int32_t topk, int32_t num_experts);
int lora_moe_route(const int32_t *expert, int64_t M, int32_t topk, int32_t num_experts, void *ws, size_t ws_bytes,
                   lora_stream_t stream);
int lora_moe_check_route(const int32_t *expert, int64_t M, int32_t topk, int32_t num_experts, void *ws,
                         size_t ws_bytes, lora_stream_t stream);
int lora_moe_gemm(const lora_bf16_t *x, int64_t M, int32_t K, const lora_bf16_t *W, int32_t N, int32_t num_experts,
                  int32_t topk, lora_bf16_t *out, void *ws, size_t ws_bytes, lora_stream_t stream);
int lora_moe_finalize(const lora_bf16_t *out, const int32_t *expert, const float *weight, int64_t M, int32_t topk,
                      int32_t num_experts, int32_t N, lora_bf16_t *y, lora_stream_t stream);
int lora_moe(const lora_bf16_t *x, int64_t M, int32_t K, const lora_bf16_t *W, int32_t N, const int32_t *expert,
             const float *weight, int32_t num_experts, int32_t topk, lora_bf16_t *out, lora_bf16_t *y, void *ws,
             size_t ws_bytes, lora_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the device status word of ws
 * into *status (a bitwise OR of LORA_DEV_* since the last read).
 */
int lora_get_status(void *ws, lora_stream_t stream, int32_t *status);

/*
 * Test knob for the bounded waits of the tiled schedule's kernel (the one
 * lora_linear runs for M > 128, lora_linear_layers, lora_shrink and
 * lora_expand use), of lora_moe_gemm's grouped expert kernel and of the
 * split-K schedule's (64 < M <= 128): each wait gives up after `cycles` SM
 * clock cycles, sets
 * LORA_DEV_TIMEOUT and lets the kernel run to its end.
 * cycles = 0 restores the default (2e9 cycles, about one second).  A budget
 * shorter than a healthy wait reports timeouts on healthy calls, so this is
 * for exercising the timeout path, not for production.  Process-wide; read
 * when a call is enqueued.  Returns LORA_ERR_SHAPE for cycles < 0.  The
 * method has no counterpart: it is part of this library's failure detection.
 */
int lora_set_wait_budget(int64_t cycles);

/*
 * Moving a step's inputs and outputs across the host link with the SMs.
 *
 * lora_device_pointer: the address a kernel on the current device uses for
 * ptr.  That is ptr itself for this device's memory or managed memory, and
 * the mapped alias for pinned host memory.  Returns LORA_ERR_ACCESS for
 * pageable host memory, another device's memory or an unknown pointer, and
 * LORA_ERR_NULL for a NULL argument.
 *
 * lora_copy_async: copies n <= LORA_MAX_COPIES buffers (dst[i] <- src[i],
 * bytes[i] each) in one small kernel on `stream`: each side may be device
 * memory or pinned host memory (given by its host address), so a step's
 * host-to-device inputs move without a copy-engine transfer.  Addresses and
 * sizes must be multiples of 16 bytes (LORA_ERR_ALIGN), sizes >= 0
 * (LORA_ERR_SHAPE); a zero-byte entry is skipped; LORA_ERR_ACCESS as above.
 * The kernel is a programmatic dependent launch: it starts while the kernel
 * ahead of it finishes, waits for that kernel (griddepcontrol.wait) before
 * it reads or writes any byte, and lets the launch behind it start its
 * prologue at once.  Buffers must not overlap.  The copy is ordered on
 * `stream` like any kernel; the host sees a host-side destination once the
 * stream has been synchronised.  This is plumbing around the layer, not a
 * step of the method.
 */
#define LORA_MAX_COPIES 4
typedef struct {
    void *dst;
    const void *src;
    int64_t bytes;
} lora_copy_t;

int lora_device_pointer(const void *ptr, void **dev_ptr);
int lora_copy_async(const lora_copy_t *copies, int32_t n, lora_stream_t stream);

/* Static text for a LORA_ERR_* code. */
const char *lora_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* LORA_GB300_LORA_H */
