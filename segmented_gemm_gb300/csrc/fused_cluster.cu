// Weight-streaming schedule of the fused multi-LoRA linear layer for
// decode-sized batches (M <= 64 tokens).
//
// Page "vLLM-Ascend dynamic LoRA" (pptc.cn/news/149022): §1.2 (a decode step
// has one token per sequence, so the layer is bound by reading the weights
// once), §4.2 #3 (the adapters of a step handled as one concatenated block
// rather than one small GEMM each), §2.2 (S = x A^T first, then S B^T into
// the same output), §2.3 (one dispatch for all segments).
//
// The MMA is swapped: 128 weight rows are the UMMA A operand (M = 128), the
// zero-padded tokens (16..64) its N side.  Each 128-feature output tile is
// owned by one thread-block cluster of C CTAs; CTA q streams the q-th part
// of K.  Every operand the tensor cores read arrives as a 32 KB box:
//   - base units: 128 rows of W x 2 K blocks;
//   - shrink units: 128 rows of the concatenated A pool x 2 K blocks.  The
//     pools are cut into windows of 8 rank panels (128 pool rows); only
//     windows that hold a panel of an adapter present are visited.  The
//     window x K-unit list is sliced evenly over the whole grid; each CTA
//     adds its fp32 partial S of a window to the window's sum in L2 with
//     atomics and releases the window's arrival counter;
//   - expand units: one window of the B pool (8 panels x this tile's 128
//     output rows) through the ring; the N operand is the window's S, which
//     the loader warps stage in a small ring of their own: as soon as the
//     window's sum is complete (early: every CTA shrinks first) they read
//     it, keep for each token only the panels of its own adapter, scale and
//     round it to bf16, while the weight stream goes on.
// Order inside a CTA: the first units of its K part (issued before any
// metadata is read, and, when the kernel follows the segment builder, before
// the builder has finished), its shrink slice, the rest of its K part, its
// share of the expand windows.  The last CTA to consume a window clears the
// window's sum and counters, so they are zero again when the call ends; the
// loaders count their reads right after staging, so this also happens while
// the weights still stream.
// The C partial tiles are then pushed with st.async into the CTA that owns
// each 128/C-row slice (distributed shared memory, mbarrier byte counting);
// the owner sums them, adds the bias and writes y.
// Roles (320 threads): warp 0 TMA producer (the weight box and the x box of
// each unit, B windows), warp 1 TMEM allocator + MMA issuer, warps 2..5
// epilogue (warp 2 also derives the metadata, warp 3 pulls the B windows
// into L2 as soon as they are known), warps 6..9 stage the S
// operand of the expand units (load-convert-store into the S ring).  All waits are bounded;
// the host only launches the grid when every cluster can be resident at once.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"
#include "seg_build_body.cuh"

namespace lora {

constexpr int kClThreads = 320;
constexpr int kClWArea = 32 * 1024;        // one W / A / B box
constexpr int kClMisc = 8192;              // barriers, segment list, window tables, bias
constexpr int kStMaxWinAll = 512;          // windows of the pool (bitmap of 16 words)
constexpr int kStMaxWinList = 2 * kStreamMaxTokens;   // windows a batch can touch
constexpr int kClMaxStages = 8;
constexpr int kClMaxSRing = 4;             // S operand slots of the expand windows (one window each)
constexpr int kFp8Box = 16 * 1024;         // an e4m3 A or B box; it lands in the upper half of the weight area
constexpr int kBarConv = 11;               // named barrier: the epilogue warps' loads of an e4m3 B box are done
constexpr int kStMaxSegs = 8;
constexpr int kStMaxRegions = 16;
constexpr int kStMaxRuns = 4;              // shrink runs (windows) of one CTA
constexpr int kStWin = 8;                  // rank panels per window
constexpr int kStMaxWinCta = 64;           // expand windows of one CTA
constexpr int kBarMeta = 1;                // named barrier: metadata ready (the producer and the epilogue warps)
constexpr int kBarMma = 2;                 // named barrier: metadata ready (MMA issuer + warp 2)
constexpr int kBarLoad = 3;                // named barrier: the four loader warps
constexpr int kBarEpi = 4;                 // named barrier: the four epilogue warps
constexpr int kBarTmem = 6;                // named barrier: TMEM allocated (warps 0..5; the loaders never read it)
constexpr int kBarTables = 7;              // named barrier: expand windows ready (table warp -> producer, MMA)
constexpr int kBarTablesEpi = 8;           // named barrier: panel tables ready (warp 2 -> the other epilogue warps)
constexpr int kTablesThreads = 96;         // warps 0, 1 and the table warp (2, or 6 when every window is processed)
constexpr int kBarTablesLd = 9;            // named barrier: panel tables ready (warp 2 -> loaders)
constexpr int kTablesLdThreads = 160;      // warp 2 + warps 6..9
constexpr int kBarTouch = 10;              // named barrier: expand windows' touched flags (warp 6 -> epilogue)
constexpr int kStFirst = 3;                // K units issued before the metadata is known
constexpr int kMetaThreads = 160;   // warps 0 and 2..5 (the loaders learn of the plan through kBarTablesLd)

enum StKind { kStBase = 0, kStShrink = 1, kStExpand = 2 };

struct StSeg {
    int kind;     // StKind
    int a, b;     // base: K units [a, b); shrink: K units [a, b) of window w; expand: windows [a, b)
    int w;        // shrink: window index in the list of present windows
    int region;   // TMEM accumulator: 0 the output tile, 1.. shrink runs
    int arow;     // shrink: first A pool row of the window
};

// the barriers and tables that follow the reduction area fit kClMisc bytes
static_assert((4 * kClMaxStages + kStMaxRegions + 1 + 2 * kClMaxSRing) * 8 + 10 * 4 + kSplitBN * 2 + 64 * 4 * 2 +
                      kStMaxSegs * static_cast<int>(sizeof(StSeg)) + kStMaxWinCta * 4 * 3 + kStMaxWinCta * kStWin * 4 +
                      kStMaxRuns * kStWin * 4 + (kStMaxWinAll / 32) * 4 * 2 + kStMaxWinList * 4 +
                      kStMaxWinCta * kStWin * 4 + kStMaxWinCta * 4 <=
                  kClMisc,
              "cluster kernel tables overflow their shared-memory area");

// Pull one box of a 3-D tensor map into L2 (no shared-memory destination,
// nothing to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *m, int x, int y, int z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(m), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_load_3d_st(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y, int z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(m), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, float4 v, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_addr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
// Arrive without release semantics: used once the barriers a peer will
// touch have been published with fence.mbarrier_init (a release arrive
// would also wait for this thread's outstanding memory operations).
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Unit list of one CTA before its expand windows.  Shrink runs are the
// CTA's slice of the (window, K unit) list of the whole grid; a shrunk
// window is named by its index w in the list of windows shrunk (s_wlist
// maps it to a pool window, identity when every window is shrunk).  With
// shrink_first the order is [shrink runs][base], else [first base units]
// [shrink runs][rest of base].  Written to segs when write.
struct SegPlan {
    int n, nruns;
    int run_w[kStMaxRuns];
    bool ok;
};

__device__ __forceinline__ SegPlan plan_segments(StSeg *segs, bool write, int NW, int KU2, int G, int cta, int b0,
                                                 int b1, int nbase_first, int max_regions, const int *s_wlist,
                                                 bool shrink_first)
{
    SegPlan r;
    int n = 0, region = 1;
    r.nruns = 0;
    r.ok = true;
    for (int i = 0; i < kStMaxRuns; ++i) r.run_w[i] = -1;
    if (!shrink_first) {
        if (write) segs[n] = {kStBase, b0, b0 + nbase_first, 0, 0, 0};
        ++n;
    }
    const int U = NW * KU2;   // the host keeps NW x KU2 x G below 2^31
    for (int u = (U * cta) / G, u1 = (U * (cta + 1)) / G; u < u1;) {
        const int wi = u / KU2;
        const int e = min(u1, (wi + 1) * KU2);
        if (r.nruns >= kStMaxRuns || region >= max_regions) {   // the host rules this out
            r.ok = false;
            break;
        }
        const int win = s_wlist ? s_wlist[wi] : wi;
        if (write) segs[n] = {kStShrink, u - wi * KU2, e - wi * KU2, wi, region, kChunk * kStWin * win};
#pragma unroll
        for (int i = 0; i < kStMaxRuns; ++i)
            if (i == r.nruns) r.run_w[i] = wi;   // constant indices: stays in registers
        ++r.nruns;
        ++n;
        ++region;
        u = e;
    }
    const int bb = shrink_first ? b0 : b0 + nbase_first;
    if (b1 > bb) {
        if (write) segs[n] = {kStBase, bb, b1, 0, 0, 0};
        ++n;
    }
    r.n = n;
    return r;
}

__global__ void __launch_bounds__(kClThreads, 1)
    lora_cluster_kernel(const __grid_constant__ CUtensorMap tm_w3, const __grid_constant__ CUtensorMap tm_a3,
                        const __grid_constant__ CUtensorMap tm_b3, const __grid_constant__ CUtensorMap tm_x3,
                        const ClusterParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (blockIdx.x >= p.C * p.NT) {
        // the extra cluster (p.build): its first CTA builds this call's
        // segment table beside the weight stream, once the kernel ahead has
        // finished with the workspace; the others have nothing to do
        pdl_launch_dependents();
        if (blockIdx.x == p.C * p.NT) {
            pdl_wait();
            SegBuild<kClThreads / 32>::run(p.seg, reinterpret_cast<int *>(smem));
        }
        return;
    }
    const int T = p.T_pad;
    const int slot_bytes = kClWArea + T * 256;    // [W / A / B box | token operand]
    const uint32_t unit_tx = kClWArea + T * 256;   // a base / shrink unit: weight box + x box
    const int SR = p.s_ring;                      // S ring slots
    const int sw_bytes = kStWin * T * 32;         // one window's S operand: [8 panels][T][16] bf16
    uint8_t *sring = smem + p.stages * slot_bytes;
    float *red = reinterpret_cast<float *>(sring + SR * sw_bytes);   // [C][128/C][T]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + kSplitBN * T);
    uint64_t *empty = full + kClMaxStages;
    uint64_t *acc_full = empty + kClMaxStages;
    uint64_t *red_full = acc_full + kStMaxRegions;
    uint64_t *s_ready = red_full + 1;             // [kClMaxSRing] S slot staged (the 128 loader threads)
    uint64_t *s_free = s_ready + kClMaxSRing;     // [kClMaxSRing] S slot read by its expand MMAs
    // e4m3 pools: the ic-th 8-bit box (in ring order) has landed on
    // codes[ic % stages] and is widened on conv[ic % stages].  The boxes get
    // barriers of their own (not the ring's full[]) because the epilogue
    // warps that widen them skip the base units in between: waiting on a
    // ring slot two phases ahead would see the parity of an older phase.
    // Here the waiters walk the 8-bit boxes in order, and the producer
    // issues box ic + stages only after the MMA issuer has consumed box ic
    // (its ring slot comes free later), so no phase is ever skipped.
    uint64_t *conv = s_free + kClMaxSRing;        // [stages]
    uint64_t *codes = conv + kClMaxStages;        // [stages]
    int *ivars = reinterpret_cast<int *>(codes + kClMaxStages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ivars);
    volatile int *abort_flag = ivars + 1;
    int *n_segs = ivars + 2;       // segments before the expand
    int *n_exp = ivars + 4;        // 1: segs[*n_segs] is my expand segment
    uint16_t *s_bias = reinterpret_cast<uint16_t *>(ivars + 10);   // [128] my output rows' bias (16-byte aligned)
    int *s_ids = reinterpret_cast<int *>(s_bias + kSplitBN);         // [64] token ids (-2 past M)
    float *s_tsc = reinterpret_cast<float *>(s_ids + 64);             // [64] token's LoRA scale (scale x factor)
    StSeg *segs = reinterpret_cast<StSeg *>(s_tsc + 64);
    int *s_win_panel = reinterpret_cast<int *>(segs + kStMaxSegs);   // [kStMaxWinCta] first panel of my windows
    int *s_win_acc = s_win_panel + kStMaxWinCta;       // [kStMaxWinCta] window-sum / counter index of my windows
    int *s_win_info = s_win_acc + kStMaxWinCta;        // [kStMaxWinCta][8] adapter of each panel, -1 if absent
    int *s_run_info = s_win_info + kStMaxWinCta * kStWin;   // [kStMaxRuns][8] the same for my shrink windows
    int *s_zero = s_run_info + kStMaxRuns * kStWin;    // [kStMaxWinCta] I am the window's last consumer
    float *s_pan_fac = reinterpret_cast<float *>(s_zero + kStMaxWinCta);   // [kStMaxWinCta][8] owner's factor
    int *s_win_touch = reinterpret_cast<int *>(s_pan_fac + kStMaxWinCta * kStWin);   // [kStMaxWinCta] a token uses it
    unsigned *s_wbits = reinterpret_cast<unsigned *>(s_zero + kStMaxWinCta);   // [16] windows touched
    int *s_wpre = reinterpret_cast<int *>(s_wbits + kStMaxWinAll / 32);       // [16] popcount prefix
    int *s_wlist = s_wpre + kStMaxWinAll / 32;         // [kStMaxWinList] windows touched, ascending

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.C * p.NT, cta = blockIdx.x;   // the compute CTAs
    const int C = p.C;
    const int q = static_cast<int>(cluster_ctarank());
    const int n0 = (cta / C) * kSplitBN;
    int32_t *status = p.counters + CNT_STATUS;
    const int KU2 = (p.kblocks + 1) / 2;          // K units of 2 K blocks
    // allw: every window of the pool is shrunk and expanded, so the unit
    // list is known at launch and the shrink goes first; otherwise warp 2
    // finds the windows the batch touches and the first units are base units
    const bool allw = p.all_windows != 0;
    // my base K units: an equal share of the tile's K (evening the shares
    // out by the CTAs' shrink and expand units was measured slower: the
    // expand windows wait on S, not on bandwidth)
    const int b0 = (KU2 * q) / C, b1 = (KU2 * (q + 1)) / C;

    const int rpo = kSplitBN / C;                 // output rows owned by each CTA of the cluster
    int nfirst;   // units issued in the prologue (no metadata needed)
    if (allw) {
        const int U = p.windows_all * KU2;
        const int nsh = (U * (cta + 1)) / G - (U * cta) / G;
        nfirst = min(p.stages, nsh + (b1 - b0));
    } else {
        nfirst = min(min(p.stages, kStFirst), b1 - b0);
    }
    // window k's arrival counter is wcnt[k * kWinCntStride], its consumer
    // counter sits in the other half of the same 128-byte line
    constexpr int kCntStride = kWinCntStride;
    int32_t *wcnt = p.wcnt;
    int32_t *ccnt = p.wcnt + kCntStride / 2;

    // ---- prologue: nothing in this kernel depends on the segment builder ------
    // Launched as a programmatic dependent (early_weights), the kernel may
    // start while the kernels ahead of it still run: until griddepcontrol.wait
    // it touches only the weights (W, the A pool) and its own shared memory
    // and TMEM; x, the ids, the workspace and y come after the wait.
    // the warp that builds the token tables: warp 2 when the batch decides
    // which windows are shrunk, else loader warp 6 (the epilogue warps then
    // need no table before the shrink runs)
    const int meta_warp = allw ? 6 : 2;
    int id0 = -1, id1 = -1;   // meta_warp: the ids of tokens lane, lane + 32 (inputs; loaded first)
    if (warp == meta_warp && !p.early_weights) {
        id0 = lane < p.M ? p.ids[lane] : -2;
        id1 = lane + 32 < p.M ? p.ids[lane + 32] : -2;
    }
    if (warp == 0) {
        // one barrier per lane
        if (lane < p.stages) {
            mbar_init(&full[lane], 1);   // the producer's expect_tx arrive (every operand comes by TMA)
            mbar_init(&empty[lane], 1);
        }
        if (lane < SR) {
            mbar_init(&s_ready[lane], 128);
            mbar_init(&s_free[lane], 1);
        }
        if (lane < p.stages) {
            mbar_init(&conv[lane], 128);   // the four epilogue warps widen each 8-bit box
            mbar_init(&codes[lane], 1);    // the producer's expect_tx arrive
        }
        if (lane < kStMaxRegions) mbar_init(&acc_full[lane], 1);
        if (lane == 0) {
            mbar_init(red_full, 1);
            *abort_flag = 0;
            mbar_expect_tx(red_full, static_cast<uint32_t>(kSplitBN * T * 4));   // the C partials of my rows
        }
        fence_mbarrier_init();
        __syncwarp();
        if (lane == 0) {
            if (allw) {
                // the first units: my shrink units (window, K unit), then base
                const int U = p.windows_all * KU2;
                const int u0 = (U * cta) / G, u1 = (U * (cta + 1)) / G;
                for (int i = 0; i < nfirst; ++i) {
                    uint8_t *wa = smem + i * slot_bytes;
                    const int u = u0 + i;
                    if (u < u1 && p.fp8) {   // 8-bit A codes (the i-th 8-bit box), widened by the epilogue warps
                        mbar_expect_tx(&full[i], T * 256);
                        mbar_expect_tx(&codes[i % p.stages], kFp8Box);
                        tma_load_2d(wa + kFp8Box, &tm_a3, &codes[i % p.stages], 2 * kBK * (u % KU2),
                                    kChunk * kStWin * (u / KU2));
                    } else {
                        mbar_expect_tx(&full[i], unit_tx);
                        if (u < u1) tma_load_3d_st(wa, &tm_a3, &full[i], 0, kChunk * kStWin * (u / KU2), 2 * (u % KU2));
                        else tma_load_3d_st(wa, &tm_w3, &full[i], 0, n0, 2 * (b0 + (u - u1)));
                    }
                }
                pdl_wait();   // x may be written by the kernel ahead of this one
                for (int i = 0; i < nfirst; ++i) {
                    const int u = u0 + i;
                    tma_load_3d_st(smem + i * slot_bytes + kClWArea, &tm_x3, &full[i], 0, 0,
                                   u < u1 ? 2 * (u % KU2) : 2 * (b0 + (u - u1)));
                }
            } else {
                for (int i = 0; i < nfirst; ++i) {
                    mbar_expect_tx(&full[i], unit_tx);
                    tma_load_3d_st(smem + i * slot_bytes, &tm_w3, &full[i], 0, n0, 2 * (b0 + i));
                }
                pdl_wait();
                for (int i = 0; i < nfirst; ++i)
                    tma_load_3d_st(smem + i * slot_bytes + kClWArea, &tm_x3, &full[i], 0, 0, 2 * (b0 + i));
            }
            tma_prefetch_map(&tm_a3);
            tma_prefetch_map(&tm_b3);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp < 6) {
        tc_fence_before();
        named_bar_sync(kBarTmem, 192);
        tc_fence_after();
    }
    // the bias of the rows this CTA finishes (a weight: read before the wait),
    // held in registers until the shrink runs are released
    uint4 bias_reg = make_uint4(0u, 0u, 0u, 0u);
    const bool bias_thread = threadIdx.x >= 160 && threadIdx.x < 160 + rpo / 8;
    if (bias_thread && p.bias && n0 + q * rpo + 8 * (threadIdx.x - 160) < p.N)
        bias_reg = __ldg(reinterpret_cast<const uint4 *>(p.bias + n0 + q * rpo + 8 * (threadIdx.x - 160)));
    if (allw && warp == meta_warp) {
        // The owner of each pool panel of my expand windows and its factor:
        // the pool table is a weight, so this is read before the wait.  Only
        // the ids are left for after it.
        const int wa0 = (p.windows_all * q) / C;
        const int wa1 = min((p.windows_all * (q + 1)) / C, wa0 + kStMaxWinCta);
        const int plo = kStWin * wa0, phi = kStWin * wa1;
        for (int k = lane; k < phi - plo; k += 32) {
            s_win_info[k] = -1;
            s_pan_fac[k] = 1.f;
        }
        __syncwarp();
        for (int i0 = 0; i0 < p.A; i0 += 8 * 32) {
            int64_t ao[8];
            int rk[8];
            float fa[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {   // all loads first
                const int i = i0 + 32 * j + lane;
                ao[j] = i < p.A ? p.a_offset[i] : 0;
                rk[j] = i < p.A ? p.rank[i] : 0;
                fa[j] = i < p.A && p.adapter_scale ? p.adapter_scale[i] : 1.f;
                if (p.fp8 && i < p.A) fa[j] *= p.dequant[2 * i] * p.dequant[2 * i + 1];   // e4m3: A and B factors
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + 32 * j + lane;
                if (i >= p.A) continue;
                const int pa = static_cast<int>(ao[j] / p.K) / kChunk, np = min(rk[j] / kChunk, LORA_MAX_RANK / kChunk);
                for (int pp = max(pa, plo); pp < min(pa + np, phi); ++pp) {
                    s_win_info[pp - plo] = i;
                    s_pan_fac[pp - plo] = fa[j];
                }
            }
        }
        __syncwarp();
    }
    pdl_launch_dependents();   // a dependent launch (the segment builder) may start on an idle SM
    cluster_arrive_relaxed();  // my barriers are initialised; peers wait for this before any st.async
    const uint32_t tmem_base = warp < 6 ? *tmem_slot : 0u;
    // the kernels ahead of this one are complete and their writes visible
    // before any thread reads an input other than the weights, touches the
    // workspace or y, or starts a bounded wait
    pdl_wait();
    if (warp == meta_warp && p.early_weights) {
        id0 = lane < p.M ? p.ids[lane] : -2;
        id1 = lane + 32 < p.M ? p.ids[lane + 32] : -2;
    }

    if (warp == 0) {
        // ===================== TMA producer: W, A and B boxes ================
        named_bar_sync(kBarMeta, kMetaThreads);
        const int nk = *n_segs;
        uint32_t it = 0;
        uint32_t ic = 0;   // e4m3: 8-bit boxes in ring order (the prologue's included)
        for (int si = 0; si <= nk; ++si) {
            if (si == nk) {   // the expand windows, once the tables are ready
                named_bar_sync(kBarTables, kTablesThreads);
                if (!*n_exp) break;
            }
            const StSeg sg = segs[si];
            for (int u = sg.a; u < sg.b; ++u) {
                if (sg.kind == kStExpand && !s_win_touch[u - sg.a]) continue;   // no token uses the window
                const uint32_t iu = it++;
                const uint32_t icu = p.fp8 && sg.kind != kStBase ? ic++ : 0;   // its index among the 8-bit boxes
                if (iu < static_cast<uint32_t>(nfirst)) continue;   // issued in the prologue
                const int s = iu % p.stages;
                const uint32_t round = iu / p.stages;
                // A slot's barriers get the unit's arrives only once their
                // previous phases have completed (immediate in a healthy run:
                // the MMA waited for them before freeing the slot), so an
                // arrive always opens a new phase, also after a timeout let a
                // wait go early; a unit whose slot never comes free is skipped.
                bool ok = true;
                if (lane == 0 && round > 0) {
                    mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                    ok = mbar_wait(&full[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                }
                if (lane == 0 && ok && p.fp8 && sg.kind != kStBase && icu >= static_cast<uint32_t>(p.stages))
                    ok = mbar_wait(&codes[icu % p.stages], (icu / p.stages - 1) & 1, abort_flag, status,
                                   LORA_DEV_TIMEOUT);
                if (lane == 0 && ok) {
                    uint8_t *wa = smem + s * slot_bytes;
                    uint64_t *cb = &codes[icu % p.stages];
                    if (sg.kind == kStExpand && p.fp8) {   // 8-bit B codes; the slot carries nothing else
                        mbar_arrive(&full[s]);
                        mbar_expect_tx(cb, kFp8Box);
                        tma_load_3d_st(wa + kFp8Box, &tm_b3, cb, 0, n0, s_win_panel[u - sg.a]);
                    } else if (sg.kind == kStExpand) {
                        mbar_expect_tx(&full[s], kClWArea);
                        tma_load_3d_st(wa, &tm_b3, &full[s], 0, n0, s_win_panel[u - sg.a]);
                    } else if (sg.kind == kStShrink && p.fp8) {   // 8-bit A codes; the x box on the slot
                        mbar_expect_tx(&full[s], T * 256);
                        mbar_expect_tx(cb, kFp8Box);
                        tma_load_2d(wa + kFp8Box, &tm_a3, cb, 2 * kBK * u, sg.arow);
                        tma_load_3d_st(wa + kClWArea, &tm_x3, &full[s], 0, 0, 2 * u);
                    } else {
                        mbar_expect_tx(&full[s], unit_tx);
                        if (sg.kind == kStShrink) tma_load_3d_st(wa, &tm_a3, &full[s], 0, sg.arow, 2 * u);
                        else tma_load_3d_st(wa, &tm_w3, &full[s], 0, n0, 2 * u);
                        tma_load_3d_st(wa + kClWArea, &tm_x3, &full[s], 0, 0, 2 * u);
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp >= 6) {
        // ===================== loaders: the S operand of the expand ==========
        // Each expand window's S is staged into slot w % SR of the S ring as
        // soon as the window's sum is complete.  Every CTA shrinks before it
        // streams its base units, so the sums are complete long before the
        // expand units' B boxes arrive: the staging overlaps the weight
        // stream.  A slot is reused only after the MMAs of the window it
        // held have read it.
        const int lt = threadIdx.x - 192;
        named_bar_sync(kBarTablesLd, kTablesLdThreads);   // the plan (written before it) and the tables   // s_win_*; and s_ids, s_tsc unless every window is shrunk
        const int ew0 = *n_exp ? segs[*n_segs].a : 0;
        const int ew1 = *n_exp ? segs[*n_segs].b : 0;
        if (allw && warp == meta_warp) {
            // each token's adapter (the panel table was built before the
            // wait); an id outside [0, A) matches no panel
            s_ids[lane] = id0;
            s_ids[lane + 32] = id1;
            for (int k = lane; k < ew1 - ew0; k += 32) s_win_touch[k] = 0;
            __syncwarp();
            // a window is expanded only if some token's adapter owns one of its panels
            for (int k = lane; k < (ew1 - ew0) * kStWin; k += 32) {
                const int owner = s_win_info[k];
                bool hit = false;
                for (int t = 0; t < 64 && owner >= 0 && !hit; ++t) hit = s_ids[t] == owner;
                if (hit) s_win_touch[k / kStWin] = 1;
            }
            __syncwarp();
            named_bar_arrive(kBarTables, kTablesThreads);   // producer and MMA: which windows to expand
            named_bar_arrive(kBarTouch, 160);                // epilogue: whether my output tile gets any MMA
        }
        // every window of my share must be complete: one lane per window
        // waits, so the checks overlap
        for (int k = ew0 + lane; k < ew1; k += 32)
            wait_flag_geq(wcnt + s_win_acc[k - ew0] * kCntStride, KU2, abort_flag, status, LORA_DEV_TIMEOUT);
        __syncwarp();
        if (allw) named_bar_sync(kBarLoad, 128);   // warp 6's token table
        // my reads of the sums of windows [counted, hi) are done (or a
        // window no token uses needs no read): count myself as their
        // consumer; the last of the NT consumers of a window clears it
        int counted = 0;
        auto count_upto = [&](int hi) {
            if (hi <= counted) return;
            named_bar_sync(kBarLoad, 128);
            if (lt == 0)
                for (int k = counted; k < hi; ++k)
                    s_zero[k] = atom_acq_rel_gpu_add(ccnt + s_win_acc[k] * kCntStride, 1) == p.NT - 1;
            named_bar_sync(kBarLoad, 128);
            for (int k = counted; k < hi; ++k) {
                if (!s_zero[k]) continue;
                const int ai = s_win_acc[k];
                float4 *ws4 = reinterpret_cast<float4 *>(p.acc + static_cast<int64_t>(ai) * T * kSplitBN);
                for (int i = lt; i < T * kSplitBN / 4; i += 128) ws4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (lt == 0) {
                    wcnt[ai * kCntStride] = 0;
                    ccnt[ai * kCntStride] = 0;
                }
            }
            counted = hi;
        };
        // the windows some token uses, staged in S ring slot wt % SR (wt:
        // their index among those windows, as the MMA issuer counts them)
        for (int w = 0, wt = 0; w < ew1 - ew0; ++w) {
            if (!s_win_touch[w]) continue;
            const int r = wt % SR;
            const uint32_t round = wt / SR;
            if (round > 0) count_upto(w);   // before waiting for a slot: the windows before w are read
            if (lane == 0 && round > 0) mbar_wait(&s_free[r], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
            __syncwarp();
            ++wt;
            uint8_t *xa = sring + r * sw_bytes;
            // S panels [8][T rows][16], 32-byte swizzle (chunk c of row t at
            // t*32 + (c ^ ((t >> 2) & 1))*16); pieces of 8 ranks (panel j,
            // token t, half c); all loads of a thread are issued before the
            // first conversion
            const int *info = s_win_info + w * kStWin;
            const float *wsum = p.acc + static_cast<int64_t>(s_win_acc[w]) * T * kSplitBN;
            const int pieces = kStWin * T * 2;           // <= 1024 for T <= 64
            constexpr int kMaxPer = kStWin * kStreamMaxTokens * 2 / 128;
            float4 f[kMaxPer][2];
            bool use[kMaxPer];
#pragma unroll
            for (int i = 0; i < kMaxPer; ++i) {
                const int pc = lt + 128 * i;
                const int j = pc / (T * 2), rem = pc - j * T * 2;
                const int t = rem >> 1, c = rem & 1;
                use[i] = pc < pieces && info[j] >= 0 && s_ids[t] == info[j];
                f[i][0] = f[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (use[i]) {
                    const float4 *src = reinterpret_cast<const float4 *>(wsum + t * kSplitBN + j * 16 + c * 8);
                    f[i][0] = __ldcg(src);
                    f[i][1] = __ldcg(src + 1);
                }
            }
#pragma unroll
            for (int i = 0; i < kMaxPer; ++i) {
                const int pc = lt + 128 * i;
                if (pc >= pieces) break;
                const int j = pc / (T * 2), rem = pc - j * T * 2;
                const int t = rem >> 1, c = rem & 1;
                // used only for tokens of the panel's adapter: the call's
                // scale times that adapter's factor
                const float sc = allw ? p.scale * s_pan_fac[w * kStWin + j] : s_tsc[t];
                const float4 f0 = f[i][0], f1 = f[i][1];
                const uint4 o = make_uint4(pack_bf16x2(f0.x * sc, f0.y * sc), pack_bf16x2(f0.z * sc, f0.w * sc),
                                           pack_bf16x2(f1.x * sc, f1.y * sc), pack_bf16x2(f1.z * sc, f1.w * sc));
                *reinterpret_cast<uint4 *>(xa + j * T * 32 + t * 32 + ((c ^ ((t >> 2) & 1)) << 4)) = o;
            }
            fence_proxy_async_smem();   // generic-proxy stores -> tensor core reads
            mbar_arrive(&s_ready[r]);
        }
        count_upto(ew1 - ew0);
    } else if (warp == 1) {
        // ===================== MMA issuer ====================================
        uint32_t started = 0;   // bit r: region r holds a partial sum
        uint32_t ic = 0;        // e4m3: 8-bit units consumed (their widening is signalled on conv[ic % stages])
        const uint32_t idesc = umma_idesc_bf16(kSplitBN, T);
        auto wait_widened = [&]() {
            mbar_wait(&conv[ic % p.stages], (ic / p.stages) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
            ++ic;
            fence_proxy_async_smem();   // the widened operand was written through the generic proxy
        };
        auto mma_kunit = [&](uint32_t it, uint32_t d, int region, bool widened) {
            const int s = it % p.stages;
            mbar_wait(&full[s], (it / p.stages) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
            if (widened) wait_widened();
            tc_fence_after();
            if (lane == 0) {
                const uint32_t wa = smem_u32(smem + s * slot_bytes);
                const uint32_t xa = wa + kClWArea;
                uint32_t acc = (started >> region) & 1;
                for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        umma_bf16(d, umma_sdesc(wa + kb * kSplitBN * kBK * 2 + kk * 32, 1024, kSwizzle128),
                                  umma_sdesc(xa + kb * T * kBK * 2 + kk * 32, 1024, kSwizzle128), idesc, acc);
                        acc = 1;
                    }
                }
                umma_commit(&empty[s]);
            }
            started |= 1u << region;
            __syncwarp();
        };
        uint32_t it = 0;
        int si0 = 0;
        if (!allw) {   // the first base units are known before the metadata
            for (; it < static_cast<uint32_t>(nfirst); ++it) mma_kunit(it, tmem_base, 0, false);
            si0 = 1;
        }
        named_bar_sync(kBarMma, 64);
        const int nk = *n_segs;
        int wt = 0;   // expand windows issued so far
        for (int si = si0; si <= nk; ++si) {
            if (si == nk) {   // the expand windows, once the tables are ready
                named_bar_sync(kBarTables, kTablesThreads);
                if (!*n_exp) break;
            }
            const StSeg sg = segs[si];
            const uint32_t d = tmem_base + sg.region * T;
            for (int u = sg.a; u < sg.b; ++u) {
                if (sg.kind != kStExpand) {
                    mma_kunit(it++, d, sg.region, p.fp8 && sg.kind == kStShrink);
                    continue;
                }
                // the window's B box through the ring, its S in slot r of the
                // S ring (windows no token uses are skipped: wt counts the others)
                if (!s_win_touch[u - sg.a]) continue;
                const int w = wt++, r = w % SR;
                const int s = static_cast<int>(it % p.stages);
                mbar_wait(&full[s], (it / p.stages) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                if (p.fp8) wait_widened();
                mbar_wait(&s_ready[r], (w / SR) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                fence_proxy_async_smem();   // the S operand arrived through the generic proxy
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t wa = smem_u32(smem + s * slot_bytes);
                    const uint32_t xa = smem_u32(sring + r * sw_bytes);
                    uint32_t acc = started & 1;
                    for (int j = 0; j < kStWin; ++j) {
                        umma_bf16(d, umma_sdesc(wa + j * kSplitBN * kChunk * 2, 256, kSwizzle32),
                                  umma_sdesc(xa + j * T * kChunk * 2, 256, kSwizzle32), idesc, acc);
                        acc = 1;
                    }
                    umma_commit(&empty[s]);
                    umma_commit(&s_free[r]);
                }
                ++it;
                started |= 1u;
                __syncwarp();
            }
            if (sg.kind == kStShrink) {
                if (lane == 0) umma_commit(&acc_full[sg.region]);
                __syncwarp();
            }
        }
        if (lane == 0) umma_commit(&acc_full[0]);   // the output tile (all MMAs above)
        __syncwarp();
    } else {
        // ===================== epilogue (warps 2..5) =========================
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int et = threadIdx.x - 64;
        if (warp == 2) {
            // ---- metadata --------------------------------------------------
            SegPlan pl;
            if (allw) {
                // every window of the pool is shrunk and expanded: the whole
                // unit list is known at launch, and the shrink runs need no
                // token table (loader warp 6 builds the one the S staging uses)
                pl = plan_segments(segs, lane == 0, p.windows_all, KU2, G, cta, b0, b1, 0, p.max_regions, nullptr,
                                   true);
                const int w0 = (p.windows_all * q) / C, w1 = (p.windows_all * (q + 1)) / C;
                const int wend = min(w1, w0 + kStMaxWinCta);
                for (int k = w0 + lane; k < wend; k += 32) {
                    s_win_panel[k - w0] = kStWin * k;
                    s_win_acc[k - w0] = k;
                }
                if (lane == 0) {
                    *n_segs = pl.n;
                    segs[pl.n] = {kStExpand, w0, wend, 0, 0, 0};
                    *n_exp = w1 > w0;
                    if (!pl.ok || w1 - w0 > kStMaxWinCta) {   // the host rules both out
                        atomicOr(status, LORA_DEV_TIMEOUT);
                        *abort_flag = 1;
                    }
                }
                __syncwarp();
                named_bar_arrive(kBarMma, 64);
                named_bar_arrive(kBarMeta, kMetaThreads);
                named_bar_arrive(kBarTablesEpi, 128);
                named_bar_arrive(kBarTablesLd, kTablesLdThreads);   // kBarTables: warp 6, once it knows the ids
            } else {
            // tokens' adapters: pool panels [pa, pa + np), windows pa/8 ..
            const bool v0 = id0 >= 0 && id0 < p.A, v1 = id1 >= 0 && id1 < p.A;
            const int64_t ao0 = v0 ? p.a_offset[id0] : 0, ao1 = v1 ? p.a_offset[id1] : 0;
            const int rk0 = v0 ? p.rank[id0] : 0, rk1 = v1 ? p.rank[id1] : 0;
            const bool fac = p.adapter_scale != nullptr;
            float f0 = fac && v0 ? p.adapter_scale[id0] : 1.f, f1 = fac && v1 ? p.adapter_scale[id1] : 1.f;
            if (p.fp8) {   // e4m3: A and B factors
                if (v0) f0 *= p.dequant[2 * id0] * p.dequant[2 * id0 + 1];
                if (v1) f1 *= p.dequant[2 * id1] * p.dequant[2 * id1 + 1];
            }
            s_ids[lane] = id0;
            s_ids[lane + 32] = id1;
            s_tsc[lane] = p.scale * f0;
            s_tsc[lane + 32] = p.scale * f1;
            const int pa0 = static_cast<int>(ao0 / p.K) / kChunk, np0 = v0 ? min(rk0 / kChunk, LORA_MAX_RANK / kChunk) : 0;
            const int pa1 = static_cast<int>(ao1 / p.K) / kChunk, np1 = v1 ? min(rk1 / kChunk, LORA_MAX_RANK / kChunk) : 0;
            // the windows the batch touches, ascending (s_wlist)
            if (lane < kStMaxWinAll / 32) s_wbits[lane] = 0u;
            __syncwarp();
            auto mark = [&](int pa, int np) {
                if (np <= 0) return;
                for (int wv = pa / kStWin; wv <= (pa + np - 1) / kStWin && wv < p.windows_all; ++wv)
                    atomicOr(&s_wbits[wv >> 5], 1u << (wv & 31));
            };
            mark(pa0, np0);
            mark(pa1, np1);
            __syncwarp();
            const unsigned bits = lane < kStMaxWinAll / 32 ? s_wbits[lane] : 0u;
            const int cnt = __popc(bits);
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int NT_ = __shfl_sync(0xffffffffu, incl, 31);   // windows touched (<= 2 per token)
            if (lane < kStMaxWinAll / 32) s_wpre[lane] = incl - cnt;
            for (unsigned b = bits, k = incl - cnt; b; b &= b - 1, ++k) s_wlist[k] = 32 * lane + __ffs(b) - 1;
            __syncwarp();
            // only the touched windows are shrunk, named by their list index
            pl = plan_segments(segs, lane == 0, NT_, KU2, G, cta, b0, b1, nfirst, p.max_regions, s_wlist, false);
            if (lane == 0) *n_segs = pl.n;
            __syncwarp();
            named_bar_arrive(kBarMma, 64);
            named_bar_arrive(kBarMeta, kMetaThreads);   // the producer may issue the shrink boxes now
            if (!pl.ok && lane == 0) {
                atomicOr(status, LORA_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            // ---- my expand windows: a share of the touched windows ------------
            const int w0 = (NT_ * q) / C, w1 = (NT_ * (q + 1)) / C;
            if (w1 - w0 > kStMaxWinCta && lane == 0) {   // the host rules this out
                atomicOr(status, LORA_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            const int wend = min(w1, w0 + kStMaxWinCta);
            for (int k = w0 + lane; k < wend; k += 32) {
                s_win_panel[k - w0] = kStWin * s_wlist[k];
                s_win_acc[k - w0] = k;   // sums are kept per shrunk window
            }
            for (int k = lane; k < (wend - w0) * kStWin; k += 32) s_win_info[k] = -1;
            for (int k = lane; k < wend - w0; k += 32) s_win_touch[k] = 1;   // only touched windows are listed
            s_run_info[lane] = -1;   // kStMaxRuns x kStWin = 32 entries
            if (lane == 0) {
                segs[pl.n] = {kStExpand, w0, wend, 0, 0, 0};
                *n_exp = w1 > w0;
            }
            __syncwarp();
            // the adapter owning each panel of my windows (absent panels stay -1)
            auto fill = [&](int id, int pa, int np) {
                if (np <= 0) return;
                for (int wv = pa / kStWin; wv <= (pa + np - 1) / kStWin && wv < p.windows_all; ++wv) {
                    const int pos = s_wpre[wv >> 5] + __popc(s_wbits[wv >> 5] & ((1u << (wv & 31)) - 1u));
                    const int lo = max(pa, kStWin * wv), hi = min(pa + np, kStWin * wv + kStWin);
                    if (pos >= w0 && pos < wend)
                        for (int pp = lo; pp < hi; ++pp) s_win_info[(pos - w0) * kStWin + pp - kStWin * wv] = id;
#pragma unroll
                    for (int r = 0; r < kStMaxRuns; ++r)
                        if (pl.run_w[r] == pos)
                            for (int pp = lo; pp < hi; ++pp) s_run_info[r * kStWin + pp - kStWin * wv] = id;
                }
            };
            fill(id0, pa0, np0);
            fill(id1, pa1, np1);
            __syncwarp();
            named_bar_arrive(kBarTablesEpi, 128);
            named_bar_arrive(kBarTables, kTablesThreads);
            named_bar_arrive(kBarTablesLd, kTablesLdThreads);
            }
        } else {
            named_bar_sync(kBarMeta, kMetaThreads);
            named_bar_sync(kBarTablesEpi, 128);   // s_run_info, s_wbits
        }
        const int ns = *n_segs;
        // The B boxes of my expand windows into L2 now (a prefetch through the
        // tensor map: the box the producer loads after the weight stream), so
        // that load finds them there instead of waiting on HBM.  The pool is
        // a weight; L2 is coherent, so this is safe before the programmatic
        // wait too.
        if (warp == 3 && *n_exp)
            for (int w = lane; w < segs[ns].b - segs[ns].a; w += 32) tma_prefetch_3d(&tm_b3, 0, n0, s_win_panel[w]);
        // ---- shrink runs: add my partial window sums, then release ------------
        auto shrink_run = [&](const StSeg &sg, int run) {
            mbar_wait(&acc_full[sg.region], 0, abort_flag, status, LORA_DEV_TIMEOUT);
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + sg.region * T;
            // the rows of every panel go into the sum when every window is
            // expanded (the S staging keeps each token's own panels); else
            // only the panels of an adapter present
            const bool live = allw || s_run_info[run * kStWin + row / kChunk] >= 0;
            float *dst = p.acc + static_cast<int64_t>(sg.w) * T * kSplitBN + row;
            for (int c = 0; c < T; c += 16) {
                uint32_t v[16];
                tmem_ld16(tbase + c, v);
                tmem_ld_wait16(v);
                if (live) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) atomicAdd(dst + (c + e) * kSplitBN, __uint_as_float(v[e]));
                }
            }
            // one release for the whole run, after all four warps' additions:
            // the window is complete once its KU2 units have arrived (every
            // shrunk window is expanded, so its consumers clear it again)
            named_bar_sync(kBarEpi, 128);
            if (et == 0) red_release_gpu_add(wcnt + sg.w * kCntStride, sg.b - sg.a);
        };
        // e4m3 pool: the 8-bit box of ring unit iu (the cic-th 8-bit box)
        // sits in the upper half of its slot's weight area once codes[] says
        // so; widen it in place to the bf16 operand the MMA reads (the bf16
        // box's layout)
        uint32_t cit = 0, cic = 0;   // ring units and 8-bit units walked, as the producer and the MMA count them
        auto widen_unit = [&](uint32_t iu, bool b_box) {
            const int s = iu % p.stages;
            mbar_wait(&codes[cic % p.stages], (cic / p.stages) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
            uint8_t *wa = smem + s * slot_bytes;
            const uint8_t *box = wa + kFp8Box;
            uint4 c[8];
            if (!b_box) {
                // A: box row et (128 K codes) -> row et of K blocks 0 and 1,
                // 128-byte swizzle (16-byte chunk q at (q ^ (row & 7)) * 16);
                // only this thread reads the row it overwrites.  Step h
                // reads the row's 16-code group h ^ (et & 7), so the eight
                // threads of a quarter warp read eight different banks.
                const int rot = et & 7;
#pragma unroll
                for (int h = 0; h < 8; ++h) c[h] = reinterpret_cast<const uint4 *>(box + et * 128)[h ^ rot];
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const int g = h ^ rot;   // the 16-code group in c[h]: K block g >> 2, chunks 2 (g & 3) and + 1
                    uint32_t o[8];
                    e4m3x16_to_bf16(c[h], o);
                    uint8_t *rowp = wa + (g >> 2) * (kSplitBN * kBK * 2) + et * 128;
                    const int q = 2 * (g & 3);
                    *reinterpret_cast<uint4 *>(rowp + ((q ^ rot) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4 *>(rowp + (((q + 1) ^ rot) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
            } else {
                // B: row et of each of the 8 panels (16 codes) -> 32-byte rows,
                // 32-byte swizzle (chunk q at (q ^ ((row >> 2) & 1)) * 16); the
                // stores overwrite other threads' codes, so all loads go first
#pragma unroll
                for (int j = 0; j < kStWin; ++j) c[j] = *reinterpret_cast<const uint4 *>(box + j * 2048 + et * 16);
                named_bar_sync(kBarConv, 128);
                const int sw = (et >> 2) & 1;
#pragma unroll
                for (int j = 0; j < kStWin; ++j) {
                    uint32_t o[8];
                    e4m3x16_to_bf16(c[j], o);
                    uint8_t *rowp = wa + j * (kSplitBN * kChunk * 2) + et * 32;
                    *reinterpret_cast<uint4 *>(rowp + (sw << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4 *>(rowp + ((1 ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
            fence_proxy_async_smem();   // generic-proxy stores -> the tensor core's reads
            mbar_arrive(&conv[cic % p.stages]);
            ++cic;
        };
        if (p.fp8) {
            // walk the units in ring order: each shrink run's boxes are widened
            // before its sums are read
            for (int si = 0, run = 0; si < ns; ++si) {
                const StSeg sg = segs[si];
                for (int u = sg.a; u < sg.b; ++u) {
                    const uint32_t iu = cit++;
                    if (sg.kind == kStShrink) widen_unit(iu, false);
                }
                if (sg.kind == kStShrink) shrink_run(sg, run++);
            }
        } else {
            for (int si = 0, run = 0; si < ns; ++si)
                if (segs[si].kind == kStShrink) shrink_run(segs[si], run++);
        }
        if (bias_thread) reinterpret_cast<uint4 *>(s_bias)[threadIdx.x - 160] = bias_reg;
        named_bar_sync(kBarTouch, allw ? 160 : 128);   // the touched flags (warp 6, or warp 2 before kBarTablesEpi)
        if (p.fp8 && *n_exp) {   // the B boxes of the expand windows some token uses
            const StSeg sg = segs[ns];
            for (int u = sg.a; u < sg.b; ++u)
                if (s_win_touch[u - sg.a]) widen_unit(cit++, true);
        }
        // ---- output tile: push my partial rows to their owners ----------------
        mbar_wait(&acc_full[0], 0, abort_flag, status, LORA_DEV_TIMEOUT);
        tc_fence_after();
        // nothing accumulated (no base units and no expand window a token
        // uses): send zeros
        bool any_touch = false;
        if (*n_exp)
            for (int k = 0; k < segs[*n_segs].b - segs[*n_segs].a; ++k) any_touch = any_touch || s_win_touch[k];
        const bool empty_run = b1 == b0 && !any_touch;
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
        cluster_wait();        // every peer's receive barrier is initialised
        const int owner = row / rpo;
        const uint32_t dst = mapa_shared(smem_u32(red) + static_cast<uint32_t>(((q * rpo) + (row - owner * rpo)) * T * 4),
                                         owner);
        const uint32_t bar = mapa_shared(smem_u32(red_full), owner);
        for (int c = 0; c < T; c += 16) {
            uint32_t v[16];
            tmem_ld16(tbase + c, v);
            tmem_ld_wait16(v);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float4 f = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                       __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
                if (empty_run) f = make_float4(0.f, 0.f, 0.f, 0.f);
                st_async_v4(dst + (c + 4 * k) * 4, f, bar);
            }
        }
        // ---- owner: sum the C partials of my rows, bias, bf16, y ---------------
        mbar_wait(red_full, 0, abort_flag, status, LORA_DEV_TIMEOUT);
        // done with distributed shared memory: every peer's bytes have landed
        // here (red_full) and nothing here touches a peer's shared memory
        // any more, so the arrive needs no release ordering
        cluster_arrive_relaxed();
        const int groups = rpo / 8;
        for (int w = et; w < T * groups; w += 128) {
            const int t = w / groups, gq = w % groups;
            const int rloc = gq * 8;
            const int n = n0 + q * rpo + rloc;
            float sum[8];
            const uint4 b = reinterpret_cast<const uint4 *>(s_bias)[gq];
            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sum[2 * e] = bf16_lo(bw[e]);
                sum[2 * e + 1] = bf16_hi(bw[e]);
            }
            for (int c = 0; c < C; ++c) {
                const float *src = red + (c * rpo + rloc) * T + t;
#pragma unroll
                for (int e = 0; e < 8; ++e) sum[e] += src[e * T];
            }
            if (t < p.M && n < p.N)
                *reinterpret_cast<uint4 *>(p.y + static_cast<int64_t>(t) * p.N + n) =
                    make_uint4(pack_bf16x2(sum[0], sum[1]), pack_bf16x2(sum[2], sum[3]), pack_bf16x2(sum[4], sum[5]),
                               pack_bf16x2(sum[6], sum[7]));
        }
    }

    // ---- teardown ---------------------------------------------------------
    if (!(warp >= 2 && warp < 6)) {
        cluster_wait();        // pairs with the start-up arrive
        cluster_arrive();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    cluster_wait();            // no CTA leaves while a peer may still touch its shared memory
}

int cluster_max_regions() { return kStMaxRegions; }
int cluster_max_runs() { return kStMaxRuns; }
int cluster_max_win_cta() { return kStMaxWinCta; }
int cluster_win() { return kStWin; }
size_t cluster_build_smem_bytes(int32_t A) { return SegBuild<kClThreads / 32>::smem_bytes(A); }

size_t cluster_smem_bytes(int T_pad, int stages, int s_ring)
{
    return static_cast<size_t>(stages) * (kClWArea + T_pad * 256) + static_cast<size_t>(s_ring) * kStWin * T_pad * 32 +
           static_cast<size_t>(kSplitBN) * T_pad * 4 + 1024 + kClMisc;
}

// Ring depth: what fits beside two S slots, at most 3.  Deeper rings
// measured no faster: with every CTA's boxes in flight the memory queues
// only grow.
int cluster_stages(int T_pad)
{
    const size_t budget = 227 * 1024 - static_cast<size_t>(kSplitBN) * T_pad * 4 - 1024 - kClMisc -
                          2 * static_cast<size_t>(kStWin) * T_pad * 32;
    int s = static_cast<int>(budget / (kClWArea + T_pad * 256));
    return s > 3 ? 3 : s;
}

// S ring slots: what fits beside the weight ring, 2 to kClMaxSRing (0 if
// not even two fit).
int cluster_s_ring(int T_pad, int stages)
{
    const size_t cap = 227 * 1024;
    const size_t used = cluster_smem_bytes(T_pad, stages, 0);
    const int n = used >= cap ? 0 : static_cast<int>((cap - used) / (static_cast<size_t>(kStWin) * T_pad * 32));
    return n < 2 ? 0 : (n > kClMaxSRing ? kClMaxSRing : n);
}

// Largest cluster size in {8, 4, 2, 1} whose grid (C x (NT + 1) CTAs, one
// per SM) can be resident all at once; 0 when none can.
int cluster_pick_size(int NT, int T_pad, int sms)
{
    const int stages = cluster_stages(T_pad);
    const int s_ring = cluster_s_ring(T_pad, stages);
    if (stages < 2 || s_ring < 2) return 0;
    const size_t smem = cluster_smem_bytes(T_pad, stages, s_ring);
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !configured[dev]) {
        if (cudaFuncSetAttribute(lora_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(227 * 1024)) != cudaSuccess)
            return 0;
        if (dev < 64) configured[dev] = 1;
    }
    // one cluster more than the output tiles: the segment builder's
    for (int C = 8; C >= 1; C >>= 1) {
        if (C * (NT + 1) > sms) continue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C * (NT + 1));
        cfg.blockDim = dim3(kClThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, lora_cluster_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (nclusters >= NT + 1) return C;
    }
    return 0;
}

// pdl: a programmatic dependent launch; the prologue (barriers, TMEM, the
// first weight boxes) may then overlap the kernel ahead on the stream, and
// everything else waits for it (griddepcontrol.wait).
cudaError_t launch_cluster(const ClusterMaps &m, const ClusterParams &p, bool pdl, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.C * (p.NT + (p.build ? 1 : 0)));
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = cluster_smem_bytes(p.T_pad, p.stages, p.s_ring);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, lora_cluster_kernel, m.w3, m.a3, m.b3, m.x3, p);
}

}  // namespace lora
