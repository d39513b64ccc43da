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
// of K.  Work of one CTA, in order through one smem ring:
//   - two base units (W boxes of 128 rows x 2 K blocks = 32 KB), issued
//     before any metadata is read;
//   - its slice of the shrink list: units (group of <= 2 rank panels of one
//     adapter) x (4 K blocks), evenly sliced over the whole grid; each run's
//     fp32 partial S is added with atomics to a per-group sum in L2 and a
//     per-group arrival counter is released;
//   - the rest of its K-part;
//   - its share of the expand steps: 8-panel windows of the B pool (32 KB
//     boxes) that hold panels of adapters present.  The loader warps wait
//     until the window's groups are complete, read the fp32 sums, mask every
//     token to its own adapter, scale, round to bf16 and stage them as the N
//     operand.
// The C partial tiles are then pushed with st.async into the CTA that owns
// each 128/C-row slice (distributed shared memory, mbarrier byte counting);
// the owner sums them, adds the bias and writes y.  The group sums and
// counters are double-buffered by a call epoch: each call zeroes the other
// half for the next call, so nothing is reset on the way out.
// Roles (320 threads): warp 0 TMA producer (W, A and B boxes only: few,
// large operations), warp 1 TMEM allocator + MMA issuer, warps 2..5
// epilogue, warps 6..9 loaders of the token-side operands (x by cp.async,
// S by load-convert-store).  All waits are bounded; the host only launches
// the grid when every cluster can be resident at once.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

constexpr int kClThreads = 320;
constexpr int kClWArea = 32 * 1024;       // W box / A box / B box
constexpr int kStMaxSegs = 24;
constexpr int kStMaxRegions = 16;
constexpr int kStFirstBase = 2;
constexpr int kStWin = 8;                  // panels per expand window

enum StKind { kStBase = 0, kStShrink = 1, kStExpand = 2, kStNone = 3 };

struct StSeg {
    int kind;     // StKind
    int a, b;     // unit range: base units / shrink units of group g / expand windows
    int g;        // shrink group
    int region;   // TMEM accumulator
    int last;     // accumulator complete after this segment
    int arow;     // shrink: first pool row of the group's A panels
    int rows;     // shrink: 16 or 32 rows
};

__device__ __forceinline__ void tma_load_3d_st(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y, int z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(m), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Number of CTAs whose slice of the shrink list [U units, KU4 per group]
// intersects group g (empty slices excluded).
__device__ __forceinline__ int shrink_contributors(int g, int64_t U, int KU4, int G)
{
    const int64_t ua = static_cast<int64_t>(g) * KU4, ub = ua + KU4 - 1;
    const int c0 = static_cast<int>(((ua + 1) * G - 1) / U), c1 = static_cast<int>(((ub + 1) * G - 1) / U);
    int n = 0;
    for (int c = c0; c <= c1; ++c)
        if ((U * (c + 1)) / G > (U * c) / G) ++n;
    return n;
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
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__global__ void __launch_bounds__(kClThreads, 1)
    lora_cluster_kernel(const __grid_constant__ CUtensorMap tm_w3, const __grid_constant__ CUtensorMap tm_a3_16,
                        const __grid_constant__ CUtensorMap tm_a3_32, const __grid_constant__ CUtensorMap tm_b3,
                        const ClusterParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int T = p.T_pad;
    const int slot_bytes = kClWArea + T * 512;    // [W / A / B box | token operand]
    float *red = reinterpret_cast<float *>(smem + p.stages * slot_bytes);   // [C][128/C][T]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + kSplitBN * T);
    uint64_t *empty = full + p.stages;
    uint64_t *acc_full = empty + p.stages;
    uint64_t *red_full = acc_full + kStMaxRegions;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(red_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *n_segs = const_cast<int *>(abort_flag) + 1;
    int *s_epoch = n_segs + 1;
    int *s_ids = s_epoch + 2;                     // [64] token ids (-2 past M)
    StSeg *segs = reinterpret_cast<StSeg *>(s_ids + 64);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int C = p.C;
    const int q = static_cast<int>(cluster_ctarank());
    const int tile_n = cta / C;
    const int n0 = tile_n * kSplitBN;
    int32_t *status = p.counters + CNT_STATUS;
    const int KU2 = (p.kblocks + 1) / 2;          // base units: 2 K blocks
    const int KU4 = (p.kblocks + 3) / 4;          // shrink units: 4 K blocks
    const int b0 = (KU2 * q) / C, b1 = (KU2 * (q + 1)) / C;
    const int nfirst = min(kStFirstBase, b1 - b0);
    const int rpo = kSplitBN / C;                 // output rows owned by each CTA of the cluster

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1 + 128);   // producer's expect_tx arrive + one arrive per loader thread
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < kStMaxRegions; ++a) mbar_init(&acc_full[a], 1);
        mbar_init(red_full, 1);
        *abort_flag = 0;
        mbar_expect_tx(red_full, static_cast<uint32_t>(kSplitBN * T * 4));   // the C partials of my rows
        fence_mbarrier_init();
        // the first base units need no metadata: start streaming W now
        for (int i = 0; i < nfirst; ++i) {
            mbar_expect_tx(&full[i], kClWArea);
            tma_load_3d_st(smem + i * slot_bytes, &tm_w3, &full[i], 0, n0, 2 * (b0 + i));
        }
        const int NG = p.hdr[HDR_DGROUPS];
        const int NW = p.hdr[HDR_NWIN];
        *s_epoch = p.counters[CNT_EPOCH] & 1;
        const int w0 = (NW * q) / C, w1 = (NW * (q + 1)) / C;   // my share of the expand windows
        int n = 0, region = 1;
        const bool has_rest = b1 - b0 > nfirst, has_expand = w1 > w0;
        if (nfirst > 0) segs[n++] = {kStBase, b0, b0 + nfirst, 0, 0, !has_rest && !has_expand, 0, 0};
        const int64_t U = static_cast<int64_t>(NG) * KU4;
        if (U > 0) {
            const int64_t u1 = (U * (cta + 1)) / G;
            for (int64_t u = (U * cta) / G; u < u1 && n < kStMaxSegs - 3 && region < p.max_regions;) {
                const int g = static_cast<int>(u / KU4);
                const int64_t e = min(u1, static_cast<int64_t>(g + 1) * KU4);
                segs[n++] = {kStShrink, static_cast<int>(u - static_cast<int64_t>(g) * KU4),
                             static_cast<int>(e - static_cast<int64_t>(g) * KU4), g, region++, 1, 0, 0};
                u = e;
            }
        }
        if (has_rest) segs[n++] = {kStBase, b0 + nfirst, b1, 0, 0, !has_expand, 0, 0};
        if (has_expand) segs[n++] = {kStExpand, w0, w1, 0, 0, 1, 0, 0};
        if (nfirst == 0 && !has_expand) segs[n++] = {kStNone, 0, 0, 0, 0, 1, 0, 0};
        for (int i = 0; i < n; ++i)   // group metadata now, so the ring never stalls on it
            if (segs[i].kind == kStShrink) {
                segs[i].arow = p.dgrp_arow[segs[i].g];
                segs[i].rows = p.dgrp_len[segs[i].g] * kChunk;
            }
        *n_segs = n;
    }
    if (threadIdx.x >= 64 && threadIdx.x < 64 + 64) {   // epilogue threads stage the token ids
        const int t = threadIdx.x - 64;
        s_ids[t] = t < p.M ? p.ids[t] : -2;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tm_a3_16);
        tma_prefetch_map(&tm_a3_32);
        tma_prefetch_map(&tm_b3);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_arrive();          // my barriers are initialised; peers wait for this before any st.async
    const uint32_t tmem_base = *tmem_slot;
    const int ns = *n_segs;
    const int ep = *s_epoch;
    const int NG = p.hdr[HDR_DGROUPS];
    const int64_t U = static_cast<int64_t>(NG) * KU4;
    float *acc_cur = p.acc + static_cast<int64_t>(ep) * p.max_groups * 32 * T;   // [group][T][32]
    int32_t *gcnt_cur = p.gcnt + ep * p.max_groups;

    if (warp == 0) {
        // ===================== TMA producer: W, A and B boxes ================
        uint32_t it = 0;
        for (int si = 0; si < ns; ++si) {
            const StSeg sg = segs[si];
            for (int u = sg.a; u < sg.b; ++u, ++it) {
                if (si == 0 && sg.kind == kStBase) continue;   // issued in the prologue
                const int s = it % p.stages;
                const uint32_t round = it / p.stages;
                if (lane == 0) {
                    if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                    uint8_t *wa = smem + s * slot_bytes;
                    if (sg.kind == kStShrink) {
                        mbar_expect_tx(&full[s], sg.rows * kBK * 2 * 4);
                        tma_load_3d_st(wa, sg.rows == kChunk ? &tm_a3_16 : &tm_a3_32, &full[s], 0, sg.arow, 4 * u);
                    } else if (sg.kind == kStBase) {
                        mbar_expect_tx(&full[s], kClWArea);
                        tma_load_3d_st(wa, &tm_w3, &full[s], 0, n0, 2 * u);
                    } else {
                        mbar_expect_tx(&full[s], kStWin * kSplitBN * kChunk * 2);
                        tma_load_3d_st(wa, &tm_b3, &full[s], 0, n0, p.ewin_first[u]);
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp >= 6) {
        // ===================== loaders: token-side operands ==================
        // x K blocks: [kb][T rows][64], 128-byte swizzle (chunk c of row r at
        //   r*128 + (c ^ (r & 7))*16), rows >= M and K blocks past K zero;
        // S panels: [panel][T rows][16], 32-byte swizzle (chunk c of row t at
        //   t*32 + (c ^ ((t >> 2) & 1))*16), from the fp32 group sums.
        const int lt = threadIdx.x - 192;
        uint32_t it = 0;
        for (int si = 0; si < ns; ++si) {
            const StSeg sg = segs[si];
            if (sg.kind == kStExpand) {
                // all groups with a panel in my windows must be complete: one
                // lane per panel waits, so the checks overlap
                for (int k = lane; k < (sg.b - sg.a) * kStWin; k += 32) {
                    const int info = p.pinfo[sg.a * kStWin + k];
                    if (info >= 0) {
                        const int g = info >> 1;
                        wait_flag_geq(gcnt_cur + g, shrink_contributors(g, U, KU4, G) * p.dgrp_len[g] * kChunk,
                                      abort_flag, status, LORA_DEV_TIMEOUT);
                    }
                }
                __syncwarp();
            }
            for (int u = sg.a; u < sg.b; ++u, ++it) {
                const int s = it % p.stages;
                const uint32_t round = it / p.stages;
                if (lane == 0 && round > 0) mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                __syncwarp();
                uint8_t *xa = smem + s * slot_bytes + kClWArea;
                if (sg.kind != kStExpand) {
                    const int nkb = sg.kind == kStShrink ? 4 : 2;
                    const int kb0 = u * nkb;
                    const int pieces = nkb * T * 8;
                    for (int pc = lt; pc < pieces; pc += 128) {
                        const int j = pc / (T * 8), rem = pc - j * T * 8;
                        const int row = rem >> 3, c = rem & 7;
                        const int kb = kb0 + j;
                        const bool ok = row < p.M && kb < p.kblocks;
                        const uint16_t *src = p.x + (ok ? static_cast<int64_t>(row) * p.K + kb * kBK + c * 8 : 0);
                        cp_async16(xa + j * T * 128 + row * 128 + ((c ^ (row & 7)) << 4), src, ok ? 16u : 0u);
                    }
                    cp_async_mbar_arrive_noinc(&full[s]);
                } else {
                    const int pieces = kStWin * T * 2;
                    for (int pc = lt; pc < pieces; pc += 128) {
                        const int j = pc / (T * 2), rem = pc - j * T * 2;
                        const int t = rem >> 1, c = rem & 1;
                        const int info = p.pinfo[u * kStWin + j];
                        uint4 o = make_uint4(0u, 0u, 0u, 0u);
                        if (info >= 0) {
                            const int g = info >> 1;
                            if (s_ids[t] == p.dgrp_adapter[g]) {
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    acc_cur + (static_cast<int64_t>(g) * T + t) * 32 + (info & 1) * 16 + c * 8);
                                const float4 f0 = __ldcg(src), f1 = __ldcg(src + 1);
                                const float sc = p.scale;
                                o = make_uint4(pack_bf16x2(f0.x * sc, f0.y * sc), pack_bf16x2(f0.z * sc, f0.w * sc),
                                               pack_bf16x2(f1.x * sc, f1.y * sc), pack_bf16x2(f1.z * sc, f1.w * sc));
                            }
                        }
                        *reinterpret_cast<uint4 *>(xa + j * T * 32 + t * 32 + ((c ^ ((t >> 2) & 1)) << 4)) = o;
                    }
                    fence_proxy_async_smem();   // generic-proxy stores -> tensor core reads
                    mbar_arrive(&full[s]);
                }
            }
        }
        // the last CTA to get here advances the call epoch (every CTA read it
        // long before); the next call uses the other buffers
        if (warp == 6 && lane == 0) {
            if (atom_acq_rel_gpu_add(p.counters + CNT_SPLIT_DONE, 1) == G - 1) {
                p.counters[CNT_SPLIT_DONE] = 0;
                atomicAdd(p.counters + CNT_EPOCH, 1);
            }
        }
        cp_async_wait_all();
    } else if (warp == 1) {
        // ===================== MMA issuer ====================================
        uint32_t it = 0, started = 0;   // bit r: region r holds a partial sum
        const uint32_t idesc = umma_idesc_bf16(kSplitBN, T);
        for (int si = 0; si < ns; ++si) {
            const StSeg sg = segs[si];
            const uint32_t d = tmem_base + sg.region * T;
            const int arows = sg.kind == kStShrink ? p.dgrp_len[sg.g] * kChunk : kSplitBN;
            for (int u = sg.a; u < sg.b; ++u, ++it) {
                const int s = it % p.stages;
                mbar_wait(&full[s], (it / p.stages) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                fence_proxy_async_smem();   // token operands arrived through the generic proxy
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t wa = smem_u32(smem + s * slot_bytes);
                    const uint32_t xa = wa + kClWArea;
                    uint32_t acc = (started >> sg.region) & 1;
                    if (sg.kind != kStExpand) {
                        const int nkb = sg.kind == kStShrink ? 4 : 2;
                        for (int kb = 0; kb < nkb; ++kb) {
                            const uint32_t a_kb = wa + kb * arows * kBK * 2;
                            const uint32_t x_kb = xa + kb * T * kBK * 2;
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk) {
                                umma_bf16(d, umma_sdesc(a_kb + kk * 32, 1024, kSwizzle128),
                                          umma_sdesc(x_kb + kk * 32, 1024, kSwizzle128), idesc, acc);
                                acc = 1;
                            }
                        }
                    } else {
                        for (int j = 0; j < kStWin; ++j) {
                            umma_bf16(d, umma_sdesc(wa + j * kSplitBN * kChunk * 2, 256, kSwizzle32),
                                      umma_sdesc(xa + j * T * kChunk * 2, 256, kSwizzle32), idesc, acc);
                            acc = 1;
                        }
                    }
                    umma_commit(&empty[s]);
                }
                started |= 1u << sg.region;
                __syncwarp();
            }
            if (sg.last) {
                if (lane == 0) umma_commit(&acc_full[sg.region]);
                __syncwarp();
            }
        }
    } else {
        // ===================== epilogue (warps 2..5) =========================
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int et = threadIdx.x - 64;
        // zero my slice of the other epoch's group sums and counters
        {
            float *acc_next = p.acc + static_cast<int64_t>(ep ^ 1) * p.max_groups * 32 * T;
            const int64_t nf = static_cast<int64_t>(p.max_groups) * 32 * T / 4;
            const int64_t f0 = nf * cta / G, f1 = nf * (cta + 1) / G;
            for (int64_t i = f0 + et; i < f1; i += 128)
                reinterpret_cast<float4 *>(acc_next)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            int32_t *gcnt_next = p.gcnt + (ep ^ 1) * p.max_groups;
            const int c0 = p.max_groups * cta / G, c1 = p.max_groups * (cta + 1) / G;
            for (int i = c0 + et; i < c1; i += 128) gcnt_next[i] = 0;
        }
        // shrink runs: add my partial to the group sums, then release
        for (int si = 0; si < ns; ++si) {
            const StSeg sg = segs[si];
            if (sg.kind != kStShrink) continue;
            if (quad != 0) continue;   // the group's rows (<= 32) live in TMEM lanes 0..31
            mbar_wait(&acc_full[sg.region], 0, abort_flag, status, LORA_DEV_TIMEOUT);
            tc_fence_after();
            const uint32_t tbase = tmem_base + sg.region * T;
            float *accum = acc_cur + static_cast<int64_t>(sg.g) * T * 32 + row;
            for (int c = 0; c < T; c += 16) {
                uint32_t v[16];
                tmem_ld16(tbase + c, v);
                tmem_ld_wait16(v);
                if (row < sg.rows) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) atomicAdd(accum + (c + e) * 32, __uint_as_float(v[e]));
                }
            }
            // each row's thread releases its own additions: the group is
            // complete once contributors x rows arrivals are in
            if (row < sg.rows) red_release_gpu_add(gcnt_cur + sg.g, 1);
        }
        // ---- output tile: push my partial rows to their owners ----------------
        mbar_wait(&acc_full[0], 0, abort_flag, status, LORA_DEV_TIMEOUT);
        tc_fence_after();
        const bool empty_run = segs[ns - 1].kind == kStNone;   // nothing accumulated: send zeros
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
        cluster_arrive();      // done with distributed shared memory
        const int groups = rpo / 8;
        for (int w = et; w < T * groups; w += 128) {
            const int t = w / groups, gq = w % groups;
            const int rloc = gq * 8;
            const int n = n0 + q * rpo + rloc;
            float sum[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) sum[e] = 0.f;
            for (int c = 0; c < C; ++c) {
                const float *src = red + (c * rpo + rloc) * T + t;
#pragma unroll
                for (int e = 0; e < 8; ++e) sum[e] += src[e * T];
            }
            if (t < p.M && n < p.N) {
                if (p.bias) {
                    const uint4 b = __ldg(reinterpret_cast<const uint4 *>(p.bias + n));
                    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        sum[2 * e] += bf16_lo(bw[e]);
                        sum[2 * e + 1] += bf16_hi(bw[e]);
                    }
                }
                *reinterpret_cast<uint4 *>(p.y + static_cast<int64_t>(t) * p.N + n) =
                    make_uint4(pack_bf16x2(sum[0], sum[1]), pack_bf16x2(sum[2], sum[3]), pack_bf16x2(sum[4], sum[5]),
                               pack_bf16x2(sum[6], sum[7]));
            }
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
    if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
    cluster_wait();            // no CTA leaves while a peer may still touch its shared memory
}

int cluster_max_regions() { return kStMaxRegions; }
int cluster_win() { return kStWin; }

size_t cluster_smem_bytes(int T_pad, int stages)
{
    return static_cast<size_t>(stages) * (kClWArea + T_pad * 512) + static_cast<size_t>(kSplitBN) * T_pad * 4 +
           1024 + 2048;
}

int cluster_stages(int T_pad)
{
    const size_t budget = 227 * 1024 - static_cast<size_t>(kSplitBN) * T_pad * 4 - 1024 - 2048;
    int s = static_cast<int>(budget / (kClWArea + T_pad * 512));
    return s > 6 ? 6 : s;
}

// Largest cluster size in {8, 4, 2, 1} whose grid (C x NT CTAs, one per SM)
// can be resident all at once; 0 when none can.
int cluster_pick_size(int NT, int T_pad, int sms)
{
    const int stages = cluster_stages(T_pad);
    if (stages < 2) return 0;
    const size_t smem = cluster_smem_bytes(T_pad, stages);
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !configured[dev]) {
        if (cudaFuncSetAttribute(lora_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(227 * 1024)) != cudaSuccess)
            return 0;
        if (dev < 64) configured[dev] = 1;
    }
    for (int C = 8; C >= 1; C >>= 1) {
        if (C * NT > sms) continue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C * NT);
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
        if (nclusters >= NT) return C;
    }
    return 0;
}

cudaError_t launch_cluster(const ClusterMaps &m, const ClusterParams &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.C * p.NT);
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = cluster_smem_bytes(p.T_pad, p.stages);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lora_cluster_kernel, m.w3, m.a3_16, m.a3_32, m.b3, p);
}

}  // namespace lora
