// Split-K (weight-streaming) schedule of the fused multi-LoRA linear layer
// for decode-sized batches (M <= 128 tokens).
//
// Page "vLLM-Ascend dynamic LoRA" (pptc.cn/news/149022): §1.2 (a decode step
// has one token per sequence, so per-request GEMMs have M of 1 and leave the
// matrix unit idle), §4.2 #3 (adapters concatenated so A is loaded as one
// [sum r, K] block), §2.2 (S = x A^T before S B^T), §2.3 (one dispatch).
//
// At this size the layer is bound by streaming W (and the A/B panels of the
// adapters present) from HBM once, so the MMA is swapped: the 128-row UMMA
// operand is a weight tile and the tokens form the N side (16..128), which
// keeps the tensor core's M dimension full.  Three lists of units, each unit
// one 64-wide K block (or four 16-wide rank panels):
//   L1 shrink : tile = 128 rows of the concatenated A panels of all adapters
//               present;  D[a_row, t] += A_cat[a_row, k] x[t, k]
//   L2 base   : tile = 128 output features;  D[n, t] += W[n, k] x[t, k]
//   L3 expand : tile = 128 output features;  D[n, t] += B_cat[n, r] S[t, r]
// Every CTA of the persistent grid takes an equal contiguous slice of L1,
// then of L2, then of L3, so the shrink is finished grid-wide long before
// any CTA reaches its expand units.  Each run of units that share a tile is
// accumulated in TMEM and written as an fp32 partial; the CTA whose arrival
// completes a tile's count sums the partials in a fixed order (deterministic
// for any timing) and finishes it:
//   shrink tile -> mask each token to its own adapter, * scale, bf16 S panels
//   output tile -> + bias, bf16, y[t, n]
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

constexpr int kSkThreads = 192;
constexpr int kSkASlot = kSplitBN * kBK * 2;   // 16 KB: W / A_cat K-block or 4 B panels
constexpr int kSkAPanel = kChunk * kBK * 2;    // 2 KB: 16 rows of A x 64
constexpr int kSkBPanel = kSplitBN * kChunk * 2;   // 4 KB: 128 rows of B x 16

struct ListGeo {
    int64_t U;   // units
    int TL;      // units per tile
    int tiles;
};

__device__ __forceinline__ int64_t slice_begin(const ListGeo &g, int c, int G)
{
    return (g.U * c) / G;
}

// CTA whose slice holds unit u (slices are monotone; empty ones are skipped).
__device__ __forceinline__ int owner_of(const ListGeo &g, int64_t u, int G)
{
    return static_cast<int>(((u + 1) * G - 1) / g.U);
}

__device__ __forceinline__ int64_t slot_of(const ListGeo &g, int list_base, int R, int c, int tile, int G)
{
    const int first_tile = static_cast<int>(slice_begin(g, c, G) / g.TL);
    return static_cast<int64_t>(list_base) + static_cast<int64_t>(c) * R + (tile - first_tile);
}

struct Geos {
    ListGeo l[3];
    int D;       // chunks (16-row A panels / 16-col B panels) of adapters present
    int RT;      // shrink tiles
};

__device__ __forceinline__ Geos make_geos(const SplitParams &p)
{
    Geos g;
    g.D = p.hdr[HDR_DCHUNKS];
    g.RT = (g.D + 7) / 8;
    const int EU = (g.D + 3) / 4;
    g.l[0] = {static_cast<int64_t>(g.RT) * p.kblocks, p.kblocks, g.RT};
    g.l[1] = {static_cast<int64_t>(p.NT) * p.kblocks, p.kblocks, p.NT};
    g.l[2] = {static_cast<int64_t>(p.NT) * EU, EU > 0 ? EU : 1, EU > 0 ? p.NT : 0};
    if (EU == 0) g.l[2].U = 0;
    return g;
}

// Number of CTAs with a non-empty slice intersecting `tile` of list g.
__device__ __forceinline__ int contributors(const ListGeo &g, int tile, int G)
{
    if (g.U == 0) return 0;
    const int64_t a = static_cast<int64_t>(tile) * g.TL, b = a + g.TL - 1;
    const int c0 = owner_of(g, a, G), c1 = owner_of(g, b, G);
    int n = 0;
    for (int c = c0; c <= c1; ++c)
        if (slice_begin(g, c + 1, G) > slice_begin(g, c, G)) ++n;
    return n;
}

__global__ void __launch_bounds__(kSkThreads, 1)
    lora_splitk_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                       const __grid_constant__ CUtensorMap tm_s, const SplitParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stage_bytes = kSkASlot + p.T_pad * kBK * 2;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.stages * stage_bytes);
    uint64_t *empty = full + p.stages;
    uint64_t *acc_full = empty + p.stages;
    uint64_t *acc_empty = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *bcast = const_cast<int *>(abort_flag) + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    int32_t *status = p.counters + CNT_STATUS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 128);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tm_x);
        tma_prefetch_map(&tm_w);
        tma_prefetch_map(&tm_a);
        tma_prefetch_map(&tm_b);
        tma_prefetch_map(&tm_s);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Geos geo = make_geos(p);
    const int list_base[3] = {0, G * p.R1, G * (p.R1 + p.R2)};
    const int list_R[3] = {p.R1, p.R2, p.R3};

    if (warp == 0) {
        // ===================== TMA producer ==================================
        uint32_t it = 0;
        for (int L = 0; L < 3; ++L) {
            const ListGeo &g = geo.l[L];
            if (g.U == 0) continue;
            const int64_t u0 = slice_begin(g, cta, G), u1 = slice_begin(g, cta + 1, G);
            if (L == 2 && u1 > u0) {
                if (lane == 0) {
                    wait_flag_geq(p.counters + CNT_SPLIT_SREADY, geo.RT, abort_flag, status, LORA_DEV_TIMEOUT);
                    fence_proxy_async_global();
                }
                __syncwarp();
            }
            for (int64_t u = u0; u < u1; ++u, ++it) {
                const int tile = static_cast<int>(u / g.TL), k = static_cast<int>(u % g.TL);
                const int s = it % p.stages;
                const uint32_t round = it / p.stages;
                if (lane == 0 && round > 0) mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                __syncwarp();
                uint8_t *as = smem + s * stage_bytes;
                uint8_t *bs = as + kSkASlot;
                if (L == 0) {
                    const int g0 = tile * 8, nch = min(8, geo.D - g0);
                    if (lane == 0) {
                        mbar_expect_tx(&full[s], nch * kSkAPanel + p.T_pad * kBK * 2);
                        tma_load_2d(bs, &tm_x, &full[s], k * kBK, 0);
                    }
                    __syncwarp();
                    if (lane < nch) tma_load_2d(as + lane * kSkAPanel, &tm_a, &full[s], k * kBK, p.dchunk_arow[g0 + lane]);
                } else if (L == 1) {
                    if (lane == 0) {
                        mbar_expect_tx(&full[s], kSkASlot + p.T_pad * kBK * 2);
                        tma_load_2d(as, &tm_w, &full[s], k * kBK, tile * kSplitBN);
                        tma_load_2d(bs, &tm_x, &full[s], k * kBK, 0);
                    }
                } else {
                    const int g0 = k * 4, nch = min(4, geo.D - g0);
                    if (lane == 0) mbar_expect_tx(&full[s], nch * (kSkBPanel + p.T_pad * kChunk * 2));
                    __syncwarp();
                    if (lane < nch) {
                        tma_load_2d(as + lane * kSkBPanel, &tm_b, &full[s], 0, p.dchunk_brow[g0 + lane] + tile * kSplitBN);
                        tma_load_2d(bs + lane * p.T_pad * kChunk * 2, &tm_s, &full[s], 0, (g0 + lane) * p.T_pad);
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ===================== MMA issuer ====================================
        uint32_t it = 0, q = 0;
        const uint32_t idesc = umma_idesc_bf16(kSplitBN, p.T_pad);
        for (int L = 0; L < 3; ++L) {
            const ListGeo &g = geo.l[L];
            if (g.U == 0) continue;
            const int64_t u0 = slice_begin(g, cta, G), u1 = slice_begin(g, cta + 1, G);
            int64_t u = u0;
            while (u < u1) {
                const int tile = static_cast<int>(u / g.TL);
                const int64_t run_end = min(u1, static_cast<int64_t>(tile + 1) * g.TL);
                const uint32_t slot = q & 1, use = q >> 1;
                if (use > 0) mbar_wait(&acc_empty[slot], (use - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                tc_fence_after();
                const uint32_t d = tmem_base + slot * p.T_pad;
                uint32_t acc = 0;
                for (; u < run_end; ++u, ++it) {
                    const int k = static_cast<int>(u % g.TL);
                    const int s = it % p.stages;
                    mbar_wait(&full[s], (it / p.stages) & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t aa = smem_u32(smem + s * stage_bytes);
                        const uint32_t ba = aa + kSkASlot;
                        if (L < 2) {
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk) {
                                umma_bf16(d, umma_sdesc(aa + kk * 32, 1024, kSwizzle128),
                                          umma_sdesc(ba + kk * 32, 1024, kSwizzle128), idesc, acc);
                                acc = 1;
                            }
                        } else {
                            const int nch = min(4, geo.D - k * 4);
                            for (int i = 0; i < nch; ++i) {
                                umma_bf16(d, umma_sdesc(aa + i * kSkBPanel, 256, kSwizzle32),
                                          umma_sdesc(ba + i * p.T_pad * kChunk * 2, 256, kSwizzle32), idesc, acc);
                                acc = 1;
                            }
                        }
                        umma_commit(&empty[s]);
                    }
                    __syncwarp();
                }
                if (lane == 0) umma_commit(&acc_full[slot]);
                __syncwarp();
                ++q;
            }
        }
    } else {
        // ===================== epilogue: partials + reductions ===============
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int et = threadIdx.x - 64;
        const int T = p.T_pad;
        uint32_t q = 0;
        for (int L = 0; L < 3; ++L) {
            const ListGeo &g = geo.l[L];
            if (g.U == 0) continue;
            const int64_t u0 = slice_begin(g, cta, G), u1 = slice_begin(g, cta + 1, G);
            int64_t u = u0;
            while (u < u1) {
                const int tile = static_cast<int>(u / g.TL);
                u = min(u1, static_cast<int64_t>(tile + 1) * g.TL);
                const uint32_t slot = q & 1, use = q >> 1;
                ++q;
                mbar_wait(&acc_full[slot], use & 1, abort_flag, status, LORA_DEV_TIMEOUT);
                tc_fence_after();
                const uint32_t tbase = tmem_base + slot * T + (static_cast<uint32_t>(quad * 32) << 16);
                float *mine = p.partials + slot_of(g, list_base[L], list_R[L], cta, tile, G) * (kSplitBN * T) +
                              static_cast<int64_t>(row) * T;
                for (int c = 0; c < T; c += 16) {
                    uint32_t r[16];
                    tmem_ld16(tbase + c, r);
                    tmem_ld_wait16(r);
                    float4 *dst = reinterpret_cast<float4 *>(mine + c);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                             __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                }
                tc_fence_before();
                mbar_arrive(&acc_empty[slot]);
                __threadfence();
                named_bar_sync(1, 128);
                const bool is_out = (L != 0);
                int32_t *cnt = p.counters + CNT_FIXED + (is_out ? tile : p.NT + tile);
                if (et == 0) {
                    const int expect = is_out ? contributors(geo.l[1], tile, G) + contributors(geo.l[2], tile, G)
                                              : contributors(geo.l[0], tile, G);
                    *bcast = (atom_acq_rel_gpu_add(cnt, 1) == expect - 1);
                }
                named_bar_sync(1, 128);
                if (!*bcast) continue;
                __threadfence();
                // ---- this CTA completes the tile: fixed-order sum of partials
                const int lists[2] = {is_out ? 1 : 0, is_out ? 2 : -1};
                for (int c = 0; c < T; c += 16) {
                    float acc16[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc16[e] = 0.f;
                    for (int li = 0; li < 2; ++li) {
                        const int LL = lists[li];
                        if (LL < 0) continue;
                        const ListGeo &gg = geo.l[LL];
                        if (gg.U == 0) continue;
                        const int64_t a = static_cast<int64_t>(tile) * gg.TL;
                        const int cfirst = owner_of(gg, a, G), clast = owner_of(gg, a + gg.TL - 1, G);
                        for (int cc = cfirst; cc <= clast; ++cc) {
                            if (slice_begin(gg, cc + 1, G) <= slice_begin(gg, cc, G)) continue;
                            const float4 *src = reinterpret_cast<const float4 *>(
                                p.partials + slot_of(gg, list_base[LL], list_R[LL], cc, tile, G) * (kSplitBN * T) +
                                static_cast<int64_t>(row) * T + c);
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const float4 f = __ldcg(src + v);
                                acc16[4 * v] += f.x;
                                acc16[4 * v + 1] += f.y;
                                acc16[4 * v + 2] += f.z;
                                acc16[4 * v + 3] += f.w;
                            }
                        }
                    }
                    if (is_out) {
                        const int n = tile * kSplitBN + row;
                        if (n < p.N) {
                            const float b = p.bias ? __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16) : 0.f;
                            for (int e = 0; e < 16; ++e) {
                                const int t = c + e;
                                if (t < p.M) {
                                    const uint32_t h = pack_bf16x2(acc16[e] + b, 0.f);
                                    p.y[static_cast<int64_t>(t) * p.N + n] = static_cast<uint16_t>(h & 0xFFFF);
                                }
                            }
                        }
                    } else {
                        const int arow = tile * kSplitBN + row;
                        const int gch = arow / kChunk;
                        if (gch < geo.D) {
                            const int adapter = p.dchunk_adapter[gch];
                            uint16_t *dst = p.s_panels + (static_cast<int64_t>(gch) * T) * kChunk + (arow % kChunk);
                            for (int e = 0; e < 16; ++e) {
                                const int t = c + e;
                                float v = 0.f;
                                if (t < p.M) {
                                    const int id = p.ids[t];
                                    if (id == adapter) v = acc16[e] * p.scale;
                                }
                                const uint32_t h = pack_bf16x2(v, 0.f);
                                dst[static_cast<int64_t>(t) * kChunk] = static_cast<uint16_t>(h & 0xFFFF);
                            }
                        }
                    }
                }
                if (!is_out) {
                    fence_proxy_async_global();
                    __threadfence();
                }
                named_bar_sync(1, 128);
                if (et == 0) {
                    *cnt = 0;
                    if (!is_out) red_release_gpu_add(p.counters + CNT_SPLIT_SREADY, 1);
                }
            }
        }
    }

    // ---- teardown ---------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
    if (threadIdx.x == 0) {
        __threadfence();
        if (atom_acq_rel_gpu_add(p.counters + CNT_SPLIT_DONE, 1) == G - 1) {
            p.counters[CNT_SPLIT_SREADY] = 0;
            p.counters[CNT_SPLIT_DONE] = 0;
        }
    }
}

size_t splitk_smem_bytes(int T_pad, int stages)
{
    return static_cast<size_t>(stages) * (kSkASlot + T_pad * kBK * 2) + 1024 + 256;
}

int splitk_stages(int T_pad)
{
    const int stage = kSkASlot + T_pad * kBK * 2;
    int s = (200 * 1024) / stage;
    return s > 12 ? 12 : s;
}

cudaError_t launch_splitk(const TcMaps &maps, const SplitParams &p, int grid, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = splitk_smem_bytes(p.T_pad, p.stages);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(lora_splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             220 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    lora_splitk_kernel<<<grid, kSkThreads, smem, stream>>>(maps.x, maps.w, maps.a, maps.b, maps.s, p);
    return cudaGetLastError();
}

}  // namespace lora
