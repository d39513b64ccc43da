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
// keeps the tensor core's M dimension full.  Units of work (one 64-wide K
// block, or four 16-wide rank panels) come in two lists:
//   shrink list : tile = 128 rows of the concatenated A panels of all adapters
//                 present;  D[a_row, t] += A_cat[a_row, k] x[t, k]
//   output list : tile = 128 output features; its units are the K blocks of
//                 the base product  D[n, t] += W[n, k] x[t, k]  followed by
//                 the expand steps  D[n, t] += B_cat[n, r] S[t, r]
// Every CTA of the persistent grid takes an equal contiguous slice of the
// shrink list, then of the output list, so the shrink is finished grid-wide
// long before the expand steps need it; a run of a slice whose first unit is
// an expand step is moved behind the CTA's other runs.  Each run (units of
// one tile) is accumulated in TMEM and added with fp32 vector atomics into a
// per-tile accumulator in L2; the CTA whose arrival completes the tile's
// count reads it once and finishes it:
//   shrink tile -> mask each token to its own adapter, * scale, bf16 S panels
//   output tile -> + bias, bf16, y[t, n]
// and zeroes the accumulator and counter for the next call.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

constexpr int kSkThreads = 192;
constexpr int kSkASlot = kSplitBN * kBK * 2;       // 16 KB: W / A_cat K-block or 4 B panels
constexpr int kSkAPanel = kChunk * kBK * 2;        // 2 KB: 16 rows of A x 64
constexpr int kSkBPanel = kSplitBN * kChunk * 2;   // 4 KB: 128 rows of B x 16
constexpr int kMaxRuns = 64;

struct ListGeo {
    int64_t U;   // units
    int TL;      // units per tile
};

__device__ __forceinline__ int64_t slice_begin(const ListGeo &g, int c, int G) { return (g.U * c) / G; }

// CTA whose slice holds unit u (slices are monotone; empty ones are skipped).
__device__ __forceinline__ int owner_of(const ListGeo &g, int64_t u, int G)
{
    return static_cast<int>(((u + 1) * G - 1) / g.U);
}

// Number of CTAs with a non-empty slice intersecting `tile`.
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

struct Run {
    int list;       // 0 shrink, 1 output
    int tile;
    int u0, u1;     // unit range inside the tile: [u0, u1)
};

__global__ void __launch_bounds__(kSkThreads, 1)
    lora_splitk_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                       const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_a32,
                       const __grid_constant__ CUtensorMap tm_a48, const __grid_constant__ CUtensorMap tm_a64,
                       const SplitParams p)
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
    int *n_runs = bcast + 1;
    Run *runs = reinterpret_cast<Run *>(n_runs + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    int32_t *status = p.counters + CNT_STATUS;
    const long long wait = p.wait_cycles;

    // rank panels of the adapters present (LORA_DEBUG build: none when the
    // segment table failed its check; the base product alone is computed)
    const int D = kDebugChecks && p.hdr[HDR_CHECK] != 0 ? 0 : p.hdr[HDR_DCHUNKS];
    const int RT = (D + 7) / 8;                     // shrink tiles (8 panels = 128 rows)
    const int EU = (D + 3) / 4;                     // expand units per output tile
    const ListGeo g_shr = {static_cast<int64_t>(RT) * p.kblocks, p.kblocks};
    const ListGeo g_out = {static_cast<int64_t>(p.NT) * (p.kblocks + EU), p.kblocks + EU};

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
        // this CTA's runs: shrink slice, then output slice
        int n = 0;
        const ListGeo *gs[2] = {&g_shr, &g_out};
        int first_out = -1;
        for (int L = 0; L < 2; ++L) {
            const ListGeo &g = *gs[L];
            if (g.U == 0) continue;
            const int64_t u1 = slice_begin(g, cta + 1, G);
            for (int64_t u = slice_begin(g, cta, G); u < u1 && n < kMaxRuns;) {
                const int tile = static_cast<int>(u / g.TL);
                const int64_t e = min(u1, static_cast<int64_t>(tile + 1) * g.TL);
                if (L == 1 && first_out < 0) first_out = n;
                runs[n++] = {L, tile, static_cast<int>(u - static_cast<int64_t>(tile) * g.TL),
                             static_cast<int>(e - static_cast<int64_t>(tile) * g.TL)};
                u = e;
            }
        }
        // an output run that starts with expand steps goes last
        if (first_out >= 0 && n - first_out > 1 && runs[first_out].u0 >= p.kblocks) {
            const Run r = runs[first_out];
            for (int i = first_out; i < n - 1; ++i) runs[i] = runs[i + 1];
            runs[n - 1] = r;
        }
        *n_runs = n;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tm_x);
        tma_prefetch_map(&tm_w);
        tma_prefetch_map(&tm_a);
        tma_prefetch_map(&tm_a64);
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
    const int nr = *n_runs;

    if (warp == 0) {
        // ===================== TMA producer ==================================
        uint32_t it = 0;
        bool s_ready = false;
        for (int ri = 0; ri < nr; ++ri) {
            const Run r = runs[ri];
            for (int k = r.u0; k < r.u1; ++k, ++it) {
                const bool expand = r.list == 1 && k >= p.kblocks;
                if (expand && !s_ready) {
                    if (lane == 0) {
                        wait_flag_geq(p.counters + CNT_SPLIT_SREADY, RT, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                        fence_proxy_async_global();
                    }
                    __syncwarp();
                    s_ready = true;
                }
                const int s = it % p.stages;
                const uint32_t round = it / p.stages;
                // the slot's full barrier gets this stage's arrive only once its
                // previous phase has completed (immediate in a healthy run), so
                // the arrive opens a new phase also after a timeout let a wait
                // go early; a stage whose slot never comes free is skipped
                int ok = 1;
                if (lane == 0 && round > 0) {
                    mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                    ok = mbar_wait(&full[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) continue;
                uint8_t *as = smem + s * stage_bytes;
                uint8_t *bs = as + kSkASlot;
                if (r.list == 0) {
                    const int g0 = r.tile * 8, g1 = min(g0 + 8, D);
                    if (lane == 0) {
                        mbar_expect_tx(&full[s], (g1 - g0) * kSkAPanel + p.T_pad * kBK * 2);
                        tma_load_2d(bs, &tm_x, &full[s], k * kBK, 0);
                        // consecutive panels of one adapter: one box of 16..64 rows
                        for (int g = g0; g < g1;) {
                            const int r0 = p.dchunk_arow[g];
                            int len = 1;
                            while (len < 4 && g + len < g1 && p.dchunk_arow[g + len] == r0 + kChunk * len) ++len;
                            const CUtensorMap *m = len == 1 ? &tm_a : len == 2 ? &tm_a32 : len == 3 ? &tm_a48 : &tm_a64;
                            tma_load_2d(as + (g - g0) * kSkAPanel, m, &full[s], k * kBK, r0);
                            g += len;
                        }
                    }
                } else if (!expand) {
                    if (lane == 0) {
                        mbar_expect_tx(&full[s], kSkASlot + p.T_pad * kBK * 2);
                        tma_load_2d(as, &tm_w, &full[s], k * kBK, r.tile * kSplitBN);
                        tma_load_2d(bs, &tm_x, &full[s], k * kBK, 0);
                    }
                } else {
                    const int g0 = (k - p.kblocks) * 4, nch = min(4, D - g0);
                    if (lane == 0) mbar_expect_tx(&full[s], nch * (kSkBPanel + p.T_pad * kChunk * 2));
                    __syncwarp();
                    if (lane < nch) {
                        tma_load_2d(as + lane * kSkBPanel, &tm_b, &full[s], 0, p.dchunk_bpanel[g0 + lane] * p.N + r.tile * kSplitBN);
                        tma_load_2d(bs + lane * p.T_pad * kChunk * 2, &tm_s, &full[s], 0, (g0 + lane) * p.T_pad);
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0) n_runs[1] = static_cast<int>(it);   // for the teardown: the stages issued
        __syncwarp();
    } else if (warp == 1) {
        // ===================== MMA issuer ====================================
        uint32_t it = 0;
        const uint32_t idesc = umma_idesc_bf16(kSplitBN, p.T_pad);
        for (int ri = 0; ri < nr; ++ri) {
            const Run r = runs[ri];
            const uint32_t slot = ri & 1, use = ri >> 1;
            if (use > 0) mbar_wait(&acc_empty[slot], (use - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
            tc_fence_after();
            const uint32_t d = tmem_base + slot * p.T_pad;
            uint32_t acc = 0;
            for (int k = r.u0; k < r.u1; ++k, ++it) {
                const bool expand = r.list == 1 && k >= p.kblocks;
                const int s = it % p.stages;
                mbar_wait(&full[s], (it / p.stages) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t aa = smem_u32(smem + s * stage_bytes);
                    const uint32_t ba = aa + kSkASlot;
                    if (!expand) {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            umma_bf16(d, umma_sdesc(aa + kk * 32, 1024, kSwizzle128),
                                      umma_sdesc(ba + kk * 32, 1024, kSwizzle128), idesc, acc);
                            acc = 1;
                        }
                    } else {
                        const int nch = min(4, D - (k - p.kblocks) * 4);
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
        }
        __syncwarp();
    } else {
        // ===================== epilogue: accumulate, finish tiles =============
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int et = threadIdx.x - 64;
        const int T = p.T_pad;
        for (int ri = 0; ri < nr; ++ri) {
            const Run r = runs[ri];
            const uint32_t slot = ri & 1, use = ri >> 1;
            mbar_wait(&acc_full[slot], use & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
            tc_fence_after();
            const uint32_t tbase = tmem_base + slot * T + (static_cast<uint32_t>(quad * 32) << 16);
            const bool is_out = r.list == 1;
            float *accum = (is_out ? p.acc_out : p.acc_shr) + (static_cast<int64_t>(r.tile) * kSplitBN + row) * T;
            for (int c = 0; c < T; c += 16) {
                uint32_t v[16];
                tmem_ld16(tbase + c, v);
                tmem_ld_wait16(v);
                float4 *dst = reinterpret_cast<float4 *>(accum + c);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    atomicAdd(dst + q, make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[slot]);
            __threadfence();
            named_bar_sync(1, 128);
            int32_t *cnt = p.counters + CNT_FIXED + (is_out ? r.tile : p.NT + r.tile);
            if (et == 0) {
                const int expect = contributors(is_out ? g_out : g_shr, r.tile, G);
                *bcast = (atom_acq_rel_gpu_add(cnt, 1) == expect - 1);
            }
            named_bar_sync(1, 128);
            if (!*bcast) continue;
            __threadfence();
            // ---- last arrival: the tile's sum is complete in `accum` ----------
            const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c = 0; c < T; c += 16) {
                float a[16];
                float4 *src = reinterpret_cast<float4 *>(accum + c);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 f = __ldcg(src + q);
                    a[4 * q] = f.x;
                    a[4 * q + 1] = f.y;
                    a[4 * q + 2] = f.z;
                    a[4 * q + 3] = f.w;
                    __stcg(src + q, zero4);
                }
                if (is_out) {
                    const int n = r.tile * kSplitBN + row;
                    if (n < p.N) {
                        const float b = p.bias ? __uint_as_float(static_cast<uint32_t>(p.bias[n]) << 16) : 0.f;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int t = c + e;
                            if (t < p.M)
                                p.y[static_cast<int64_t>(t) * p.N + n] =
                                    static_cast<uint16_t>(pack_bf16x2(a[e] + b, 0.f) & 0xFFFF);
                        }
                    }
                } else {
                    const int arow = r.tile * kSplitBN + row;
                    const int gch = arow / kChunk;
                    if (gch < D) {
                        const int adapter = p.dchunk_adapter[gch];
                        const float sc = p.adapter_scale ? p.scale * p.adapter_scale[adapter] : p.scale;
                        uint16_t *dst = p.s_panels + static_cast<int64_t>(gch) * T * kChunk + (arow % kChunk);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int t = c + e;
                            const float v = (t < p.M && p.ids[t] == adapter) ? a[e] * sc : 0.f;
                            dst[static_cast<int64_t>(t) * kChunk] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFF);
                        }
                    }
                }
            }
            if (!is_out) fence_proxy_async_global();
            __threadfence();
            named_bar_sync(1, 128);
            if (et == 0) {
                *cnt = 0;
                if (!is_out) red_release_gpu_add(p.counters + CNT_SPLIT_SREADY, 1);
            }
        }
    }

    // ---- teardown ---------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // After a timeout let a wait of this CTA go early, its loads and MMAs
    // still in flight are waited for (bounded) before the tensor memory is
    // freed and the CTA ends: the last phase of each stage and the last
    // commit, which covers every MMA.  In a healthy run every one of them has
    // been waited for already.
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t it = static_cast<uint32_t>(n_runs[1]), ns = static_cast<uint32_t>(p.stages);
            for (uint32_t i = it > ns ? it - ns : 0; i < it; ++i)
                mbar_wait(&full[i % ns], (i / ns) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
        }
        if (warp == 1 && lane == 0 && nr > 0)
            mbar_wait(&acc_full[(nr - 1) & 1], ((nr - 1) >> 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
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
    return static_cast<size_t>(stages) * (kSkASlot + T_pad * kBK * 2) + 1024 + 256 + kMaxRuns * sizeof(Run);
}

int splitk_stages(int T_pad)
{
    const int stage = kSkASlot + T_pad * kBK * 2;
    int s = (200 * 1024) / stage;
    return s > 12 ? 12 : s;
}

int splitk_max_runs() { return kMaxRuns; }

cudaError_t launch_splitk(const TcMaps &maps, const SplitParams &p, int grid, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = splitk_smem_bytes(p.T_pad, p.stages);
    if (dev >= 64 || !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(lora_splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             220 * 1024);
        if (e != cudaSuccess) return e;
        if (dev < 64) configured[dev] = 1;
    }
    lora_splitk_kernel<<<grid, kSkThreads, smem, stream>>>(maps.x, maps.w, maps.a, maps.b, maps.s, maps.a32, maps.a48,
                                                           maps.a64, p);
    return cudaGetLastError();
}

}  // namespace lora
