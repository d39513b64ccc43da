// Grouped expert GEMM of a mixture-of-experts layer, two token tiles of one
// expert per work item.
//
// Page "Qwen3-MoE low-latency inference on Atlas A3" (mokono.cn/news/2297686),
// its MoE section: the (token, slot) pairs, sorted by expert, go through one
// grouped matmul, each expert's rows against that expert's weights.
//
// The routing pads each expert's pairs to whole 128-row tiles of the padded
// order, an expert's tiles consecutive.  A work item here is one column tile
// (256 output features) of one expert and up to two consecutive token tiles
// of that expert: every K step's weight box (32 KB) feeds the MMAs of both
// tiles, so a stage of shared memory carries half the weight bytes per MMA
// of the tiled kernel's expert mode (one token tile per item), whose K steps
// measured bound by how fast one SM takes in its stages.  The two 128x256
// fp32 accumulators fill the TMEM, so an item's epilogue does not overlap the
// next item's K loop.  Items run in the one-group order: every tile pair of
// column tile n, then n + 1, so the pairs that read one weight tile run in
// the same wave and it comes from HBM once.
//
// Roles (320 threads): warp 0 TMA producer (the weight box of each K step),
// warp 1 TMEM allocator + MMA issuer, warps 2..5 epilogue (warp 2 first
// builds the item list), warps 6..9 gather both token tiles' x rows
// (cp.async, a pair's token is pair / topk).  Shared memory: 3 stages of
// [x 32 KB | W 32 KB] under one full and one empty barrier each, and the
// item list.  Every wait is bounded.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "moe_pair.h"
#include "ptx.cuh"

namespace lora {

constexpr int kMpThreads = 320;
constexpr int kMpStages = 3;
constexpr int kMpXHalf = kBM * kBK * 2;       // one 128-row x tile of a K step, 16 KB
constexpr int kMpXSlot = 2 * kMpXHalf;        // 32 KB
constexpr int kMpWSlot = kBN * kBK * 2;       // 32 KB
constexpr size_t kMpSmem =
    1024 /*align*/ + kMpStages * (kMpXSlot + kMpWSlot) + 256 /*barriers*/ + 2 * sizeof(int32_t) * kMoePairMaxTiles;
static_assert(kMpSmem <= 232448, "fits the opt-in shared memory of a CTA");

__global__ void __launch_bounds__(kMpThreads, 1) moe_pair_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                                  const MoePairParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xring = smem;                              // kMpStages x 32 KB: rows 0..127 tile m0, 128..255 tile m0 + 1
    uint8_t *wring = smem + kMpStages * kMpXSlot;       // kMpStages x 32 KB
    uint64_t *full = reinterpret_cast<uint64_t *>(wring + kMpStages * kMpWSlot);
    uint64_t *empty = full + kMpStages;
    uint64_t *acc_full = empty + kMpStages;
    uint64_t *acc_empty = acc_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *drain = const_cast<int *>(abort_flag) + 1;     // [0] stages the producer issued, [1] the MMA's last item
    int *n_pairs_s = drain + 2;
    // the item list: tile pair k starts at token tile s_pm[k] >> 1 and holds
    // (s_pm[k] & 1) + 1 tiles of expert s_pe[k]
    int32_t *s_pm = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(full) + 256);
    int32_t *s_pe = s_pm + kMoePairMaxTiles;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = p.status;
    const long long wait = p.wait_cycles;
    pdl_launch_dependents();   // the finalize may place its CTAs as this grid's CTAs leave

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMpStages; ++s) {
            mbar_init(&full[s], 128 + 1);   // a cp.async-completion arrive per loader thread, the producer's expect_tx
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 128);
        *abort_flag = 0;
        drain[0] = 0;
        drain[1] = -1;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_map(&tm_w);
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();   // the routing ahead of this kernel wrote the padded order and the tiles' experts

    if (warp == 2) {
        // The item list, one chunk of 32 token tiles at a time: a tile starts
        // a pair if it is an even number of tiles past its expert's first.
        const bool bad = kDebugChecks && p.hdr[HDR_CHECK] != 0;   // LORA_DEBUG: a routing that failed its check
        const int nt = bad ? 0 : min(p.hdr[HDR_MOE_TILES], min(p.max_mtiles, kMoePairMaxTiles));
        int npairs = 0, last_start = 0, carry_e = -1;
        for (int c0 = 0; c0 < nt; c0 += 32) {
            const int m = c0 + lane;
            const int e = m < nt ? p.mt_expert[m] : -1;
            const int up = __shfl_up_sync(0xffffffffu, e, 1);
            const int e_prev = lane == 0 ? carry_e : up;
            const bool start = m < nt && (m == 0 || e != e_prev);
            const unsigned starts = __ballot_sync(0xffffffffu, start);
            const unsigned upto = starts & ((2u << lane) - 1u);   // starts at or below this lane
            const int first = upto ? c0 + 31 - __clz(upto) : last_start;
            const bool pstart = m < nt && ((m - first) & 1) == 0;
            const unsigned pmask = __ballot_sync(0xffffffffu, pstart);
            const int down = __shfl_down_sync(0xffffffffu, e, 1);
            const int e_next = m + 1 >= nt ? -1 : lane == 31 ? p.mt_expert[m + 1] : down;
            if (pstart) {
                const int k = npairs + __popc(pmask & ((1u << lane) - 1u));
                s_pm[k] = 2 * m + (e_next == e ? 1 : 0);
                s_pe[k] = e;
            }
            npairs += __popc(pmask);
            last_start = __shfl_sync(0xffffffffu, first, 31);
            carry_e = __shfl_sync(0xffffffffu, e, 31);
        }
        if (lane == 0) *n_pairs_s = npairs;
    }
    __syncthreads();
    const int npairs = *n_pairs_s;
    const int n_items = npairs * p.num_ntiles;   // item i: tile pair i % npairs, column tile i / npairs

    if (warp == 0) {
        // ===================== TMA producer: the weight box of each K step ====
        if (lane == 0) {
            uint32_t it = 0;
            for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
                const int k = i % npairs, n = i / npairs;
                const int w_row = s_pe[k] * p.N + n * kBN;   // the expert's rows of the stacked weights
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const int s = it % kMpStages;
                    const uint32_t round = it / kMpStages;
                    // refill only once the MMA has freed the stage and its
                    // previous phase has completed (a stage whose wait gave
                    // up is skipped)
                    if (round > 0) {
                        mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                        if (!mbar_wait(&full[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait))
                            continue;
                    }
                    mbar_expect_tx(&full[s], kMpWSlot);
                    tma_load_2d(wring + s * kMpWSlot, &tm_w, &full[s], kb * kBK, w_row);
                }
            }
            drain[0] = static_cast<int>(it);
        }
    } else if (warp >= 6) {
        // ===================== x loaders: both tiles' rows (cp.async) =========
        // Thread lt copies 16-byte chunk (lt % 8) of slot rows lt / 8 + 16 q,
        // q < 16, into the 128-byte-swizzled x slot: rows 0..127 belong to
        // the pair's first tile, 128..255 to its second (zeros when the
        // pair has one tile, and for the padded order's gaps).
        const int lt = threadIdx.x - 192;
        const int chunk = lt & 7, rb = lt >> 3;
        const uint32_t swz = static_cast<uint32_t>((chunk ^ (rb & 7)) << 4);
        uint32_t it = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
            const int k = i % npairs;
            const int m0 = s_pm[k] >> 1, cnt = (s_pm[k] & 1) + 1;
            const uint16_t *src[16];
            uint32_t live = 0;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int h = q >> 3, r = rb + 16 * (q & 7);
                int pair = -1;
                if (h < cnt) pair = p.perm_pad[static_cast<int64_t>(m0 + h) * kBM + r];
                bool ok = pair >= 0;
                if (kDebugChecks && ok) ok = debug_index_ok(pair < p.out_rows, status);
                src[q] = p.x + static_cast<int64_t>(ok ? pair / p.topk : 0) * p.K + chunk * 8;
                live |= static_cast<uint32_t>(ok) << q;
            }
            for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                const int s = it % kMpStages;
                const uint32_t round = it / kMpStages;
                int ok = 1;   // as the producer: the stage's previous phase has completed
                if (lane == 0 && round > 0) {
                    mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                    ok = mbar_wait(&full[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) continue;
                uint8_t *xs = xring + s * kMpXSlot + swz;
                const bool k_in = kb * kBK + chunk * 8 < p.K;
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    cp_async16(xs + (rb + 16 * q) * 128, src[q] + kb * kBK, (k_in && ((live >> q) & 1u)) ? 16u : 0u);
                cp_async_mbar_arrive_noinc(&full[s]);
            }
        }
        cp_async_wait_all();
    } else if (warp == 1) {
        // ===================== MMA issuer ======================================
        const uint64_t xdesc0 = umma_sdesc(smem_u32(xring), 1024, kSwizzle128);
        const uint64_t wdesc0 = umma_sdesc(smem_u32(wring), 1024, kSwizzle128);
        const uint32_t idesc = umma_idesc_bf16(kBM, kBN);
        uint32_t it = 0;
        int q = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++q) {
            const int cnt = (s_pm[i % npairs] & 1) + 1;
            if (q > 0) mbar_wait(acc_empty, (q - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
            tc_fence_after();
            uint32_t acc = 0;
            for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                const int s = it % kMpStages;
                mbar_wait(&full[s], (it / kMpStages) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                fence_proxy_async_smem();   // x arrived through the generic proxy (cp.async)
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t xd = xdesc0 + static_cast<uint64_t>((s * kMpXSlot) >> 4);
                    const uint64_t wd = wdesc0 + static_cast<uint64_t>((s * kMpWSlot) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {   // 16 K columns of bf16 = 32 bytes
                        umma_bf16(tmem_base, xd + 2 * kk, wd + 2 * kk, idesc, acc);
                        if (cnt == 2)
                            umma_bf16(tmem_base + kBN, xd + (kMpXHalf >> 4) + 2 * kk, wd + 2 * kk, idesc, acc);
                        acc = 1;
                    }
                    umma_commit(&empty[s]);
                }
                __syncwarp();
            }
            if (lane == 0) {
                umma_commit(acc_full);
                drain[1] = q;
            }
            __syncwarp();
        }
    } else {
        // ===================== epilogue (warps 2..5): bf16 rows of both tiles ==
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        int q = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++q) {
            const int k = i % npairs, n = i / npairs;
            const int m0 = s_pm[k] >> 1, cnt = (s_pm[k] & 1) + 1;
            // my row's pair in each tile, read while the MMAs run
            int pr[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int pair = h < cnt ? p.perm_pad[static_cast<int64_t>(m0 + h) * kBM + row] : -1;
                if (pair >= 0 && !(pair < p.out_rows)) {
                    if (kDebugChecks) debug_index_ok(false, status);
                    pair = -1;
                }
                pr[h] = pair;
            }
            mbar_wait(acc_full, q & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
            tc_fence_after();
            for (int h = 0; h < cnt; ++h) {
                const uint32_t tbase = tmem_base + h * kBN + (static_cast<uint32_t>(quad * 32) << 16);
                uint16_t *dst_row = p.out + static_cast<int64_t>(pr[h] < 0 ? 0 : pr[h]) * p.N;
                for (int cc = 0; cc < kBN / 16; cc += 4) {
                    uint32_t r[4][16];
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) tmem_ld16(tbase + (cc + hh) * 16, r[hh]);
                    tmem_ld_wait16(r[0]);
#pragma unroll
                    for (int hh = 1; hh < 4; ++hh) tmem_regs_after_wait16(r[hh]);
                    if (pr[h] < 0) continue;
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        const int col = n * kBN + (cc + hh) * 16;
                        if (col >= p.N) continue;
                        float v[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[hh][e]);
                        uint4 *o = reinterpret_cast<uint4 *>(dst_row + col);
                        o[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                          pack_bf16x2(v[6], v[7]));
                        if (col + 8 < p.N)
                            o[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                                              pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acc_empty);   // both accumulators read: the next item's MMAs may start
        }
    }

    // ---- teardown ---------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // after a timeout let a wait go early, the loads and MMAs still in flight
    // are waited for (bounded) before the tensor memory is freed
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t it = static_cast<uint32_t>(drain[0]);
            for (uint32_t i = it > kMpStages ? it - kMpStages : 0; i < it; ++i)
                mbar_wait(&full[i % kMpStages], (i / kMpStages) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
        }
        if (warp == 1 && lane == 0 && drain[1] >= 0)
            mbar_wait(acc_full, drain[1] & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

cudaError_t launch_moe_pair(const CUtensorMap &w, const MoePairParams &p, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev >= 64 || !configured[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(moe_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kMpSmem));
        if (e != cudaSuccess) return e;
        if (dev < 64) configured[dev] = 1;
    }
    // persistent, one CTA per SM; a programmatic dependent launch: the CTAs
    // start their prologue as the routing releases SMs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms_current_device()));
    cfg.blockDim = dim3(kMpThreads);
    cfg.dynamicSmemBytes = kMpSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_pair_kernel, w, p);
}

}  // namespace lora
