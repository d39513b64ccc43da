// Mixture of experts (the page "Qwen3-MoE low-latency inference on Atlas
// A3", mokono.cn/news/2297686, its MoE section): route the (token, slot)
// pairs to their experts, run the grouped expert matmul, then put every
// token's rows back and sum them with the routing weights.  The grouped GEMM
// is moe_pair.cu's kernel (the tiled kernel in kModeMoe for routings of more
// token tiles than its item list holds); this file holds the routing and the
// weighted finalize.
//
// Routing, in two launches over chunks of the pairs (one CTA per chunk):
//   count    each CTA's bucket histogram (bucket 0: invalid ids, e + 1:
//            expert e); the padded order is cleared
//   scatter  every CTA sums the histograms (all of them, and those of the
//            chunks before its own), scans the bucket totals, and places its
//            pairs: each warp's pairs in order, ranked among equal buckets
//            with __match_any_sync, so the sort is stable.  The first CTA
//            also writes the bucket offsets, the segment table (one segment
//            per expert with pairs) and each 128-row tile's expert.
//
// Finalize:
//   y[t, n] = bf16( sum_{j < topk, expert[t,j] valid} weight[t,j] * out[t * topk + j, n] )
//
// out holds the experts' bf16 rows in (token, slot) pair order.  Memory-bound:
// one thread per 8 output columns of one token, 16-byte loads and stores,
// coalesced along n; the fp32 sum runs in the slots' order.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"
#include "seg_build_body.cuh"

namespace lora {

constexpr int kRouteWarps = 8;
constexpr int kRouteThreads = kRouteWarps * 32;
constexpr int kRouteBatch = 4;   // ids per lane loaded ahead of a warp's steps
using RouteScan = SegBuild<kRouteWarps>;

__global__ void __launch_bounds__(kRouteThreads) moe_route_count_kernel(RouteParams p)
{
    // the scatter launch may start now; it waits for this grid before
    // reading anything written here
    pdl_launch_dependents();
    extern __shared__ int hist[];   // [nb]
    const int tid = threadIdx.x;
    for (int b = tid; b < p.nb; b += kRouteThreads) hist[b] = 0;
    __syncthreads();
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * p.chunk;
    const int64_t c1 = c0 + p.chunk < p.P ? c0 + p.chunk : p.P;
    int bad = 0;
    for (int64_t t = c0 + tid; t < c1; t += kRouteThreads) {
        const int id = __ldg(p.expert + t);
        const int b = id_bucket(id, p.E);
        bad |= (b == 0 && id != -1);
        atomicAdd(&hist[b], 1);
    }
    if (__syncthreads_or(bad) && tid == 0) atomicOr(p.counters + CNT_STATUS, LORA_DEV_BAD_ID);
    for (int b = tid; b < p.nb; b += kRouteThreads) p.cnt[static_cast<int64_t>(blockIdx.x) * p.nb + b] = hist[b];
    // the padded order starts empty
    const int64_t npad = static_cast<int64_t>(p.max_mtiles) * kBM;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kRouteThreads + tid; i < npad;
         i += static_cast<int64_t>(gridDim.x) * kRouteThreads)
        p.perm_pad[i] = -1;
}

__global__ void __launch_bounds__(kRouteThreads) moe_route_scatter_kernel(RouteParams p)
{
    extern __shared__ int sm[];
    const int nb = p.nb;
    int *whist = sm;                // [warps][nb] per-warp counts, then running positions
    int *bsum = whist + kRouteWarps * nb;   // [nb + 1] first position of each bucket
    int *cbase = bsum + nb + 1;     // [nb] this CTA's first position in each bucket
    int *padt = cbase + nb;         // [nb + 1] first padded tile of each bucket (bucket 0 has none)
    int *wsum = padt + nb + 1;      // [32] scan scratch
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;

    pdl_wait();   // the count grid has finished: its histograms are visible

    for (int i = tid; i < kRouteWarps * nb; i += kRouteThreads) whist[i] = 0;
    // bucket totals over all chunks, and over the chunks before this one
    int carry = 0, carry_t = 0;
    for (int b0 = 0; b0 < nb; b0 += kRouteThreads) {
        const int b = b0 + tid;
        int tot = 0, pre = 0;
        if (b < nb)
            for (int c = 0; c < p.nchunks; ++c) {
                const int v = p.cnt[static_cast<int64_t>(c) * nb + b];
                tot += v;
                if (c < static_cast<int>(blockIdx.x)) pre += v;
            }
        int total, total_t;
        const int ex = RouteScan::block_exclusive_scan(tot, wsum, &total);
        const int tiles = (b >= 1 && b < nb) ? (tot + kBM - 1) / kBM : 0;
        const int ext = RouteScan::block_exclusive_scan(tiles, wsum, &total_t);
        if (b < nb) {
            bsum[b] = carry + ex;
            cbase[b] = carry + ex + pre;
            padt[b] = carry_t + ext;
        }
        carry += total;
        carry_t += total_t;
    }
    if (tid == 0) {
        bsum[nb] = carry;
        padt[nb] = carry_t;
    }
    __syncthreads();

    // each warp's pairs: a contiguous range of the chunk, in steps of 32
    const int64_t per = p.chunk / kRouteWarps;   // a multiple of 32
    const int64_t t_begin = static_cast<int64_t>(blockIdx.x) * p.chunk + w * per;
    const int64_t t_end = t_begin + per < p.P ? t_begin + per : p.P;
    auto for_each_step = [&](auto &&step) {
        for (int64_t base = t_begin; base < t_begin + per; base += 32 * kRouteBatch) {
            int idv[kRouteBatch];
#pragma unroll
            for (int u = 0; u < kRouteBatch; ++u) {
                const int64_t t = base + 32 * u + lane;
                idv[u] = t < t_end ? __ldg(p.expert + t) : 0;
            }
#pragma unroll
            for (int u = 0; u < kRouteBatch; ++u) step(base + 32 * u + lane, idv[u]);
        }
    };
    // per-warp histograms
    for_each_step([&](int64_t t, int id) {
        const bool act = t < t_end;
        const unsigned amask = __ballot_sync(0xffffffffu, act);
        if (act) {
            const int b = id_bucket(id, p.E);
            const unsigned peers = __match_any_sync(amask, b);
            if (lane == __ffs(peers) - 1) whist[w * nb + b] += __popc(peers);
        }
        __syncwarp();
    });
    __syncthreads();
    for (int b = tid; b < nb; b += kRouteThreads) {
        int run = cbase[b];
        for (int ww = 0; ww < kRouteWarps; ++ww) {
            const int c = whist[ww * nb + b];
            whist[ww * nb + b] = run;
            run += c;
        }
    }
    __syncthreads();
    // stable scatter: perm, and each expert's pairs in its padded tiles
    const int64_t npad = static_cast<int64_t>(p.max_mtiles) * kBM;
    for_each_step([&](int64_t t, int id) {
        const bool act = t < t_end;
        const unsigned amask = __ballot_sync(0xffffffffu, act);
        unsigned peers = 0;
        int b = 0;
        if (act) {
            b = id_bucket(id, p.E);
            peers = __match_any_sync(amask, b);
            const int pos = whist[w * nb + b] + __popc(peers & lt_mask);
            p.perm[pos] = static_cast<int32_t>(t);
            if (b > 0) {
                const int64_t pp = static_cast<int64_t>(padt[b]) * kBM + (pos - bsum[b]);
                if (pp < npad) p.perm_pad[pp] = static_cast<int32_t>(t);
            }
        }
        __syncwarp();
        if (act && lane == __ffs(peers) - 1) whist[w * nb + b] += __popc(peers);
        __syncwarp();
    });

    if (blockIdx.x != 0) return;
    // ---- the first CTA: offsets, counters, tile experts, segment table ------
    for (int b = tid; b <= nb; b += kRouteThreads) p.offsets[b] = bsum[b];
    for (int i = tid; i < p.n_counters; i += kRouteThreads)
        if (i != CNT_STATUS) p.counters[i] = 0;
    for (int b = 1 + tid; b < nb; b += kRouteThreads)
        for (int m = padt[b]; m < padt[b + 1] && m < p.max_mtiles; ++m) p.mt_expert[m] = b - 1;
    for (int m = padt[nb] + tid; m < p.max_mtiles; m += kRouteThreads) p.mt_expert[m] = -1;
    if (tid == 0) p.hdr[HDR_MOE_TILES] = padt[nb] < p.max_mtiles ? padt[nb] : p.max_mtiles;
    if (w == 0) {
        int n = 0;
        for (int i0 = 0; i0 < p.E; i0 += 32) {
            const int i = i0 + lane;
            const int cnt = i < p.E ? bsum[i + 2] - bsum[i + 1] : 0;
            const unsigned m = __ballot_sync(0xffffffffu, cnt > 0);
            if (cnt > 0) {
                const int s = n + __popc(m & lt_mask);
                p.seg_id[s] = i;
                p.seg_start[s] = bsum[i + 1];
                p.seg_len[s] = cnt;
                p.seg_rank[s] = 0;
            }
            n += __popc(m);
        }
        if (lane == 0) {
            *p.num_segments = n;
            p.hdr[HDR_NSEG] = n;
        }
    }
}

static size_t route_scatter_smem(int nb) { return static_cast<size_t>(kRouteWarps * nb + 3 * nb + 2 + 32) * 4; }

cudaError_t launch_moe_route(const RouteParams &p, cudaStream_t stream)
{
    moe_route_count_kernel<<<p.nchunks, kRouteThreads, static_cast<size_t>(p.nb) * 4, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nchunks);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = route_scatter_smem(p.nb);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_route_scatter_kernel, p);
}

__global__ void __launch_bounds__(256) moe_finalize_kernel(const uint16_t *out, const int32_t *expert,
                                                          const float *weight, int64_t M, int topk, int E, int N,
                                                          uint16_t *y)
{
    const int groups = N / 8;
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t t = gid / groups;
    const int g = static_cast<int>(gid - t * groups);
    if (t >= M) return;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < topk; ++j) {
        const int64_t pair = t * topk + j;
        const int e = expert[pair];
        if (e < 0 || e >= E) continue;
        const float w = weight[pair];
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(out + pair * N) + g);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc[2 * k] += w * bf16_lo(u[k]);
            acc[2 * k + 1] += w * bf16_hi(u[k]);
        }
    }
    reinterpret_cast<uint4 *>(y + t * N)[g] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                         pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

cudaError_t launch_moe_finalize(const uint16_t *out, const int32_t *expert, const float *weight, int64_t M, int topk,
                                int E, int N, uint16_t *y, cudaStream_t stream)
{
    const int64_t threads = M * (N / 8);
    if (threads == 0) return cudaSuccess;
    const int64_t blocks = (threads + 255) / 256;
    moe_finalize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, expert, weight, M, topk, E, N, y);
    return cudaGetLastError();
}

}  // namespace lora
