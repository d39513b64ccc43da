// Segment builder ("vLLM-Ascend dynamic LoRA", §2.3): bucket the tokens by
// lora_id so that tokens of one adapter become contiguous, and derive the
// work lists the fused kernels consume (§2.4: which token block a core
// handles, which segment it belongs to and its rank are decided before the
// GEMM launches, not by branching inside it).
//
// One CTA of 1024 threads.  Each warp owns a contiguous range of tokens:
//   pass 1  warp-aggregated histogram (__match_any_sync peers, leader adds
//           popc) into a per-warp row of a [32][A+1] shared table
//   scan    bucket totals -> exclusive scan -> per-warp running bases
//   pass 2  stable scatter: rank inside a 32-token step = popc of the peers
//           below the lane, plus the warp's running base for the bucket
// Bucket 0 holds id -1, bucket i+1 adapter i; ids outside [-1, A) are
// counted as -1 and flagged in the status word.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {


constexpr int kSegThreads = 1024;

// Exclusive scan of one int per thread over the 1024-thread block.
__device__ int block_exclusive_scan(int v, int *wsum, int *total)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        wsum[lane] = s;
    }
    __syncthreads();
    const int excl = x - v + (w > 0 ? wsum[w - 1] : 0);
    *total = wsum[31];
    __syncthreads();
    return excl;
}

__global__ void __launch_bounds__(kSegThreads, 1) seg_build_kernel(SegParams p)
{
    extern __shared__ int sm[];
    const int nb = p.A + 1;
    int *whist = sm;                 // [32][nb]
    int *bsum = whist + 32 * nb;     // [nb + 1]
    int *wsum = bsum + nb + 1;       // [32]
    // the segment table and per-adapter pool rows, kept on chip for the
    // per-tile loops below (A entries each)
    int *s_id = wsum + 32, *s_start = s_id + p.A, *s_len = s_start + p.A, *s_rank = s_len + p.A;
    int *s_arow = s_rank + p.A;      // a_offset / K
    int *s_brow = s_arow + p.A;      // b_offset / 16
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int32_t *status = p.counters + CNT_STATUS;

    for (int i = tid; i < p.n_counters; i += kSegThreads)
        if (i != CNT_STATUS && i != CNT_EPOCH) p.counters[i] = 0;
    for (int i = tid; i < 32 * nb; i += kSegThreads) whist[i] = 0;
    for (int i = tid; i < p.A; i += kSegThreads) {
        s_arow[i] = static_cast<int>(p.a_offset[i] / p.K);
        s_brow[i] = static_cast<int>(p.b_offset[i] / kChunk);
    }
    __syncthreads();

    const int64_t per = (p.M + 31) / 32;
    const int64_t t_begin = w * per;
    const int64_t t_end = t_begin + per < p.M ? t_begin + per : p.M;

    // ---- pass 1: per-warp histograms --------------------------------------
    int bad = 0;
    for (int64_t base = t_begin; base < t_end; base += 32) {
        const int64_t t = base + lane;
        const bool act = t < t_end;
        const unsigned amask = __ballot_sync(0xffffffffu, act);
        if (act) {
            const int id = p.ids[t];
            const int e = (id >= 0 && id < p.A) ? id : -1;
            bad |= (e != id);
            const int b = e + 1;
            const unsigned peers = __match_any_sync(amask, b);
            if (lane == __ffs(peers) - 1) whist[w * nb + b] += __popc(peers);
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, LORA_DEV_BAD_ID);
    __syncthreads();

    // ---- bucket totals, exclusive scan, per-warp running bases ------------
    int carry = 0;
    for (int b0 = 0; b0 < nb; b0 += kSegThreads) {
        const int b = b0 + tid;
        int tot = 0;
        if (b < nb)
            for (int ww = 0; ww < 32; ++ww) tot += whist[ww * nb + b];
        int total;
        const int ex = block_exclusive_scan(tot, wsum, &total);
        if (b < nb) {
            int run = carry + ex;
            bsum[b] = run;
            for (int ww = 0; ww < 32; ++ww) {
                const int c = whist[ww * nb + b];
                whist[ww * nb + b] = run;
                run += c;
            }
        }
        carry += total;
    }
    if (tid == 0) bsum[nb] = carry;
    __syncthreads();
    for (int b = tid; b <= nb; b += kSegThreads) p.offsets[b] = bsum[b];

    // ---- pass 2: stable scatter -------------------------------------------
    for (int64_t base = t_begin; base < t_end; base += 32) {
        const int64_t t = base + lane;
        const bool act = t < t_end;
        const unsigned amask = __ballot_sync(0xffffffffu, act);
        unsigned peers = 0;
        int b = 0;
        if (act) {
            const int id = p.ids[t];
            b = ((id >= 0 && id < p.A) ? id : -1) + 1;
            peers = __match_any_sync(amask, b);
            const int below = __popc(peers & ((1u << lane) - 1u));
            p.perm[whist[w * nb + b] + below] = static_cast<int32_t>(t);
        }
        __syncwarp();
        if (act && lane == __ffs(peers) - 1) whist[w * nb + b] += __popc(peers);
        __syncwarp();
    }

    // ---- segments: one per non-empty adapter bucket, ascending id ---------
    carry = 0;
    for (int i0 = 0; i0 < p.A; i0 += kSegThreads) {
        const int i = i0 + tid;
        const int cnt = i < p.A ? bsum[i + 2] - bsum[i + 1] : 0;
        const int flag = cnt > 0;
        int total;
        const int ex = block_exclusive_scan(flag, wsum, &total);
        if (flag) {
            const int s = carry + ex;
            const int rk = p.rank[i];
            p.seg_id[s] = i;
            p.seg_start[s] = bsum[i + 1];
            p.seg_len[s] = cnt;
            p.seg_rank[s] = rk;
            s_id[s] = i;
            s_start[s] = bsum[i + 1];
            s_len[s] = cnt;
            s_rank[s] = rk;
        }
        carry += total;
    }
    const int nseg = carry;
    if (tid == 0) {
        *p.num_segments = nseg;
        p.hdr[HDR_NSEG] = nseg;
    }
    __syncthreads();

    // ---- split-K chunk list: every rank panel of every adapter present ----
    carry = 0;
    for (int s0 = 0; s0 < nseg; s0 += kSegThreads) {
        const int s = s0 + tid;
        const int nc = s < nseg ? s_rank[s] / kChunk : 0;
        int total;
        const int ex = block_exclusive_scan(nc, wsum, &total);
        if (s < nseg) {
            const int i = s_id[s];
            const int c = carry + ex;
            for (int q = 0; q < nc; ++q) {
                p.dchunk_arow[c + q] = s_arow[i] + kChunk * q;
                p.dchunk_brow[c + q] = s_brow[i] + q * p.N;
                p.dchunk_adapter[c + q] = i;
            }
        }
        carry += total;
    }
    if (tid == 0) p.hdr[HDR_DCHUNKS] = carry;

    // ---- cluster schedule: each adapter's panels in groups of <= 2, and
    //      the first panel of every segment -----------------------------------
    carry = 0;
    int carry_c2 = 0;
    for (int s0 = 0; s0 < nseg; s0 += kSegThreads) {
        const int s = s0 + tid;
        const int nc = s < nseg ? s_rank[s] / kChunk : 0;
        const int ng = (nc + 1) / 2;
        int total, total_c;
        const int exg = block_exclusive_scan(ng, wsum, &total);
        const int exc = block_exclusive_scan(nc, wsum, &total_c);
        if (s < nseg) {
            const int c = carry_c2 + exc;
            const int i = s_id[s];
            p.dseg_first[s] = c;
            p.dseg_group[s] = carry + exg;
            for (int q = 0; q < ng; ++q) {
                p.dgrp_first[carry + exg + q] = c + 2 * q;
                p.dgrp_len[carry + exg + q] = min(2, nc - 2 * q);
                p.dgrp_arow[carry + exg + q] = s_arow[i] + 2 * q * kChunk;
                p.dgrp_adapter[carry + exg + q] = i;
            }
        }
        carry += total;
        carry_c2 += total_c;
    }
    if (tid == 0) p.hdr[HDR_DGROUPS] = carry;
    __syncthreads();

    // ---- stream schedule: which panels of the B pool belong to adapters
    //      present, in 8-panel windows (pool order).  ppinfo[p] = 2 * group +
    //      half for a present panel p, -1 otherwise ----------------------------
    int *ppinfo = whist;   // the histogram space is free again
    for (int pp = tid; pp < p.P; pp += kSegThreads) ppinfo[pp] = -1;
    __syncthreads();
    for (int s = tid; s < nseg; s += kSegThreads) {
        const int i = s_id[s];
        const int pp0 = s_brow[i] / p.N;        // first pool panel of adapter i
        const int np = s_rank[s] / kChunk;
        const int g0 = p.dseg_group[s];
        for (int j = 0; j < np; ++j) ppinfo[pp0 + j] = 2 * (g0 + j / 2) + (j & 1);
    }
    __syncthreads();
    carry = 0;
    const int nwin_all = (p.P + 7) / 8;
    for (int w0 = 0; w0 < nwin_all; w0 += kSegThreads) {
        const int w = w0 + tid;
        int any = 0;
        if (w < nwin_all)
            for (int j = 0; j < 8 && 8 * w + j < p.P; ++j) any |= ppinfo[8 * w + j] >= 0;
        int total;
        const int ex = block_exclusive_scan(any, wsum, &total);
        if (any) {
            const int k = carry + ex;
            p.ewin_first[k] = 8 * w;
            for (int j = 0; j < 8; ++j) p.pinfo[8 * k + j] = 8 * w + j < p.P ? ppinfo[8 * w + j] : -1;
        }
        carry += total;
    }
    if (tid == 0) p.hdr[HDR_NWIN] = carry;

    // ---- tiled schedule: per 128-token tile of the permuted order, the
    //      rank panels of the segments it intersects, and its shrink jobs ---
    int carry_c = 0, carry_j = 0;
    for (int m0 = 0; m0 < p.num_mtiles; m0 += kSegThreads) {
        const int m = m0 + tid;
        int nch = 0, sfirst = 0;
        int64_t lo = 0, hi = 0;
        if (m < p.num_mtiles) {
            lo = static_cast<int64_t>(m) * kBM;
            hi = lo + kBM < p.M ? lo + kBM : p.M;
            int L = 0, R = nseg;   // first segment whose end is past lo
            while (L < R) {
                const int mid = (L + R) >> 1;
                if (s_start[mid] + s_len[mid] > lo) R = mid; else L = mid + 1;
            }
            sfirst = L;
            for (int s = sfirst; s < nseg && s_start[s] < hi; ++s) nch += s_rank[s] / kChunk;
        }
        int totc, totj;
        const int exc = block_exclusive_scan(nch, wsum, &totc);
        const int nj = (nch + kMaxShrinkChunks - 1) / kMaxShrinkChunks;
        const int exj = block_exclusive_scan(nj, wsum, &totj);
        if (m < p.num_mtiles) {
            int c = carry_c + exc;
            const int cfirst = c;
            p.tile_chunk_off[m] = c;
            p.tile_njobs[m] = nj;
            for (int s = sfirst; s < nseg && s_start[s] < hi; ++s) {
                const int64_t s0 = s_start[s], s1 = s0 + s_len[s];
                const int rlo = static_cast<int>((s0 > lo ? s0 : lo) - lo);
                const int rhi = static_cast<int>((s1 < hi ? s1 : hi) - lo);
                const int i = s_id[s];
                for (int q = 0; q < s_rank[s] / kChunk; ++q, ++c) {
                    p.chunk_arow[c] = s_arow[i] + kChunk * q;
                    p.chunk_brow[c] = s_brow[i] + q * p.N;
                    p.chunk_rng[c] = pack_rng(rlo, rhi, q);
                }
            }
            const int j = carry_j + exj;
            for (int q = 0; q < nj; ++q) {
                p.sjob_tile[j + q] = m;
                p.sjob_c0[j + q] = cfirst + kMaxShrinkChunks * q;
                const int c1 = cfirst + kMaxShrinkChunks * (q + 1);
                p.sjob_c1[j + q] = c1 < cfirst + nch ? c1 : cfirst + nch;
            }
        }
        carry_c += totc;
        carry_j += totj;
    }
    if (tid == 0) {
        p.tile_chunk_off[p.num_mtiles] = carry_c;
        p.hdr[HDR_NCHUNKS] = carry_c;
        p.hdr[HDR_NSJOBS] = carry_j;
    }
}

size_t seg_build_smem_bytes(int32_t A)
{
    // the [32][A+1] histogram space is reused for the pool panel table (<= 4 A entries)
    return static_cast<size_t>(32 * (A + 1) + (A + 2) + 32 + 6 * A) * 4;
}

cudaError_t launch_seg_build(const SegParams &p, cudaStream_t stream)
{
    const size_t smem = seg_build_smem_bytes(p.A);
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem > 48 * 1024 && (dev >= 64 || !configured[dev])) {
        cudaError_t e = cudaFuncSetAttribute(seg_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(seg_build_smem_bytes(LORA_MAX_ADAPTERS)));
        if (e != cudaSuccess) return e;
        if (dev < 64) configured[dev] = 1;
    }
    seg_build_kernel<<<1, kSegThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace lora
