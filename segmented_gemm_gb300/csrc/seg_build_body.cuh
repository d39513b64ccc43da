// Segment builder body, shared by the stand-alone builder kernel (one CTA of
// 16 warps) and the decode-sized fused kernel, one of whose CTAs (10 warps)
// runs it beside the weight stream.
//
// Segment builder ("vLLM-Ascend dynamic LoRA", §2.3): bucket the tokens by
// lora_id so that tokens of one adapter become contiguous, and derive the
// work lists the fused kernels consume (§2.4: which token block a core
// handles, which segment it belongs to and its rank are decided before the
// GEMM launches, not by branching inside it).
//
// One CTA of W warps (16 or 10), three block-wide barriers:
//   phase 0  zero the counter block, stage ranks and pool offsets on chip
//   phase 1  each warp owns a contiguous range of tokens and builds its own
//            histogram row (__match_any_sync peers, the leader adds popc)
//   phase 2  bucket totals -> exclusive scan -> per-warp running bases
//   phase 3  every warp scatters its own tokens (stable: the rank inside a
//            32-token step is the popc of the peers below the lane plus the
//            warp's running base), then the warps build one list each, in
//            parallel and without further block barriers:
//              warp 0       the segment table (one segment per non-empty
//                           adapter bucket, ascending id)
//              warp 1       split-K chunk list (rank panels of adapters present)
//              warps 2..W-1 tiled-schedule chunk lists and shrink jobs: one
//                           warp per 128-token tile (a lane per adapter
//                           bucket) when there are at most W-2 tiles, else
//                           one thread per tile
// Bucket 0 holds id -1, bucket i+1 adapter i; ids outside [-1, A) are
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

// Bucket of a token id: 0 for -1 and for ids outside [-1, A), else id + 1.
__device__ __forceinline__ int id_bucket(int id, int A) { return (id >= 0 && id < A) ? id + 1 : 0; }

__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// Everything sized by the warp count of the CTA that runs the build.
template <int kSegWarpsT>
struct SegBuild {
    static constexpr int kSegWarps = kSegWarpsT;
    static constexpr int kSegThreads = kSegWarps * 32;
    static constexpr int kTileWarp0 = 2;                 // first warp of the tile-list group
    static constexpr int kTileWarps = kSegWarps - kTileWarp0;
    static constexpr int kTileBar = 1;                   // named barrier of the tile-list group
    static constexpr int kIdBatch = 8;                   // ids per lane loaded ahead of the histogram / scatter steps
    static_assert(kTileWarps >= 1 && 2 * kTileWarps <= 32 && kTileWarps <= 16,
                  "tile-list scan scratch lives in the 32-int wsum");

    // histograms, bucket offsets, scan scratch and three per-adapter tables
    static __host__ __device__ size_t smem_bytes(int32_t A)
    {
        return static_cast<size_t>(kSegWarps * (A + 1) + (A + 2) + 32 + 3 * A) * 4;
    }

    // Exclusive scan of one int per thread over the whole block.
    static __device__ int block_exclusive_scan(int v, int *wsum, int *total)
    {
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        const int x = warp_incl_scan(v, lane);
        if (lane == 31) wsum[w] = x;
        __syncthreads();
        if (w == 0) {
            int s = lane < kSegWarps ? wsum[lane] : 0;
            s = warp_incl_scan(s, lane);
            if (lane < kSegWarps) wsum[lane] = s;
        }
        __syncthreads();
        const int excl = x - v + (w > 0 ? wsum[w - 1] : 0);
        *total = wsum[kSegWarps - 1];
        __syncthreads();
        return excl;
    }

    // Exclusive scan of two ints per thread over the tile-list warps only.
    static __device__ void tile_group_scan(int a, int b, int *ws2, int *ea, int *eb, int *ta, int *tb)
    {
        const int lane = threadIdx.x & 31, gw = (threadIdx.x >> 5) - kTileWarp0;
        const int xa = warp_incl_scan(a, lane), xb = warp_incl_scan(b, lane);
        if (lane == 31) {
            ws2[2 * gw] = xa;
            ws2[2 * gw + 1] = xb;
        }
        named_bar_sync(kTileBar, kTileWarps * 32);
        if (gw == 0) {
            int sa = lane < kTileWarps ? ws2[2 * lane] : 0, sb = lane < kTileWarps ? ws2[2 * lane + 1] : 0;
            sa = warp_incl_scan(sa, lane);
            sb = warp_incl_scan(sb, lane);
            if (lane < kTileWarps) {
                ws2[2 * lane] = sa;
                ws2[2 * lane + 1] = sb;
            }
        }
        named_bar_sync(kTileBar, kTileWarps * 32);
        *ea = xa - a + (gw > 0 ? ws2[2 * (gw - 1)] : 0);
        *eb = xb - b + (gw > 0 ? ws2[2 * (gw - 1) + 1] : 0);
        *ta = ws2[2 * (kTileWarps - 1)];
        *tb = ws2[2 * (kTileWarps - 1) + 1];
        named_bar_sync(kTileBar, kTileWarps * 32);
    }

    // The whole build, by every thread of the calling CTA (kSegThreads of
    // them), with `sm` holding smem_bytes(p.A) bytes of shared memory.
    static __device__ void run(const SegParams &p, int *sm)
    {
        const int A = p.A, nb = A + 1;
        const int nsl = p.num_slices > 1 ? p.num_slices : 1;   // output slices (merged projection)
        int *whist = sm;                          // [kSegWarps][nb]
        int *bsum = whist + kSegWarps * nb;       // [nb + 1] bucket offsets
        int *wsum = bsum + nb + 1;                // [32] scan scratch
        int *s_rank = wsum + 32;                  // [A] padded ranks
        int *s_arow = s_rank + A;                 // [A] first A pool row (a_offset / K)
        int *s_bpan = s_arow + A;                 // [A] b_offset / (16 N): first [N, 16] B panel
        const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
        int32_t *status = p.counters + CNT_STATUS;

        const int64_t per = (p.M + kSegWarps - 1) / kSegWarps;
        const int64_t t_begin = w * per;
        const int64_t t_end = t_begin + per < p.M ? t_begin + per : p.M;

        // ---- phase 0 -------------------------------------------------------------
        for (int i = tid; i < p.n_counters; i += kSegThreads)
            if (i != CNT_STATUS) p.counters[i] = 0;
        for (int i = tid; i < kSegWarps * nb; i += kSegThreads) whist[i] = 0;
        for (int i = tid; i < A; i += kSegThreads) {
            s_rank[i] = p.rank[i];
            s_arow[i] = static_cast<int>(p.a_offset[i] / p.K);
            // B panels are counted in whole [N, 16] panels, so that the
            // table does not depend on N (nor on K: A rows are rank rows)
            s_bpan[i] = static_cast<int>(p.b_offset[i] / (static_cast<int64_t>(kChunk) * p.N));
            if (p.b_offset[i] % (static_cast<int64_t>(kChunk) * p.N) != 0) atomicOr(p.counters + CNT_STATUS, LORA_DEV_BAD_POOL);
            // a merged output needs every adapter's rank in whole 16-wide
            // panels per slice
            if (s_rank[i] % (kChunk * nsl) != 0) atomicOr(p.counters + CNT_STATUS, LORA_DEV_BAD_POOL);
        }
        __syncthreads();

        // ---- phase 1: per-warp histograms ----------------------------------------
        int bad = 0;
        auto hist_step = [&](int64_t t, int id) {
            const bool act = t < t_end;
            const unsigned amask = __ballot_sync(0xffffffffu, act);
            if (act) {
                const int b = id_bucket(id, A);
                bad |= (b == 0 && id != -1);
                const unsigned peers = __match_any_sync(amask, b);
                if (lane == __ffs(peers) - 1) whist[w * nb + b] += __popc(peers);
            }
        };
        // eight ids per lane in flight, then the steps in token order
        for (int64_t base = t_begin; base < t_end; base += 32 * kIdBatch) {
            int idv[kIdBatch];
#pragma unroll
            for (int u = 0; u < kIdBatch; ++u) {
                const int64_t t = base + 32 * u + lane;
                idv[u] = t < t_end ? __ldg(p.ids + t) : 0;
            }
#pragma unroll
            for (int u = 0; u < kIdBatch; ++u) hist_step(base + 32 * u + lane, idv[u]);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, LORA_DEV_BAD_ID);
        __syncthreads();

        // ---- phase 2: bucket totals, exclusive scan, per-warp running bases ------
        int carry = 0;
        for (int b0 = 0; b0 < nb; b0 += kSegThreads) {
            const int b = b0 + tid;
            int tot = 0;
            if (b < nb)
                for (int ww = 0; ww < kSegWarps; ++ww) tot += whist[ww * nb + b];
            int total;
            const int ex = block_exclusive_scan(tot, wsum, &total);
            if (b < nb) {
                int run = carry + ex;
                bsum[b] = run;
                for (int ww = 0; ww < kSegWarps; ++ww) {
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
        // ---- phase 3a: stable scatter (every warp, its own tokens in order) ------
        auto scatter_step = [&](int64_t t, int id) {
            const bool act = t < t_end;
            const unsigned amask = __ballot_sync(0xffffffffu, act);
            unsigned peers = 0;
            int b = 0;
            if (act) {
                b = id_bucket(id, A);
                peers = __match_any_sync(amask, b);
                const int below = __popc(peers & ((1u << lane) - 1u));
                const int pos = whist[w * nb + b] + below;
                p.perm[pos] = static_cast<int32_t>(t);
            }
            __syncwarp();
            if (act && lane == __ffs(peers) - 1) whist[w * nb + b] += __popc(peers);
            __syncwarp();
        };
        // eight ids per lane in flight, then the steps in token order
        for (int64_t base = t_begin; base < t_end; base += 32 * kIdBatch) {
            int idv[kIdBatch];
#pragma unroll
            for (int u = 0; u < kIdBatch; ++u) {
                const int64_t t = base + 32 * u + lane;
                idv[u] = t < t_end ? __ldg(p.ids + t) : 0;
            }
#pragma unroll
            for (int u = 0; u < kIdBatch; ++u) scatter_step(base + 32 * u + lane, idv[u]);
        }

        // ---- phase 3b: one list per warp (group) ---------------------------------
        const unsigned lt_mask = (1u << lane) - 1u;
        if (w == 0) {
            // the segment table
            int n = 0;
            for (int i0 = 0; i0 < A; i0 += 32) {
                const int i = i0 + lane;
                const int cnt = i < A ? bsum[i + 2] - bsum[i + 1] : 0;
                const unsigned m = __ballot_sync(0xffffffffu, cnt > 0);
                if (cnt > 0) {
                    const int s = n + __popc(m & lt_mask);
                    p.seg_id[s] = i;
                    p.seg_start[s] = bsum[i + 1];
                    p.seg_len[s] = cnt;
                    p.seg_rank[s] = s_rank[i];
                }
                n += __popc(m);
            }
            if (lane == 0) {
                *p.num_segments = n;
                p.hdr[HDR_NSEG] = n;
            }
        } else if (w == 1) {
            // split-K chunk list: every rank panel of every adapter present
            int n = 0;
            for (int i0 = 0; i0 < A; i0 += 32) {
                const int i = i0 + lane;
                const int nc = (i < A && bsum[i + 2] > bsum[i + 1]) ? s_rank[i] / kChunk : 0;
                const int incl = warp_incl_scan(nc, lane);
                const int c = n + incl - nc;
                for (int q = 0; q < nc; ++q) {
                    p.dchunk_arow[c + q] = s_arow[i] + kChunk * q;
                    p.dchunk_bpanel[c + q] = s_bpan[i] + q;
                    p.dchunk_adapter[c + q] = i;
                }
                n += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) p.hdr[HDR_DCHUNKS] = n;
        } else if (p.num_mtiles <= kTileWarps) {
            // tiled schedule, few tiles: warp (w - 2) builds tile m's chunk list,
            // one lane per adapter bucket
            const int m = w - kTileWarp0;
            int *t_nch = wsum, *t_nj = wsum + 16;     // per-tile counts (<= kTileWarps <= 16 tiles)
            int64_t lo = 0, hi = 0;
            int bfirst = A + 1, nch = 0;
            if (m < p.num_mtiles) {
                lo = static_cast<int64_t>(m) * kBM;
                hi = lo + kBM < p.M ? lo + kBM : p.M;
                int L = 1, R = A + 1;   // first adapter bucket that ends past lo
                while (L < R) {
                    const int mid = (L + R) >> 1;
                    if (bsum[mid + 1] > lo) R = mid; else L = mid + 1;
                }
                bfirst = L;
                for (int b0 = bfirst; b0 <= A; b0 += 32) {
                    const int b = b0 + lane;
                    const bool in = b <= A && bsum[b] < hi;
                    int nc = (in && bsum[b + 1] > bsum[b]) ? s_rank[b - 1] / kChunk / nsl * nsl : 0;
    #pragma unroll
                    for (int o = 16; o > 0; o >>= 1) nc += __shfl_xor_sync(0xffffffffu, nc, o);
                    nch += nc;
                    if (__ballot_sync(0xffffffffu, in) != 0xffffffffu) break;
                }
                if (lane == 0) {
                    t_nch[m] = nch;
                    t_nj[m] = (nch + kMaxShrinkChunks - 1) / kMaxShrinkChunks;
                }
            }
            named_bar_sync(kTileBar, kTileWarps * 32);
            if (m < p.num_mtiles) {
                int cbase = 0, jbase = 0;
                for (int k = 0; k < m; ++k) {
                    cbase += t_nch[k];
                    jbase += t_nj[k];
                }
                // slice-major: the panels of output slice 0 of every segment,
                // then slice 1's, ... (one slice unless the output is merged)
                int c = cbase;
                for (int sl = 0; sl < nsl; ++sl) {
                    if (lane == 0) p.tile_chunk_off[m * nsl + sl] = c;
                    for (int b0 = bfirst; b0 <= A; b0 += 32) {
                        const int b = b0 + lane;
                        const bool in = b <= A && bsum[b] < hi;
                        const bool live = in && bsum[b + 1] > bsum[b];
                        const int nc = live ? s_rank[b - 1] / kChunk / nsl : 0;   // panels per slice
                        const int incl = warp_incl_scan(nc, lane);
                        if (live) {
                            const int64_t s0 = bsum[b], s1 = bsum[b + 1];
                            const int rlo = static_cast<int>((s0 > lo ? s0 : lo) - lo);
                            const int rhi = static_cast<int>((s1 < hi ? s1 : hi) - lo);
                            const int i = b - 1;
                            for (int qq = 0; qq < nc; ++qq) {
                                const int cc = c + incl - nc + qq, q = sl * nc + qq;
                                p.chunk_arow[cc] = s_arow[i] + kChunk * q;
                                p.chunk_bpanel[cc] = s_bpan[i] + q;
                                p.chunk_rng[cc] = pack_rng(rlo, rhi, q);
                            }
                        }
                        c += __shfl_sync(0xffffffffu, incl, 31);
                        if (__ballot_sync(0xffffffffu, in) != 0xffffffffu) break;
                    }
                }
                const int nj = t_nj[m];
                if (lane == 0) p.tile_njobs[m] = nj;
                for (int q = lane; q < nj; q += 32) {
                    p.sjob_tile[jbase + q] = m;
                    p.sjob_c0[jbase + q] = cbase + kMaxShrinkChunks * q;
                    const int c1 = cbase + kMaxShrinkChunks * (q + 1);
                    p.sjob_c1[jbase + q] = c1 < cbase + nch ? c1 : cbase + nch;
                }
                if (m == p.num_mtiles - 1 && lane == 0) {
                    p.tile_chunk_off[p.num_mtiles * nsl] = cbase + nch;
                    p.hdr[HDR_NCHUNKS] = cbase + nch;
                    p.hdr[HDR_NSJOBS] = jbase + nj;
                }
            }
        } else {
            // tiled schedule, many tiles: per 128-token tile of the permuted
            // order (one thread each), the rank panels of the segments it
            // intersects (ascending adapter), and its shrink jobs of
            // <= kMaxShrinkChunks panels
            const int gt = tid - kTileWarp0 * 32;
            int carry_c = 0, carry_j = 0;
            for (int m0 = 0; m0 < p.num_mtiles; m0 += kTileWarps * 32) {
                const int m = m0 + gt;
                int nch = 0, bfirst = 1;
                int64_t lo = 0, hi = 0;
                if (m < p.num_mtiles) {
                    lo = static_cast<int64_t>(m) * kBM;
                    hi = lo + kBM < p.M ? lo + kBM : p.M;
                    int L = 1, R = A + 1;   // first adapter bucket that ends past lo
                    while (L < R) {
                        const int mid = (L + R) >> 1;
                        if (bsum[mid + 1] > lo) R = mid; else L = mid + 1;
                    }
                    bfirst = L;
                    for (int b = bfirst; b <= A && bsum[b] < hi; ++b)
                        if (bsum[b + 1] > bsum[b]) nch += s_rank[b - 1] / kChunk / nsl * nsl;
                }
                const int nj = (nch + kMaxShrinkChunks - 1) / kMaxShrinkChunks;
                int exc, exj, totc, totj;
                tile_group_scan(nch, nj, wsum, &exc, &exj, &totc, &totj);
                if (m < p.num_mtiles) {
                    int c = carry_c + exc;
                    const int cfirst = c;
                    p.tile_njobs[m] = nj;
                    for (int sl = 0; sl < nsl; ++sl) {   // slice-major, as above
                        p.tile_chunk_off[m * nsl + sl] = c;
                        for (int b = bfirst; b <= A && bsum[b] < hi; ++b) {
                            const int64_t s0 = bsum[b], s1 = bsum[b + 1];
                            if (s1 == s0) continue;
                            const int rlo = static_cast<int>((s0 > lo ? s0 : lo) - lo);
                            const int rhi = static_cast<int>((s1 < hi ? s1 : hi) - lo);
                            const int i = b - 1;
                            const int np = s_rank[i] / kChunk / nsl;
                            for (int q = sl * np; q < (sl + 1) * np; ++q, ++c) {
                                p.chunk_arow[c] = s_arow[i] + kChunk * q;
                                p.chunk_bpanel[c] = s_bpan[i] + q;
                                p.chunk_rng[c] = pack_rng(rlo, rhi, q);
                            }
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
            if (gt == 0) {
                p.tile_chunk_off[p.num_mtiles * nsl] = carry_c;
                p.hdr[HDR_NCHUNKS] = carry_c;
                p.hdr[HDR_NSJOBS] = carry_j;
            }
        }
    }
};

}  // namespace lora
