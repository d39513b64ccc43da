// Consistency check of a segment table in the workspace against the ids it
// was built from ("vLLM-Ascend dynamic LoRA", §2.3: tokens bucketed by
// lora_id, a stable order, one segment per adapter present, and §2.4: the
// tile and chunk work lists derived from it before the GEMM runs).
//
// One CTA.  It reads every word of the table once and writes only its
// verdict (below) and the status bit LORA_DEV_CHECK, set when
//   - a bucket's width in bucket_offsets differs from the number of ids in
//     that bucket (the segment sums), or bucket_offsets[0] != 0;
//   - a perm entry is outside [0, M), names a token of another bucket than
//     its position's, or is not above the entry before it in the same bucket
//     (with the widths right, this makes perm a permutation and stable);
//   - the segment list is not the non-empty adapter buckets in ascending id
//     with their start, length and padded rank;
//   - a work list of the tiled or split-K schedule is out of range: chunk
//     offsets not ascending from 0 to the chunk count, a row range or rank
//     panel outside a 128-row tile and LORA_MAX_RANK, a pool row or panel
//     past the pool, a shrink job outside its tile's chunks, counts past
//     the workspace's capacity.
// Every index it follows is range-checked before it is used.  The verdict
// also goes into the table's header (HDR_CHECK), where the fused kernels of
// the library built with LORA_DEBUG read it: that build runs this check on
// every table before a fused kernel consumes it, and a table that failed
// leaves the kernel's work list empty.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

constexpr int kCheckThreads = 512;

__device__ __forceinline__ int check_bucket(int id, int A) { return (id >= 0 && id < A) ? id + 1 : 0; }

__global__ void __launch_bounds__(kCheckThreads) seg_check_kernel(const SegCheckParams q)
{
    const SegParams &p = q.s;
    __shared__ int s_off[LORA_MAX_ADAPTERS + 2];
    __shared__ int s_cnt[LORA_MAX_ADAPTERS + 1];
    __shared__ int s_present, s_njobs;
    const int A = p.A, nb = A + 1, tid = threadIdx.x;
    const int64_t M = p.M;
    bool bad = false;

    for (int b = tid; b < nb; b += kCheckThreads) s_cnt[b] = 0;
    for (int b = tid; b <= nb; b += kCheckThreads) s_off[b] = p.offsets[b];
    if (tid == 0) {
        s_present = 0;
        s_njobs = 0;
    }
    __syncthreads();
    for (int64_t t = tid; t < M; t += kCheckThreads) atomicAdd(&s_cnt[check_bucket(p.ids[t], A)], 1);
    __syncthreads();

    // ---- the segment sums: each bucket's width is its count of ids ---------
    if (tid == 0 && s_off[0] != 0) bad = true;
    for (int b = tid; b < nb; b += kCheckThreads) {
        if (s_off[b + 1] - s_off[b] != s_cnt[b]) bad = true;
        if (b >= 1 && s_cnt[b] > 0) atomicAdd(&s_present, 1);
    }
    // with the widths right, the offsets ascend from 0 to M
    const bool offs_bad = __syncthreads_or(bad) != 0;

    // ---- perm: a stable permutation that lists each bucket's tokens --------
    for (int64_t j = tid; j < M; j += kCheckThreads) {
        const int t = p.perm[j];
        if (t < 0 || t >= M) {
            bad = true;
            continue;
        }
        if (offs_bad) continue;
        int lo = 0, hi = nb - 1;   // the bucket of position j: the last b with s_off[b] <= j
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= j) lo = mid;
            else hi = mid - 1;
        }
        if (check_bucket(p.ids[t], A) != lo) bad = true;
        if (j + 1 < s_off[lo + 1] && p.perm[j + 1] <= t) bad = true;
    }

    // ---- the segment list ------------------------------------------------------
    const int n = *p.num_segments;
    if (tid == 0 && (n < 0 || n > A || n != s_present || p.hdr[HDR_NSEG] != n)) bad = true;
    const int nn = (n >= 0 && n <= A) ? n : 0;
    for (int s = tid; s < nn; s += kCheckThreads) {
        const int id = p.seg_id[s];
        if (id < 0 || id >= A) {
            bad = true;
            continue;
        }
        if (s > 0 && p.seg_id[s - 1] >= id) bad = true;
        if (p.seg_len[s] <= 0 || p.seg_rank[s] != p.rank[id]) bad = true;
        if (!offs_bad && (p.seg_start[s] != s_off[id + 1] || p.seg_len[s] != s_off[id + 2] - s_off[id + 1])) bad = true;
    }

    // ---- the tiled schedule's chunk lists and shrink jobs -----------------------
    const int nsl = p.num_slices > 1 ? p.num_slices : 1;
    const int nch = p.hdr[HDR_NCHUNKS], nsj = p.hdr[HDR_NSJOBS], ndc = p.hdr[HDR_DCHUNKS];
    const bool nch_ok = nch >= 0 && nch <= q.max_chunks;
    const bool nsj_ok = nsj >= 0 && nsj <= q.max_sjobs;
    const bool ndc_ok = ndc >= 0 && ndc <= q.max_dchunks;
    if (tid == 0 && !(nch_ok && nsj_ok && ndc_ok)) bad = true;
    const int ntc = p.num_mtiles * nsl;
    bool offs_list_bad = false;
    for (int i = tid; i <= ntc; i += kCheckThreads) {
        const int v = p.tile_chunk_off[i];
        if (v < 0 || v > nch || (i > 0 && p.tile_chunk_off[i - 1] > v) || (i == 0 && v != 0) || (i == ntc && v != nch))
            offs_list_bad = true;
    }
    bad |= offs_list_bad;
    const bool tco_bad = __syncthreads_or(offs_list_bad) != 0;
    for (int c = tid; c < (nch_ok ? nch : 0); c += kCheckThreads) {
        const int32_t r = p.chunk_rng[c];
        if (rng_lo(r) >= rng_hi(r) || rng_hi(r) > kBM || rng_panel(r) >= LORA_MAX_RANK / kChunk) bad = true;
        if (p.chunk_arow[c] < 0 || p.chunk_arow[c] + kChunk > q.a_rows) bad = true;
        if (p.chunk_bpanel[c] < 0 || p.chunk_bpanel[c] >= q.b_panels) bad = true;
    }
    for (int j = tid; j < (nsj_ok ? nsj : 0); j += kCheckThreads) {
        const int m = p.sjob_tile[j], c0 = p.sjob_c0[j], c1 = p.sjob_c1[j];
        if (m < 0 || m >= p.num_mtiles) {
            bad = true;
            continue;
        }
        if (c0 >= c1 || c1 - c0 > kMaxShrinkChunks) bad = true;
        if (!tco_bad && (c0 < p.tile_chunk_off[m * nsl] || c1 > p.tile_chunk_off[(m + 1) * nsl])) bad = true;
    }
    for (int m = tid; m < p.num_mtiles; m += kCheckThreads) {
        const int v = p.tile_njobs[m];
        if (v < 0) bad = true;
        else atomicAdd(&s_njobs, v);
    }

    // ---- the split-K schedule's chunk list --------------------------------------
    for (int c = tid; c < (ndc_ok ? ndc : 0); c += kCheckThreads) {
        const int a = p.dchunk_adapter[c];
        if (a < 0 || a >= A) bad = true;
        if (p.dchunk_arow[c] < 0 || p.dchunk_arow[c] + kChunk > q.a_rows) bad = true;
        if (p.dchunk_bpanel[c] < 0 || p.dchunk_bpanel[c] >= q.b_panels) bad = true;
    }
    __syncthreads();
    if (tid == 0 && nsj_ok && s_njobs != nsj) bad = true;
    const bool any_bad = __syncthreads_or(bad) != 0;
    if (tid == 0) {
        p.hdr[HDR_CHECK] = any_bad ? 1 : 0;
        if (any_bad) atomicOr(p.counters + CNT_STATUS, LORA_DEV_CHECK);
    }
}

// The routing of a mixture-of-experts layer ("Qwen3-MoE low-latency
// inference on Atlas A3", its MoE section: the (token, slot) pairs sorted by
// expert before the grouped matmul), checked against the pairs' experts the
// same way: bucket widths against the counts (bucket 0: ids outside [0, E)),
// perm a stable permutation by bucket, one segment per expert with pairs,
// and the padded order: each expert's pairs, in perm's order, from a fresh
// 128-row tile, -1 in the gaps, each tile's expert, the tile count.
__global__ void __launch_bounds__(kCheckThreads) moe_route_check_kernel(const RouteParams p)
{
    __shared__ int s_off[LORA_MAX_ADAPTERS + 2];
    __shared__ int s_cnt[LORA_MAX_ADAPTERS + 1];
    __shared__ int s_padt[LORA_MAX_ADAPTERS + 2];   // first padded tile of each expert (index e + 1: bucket)
    __shared__ int s_present;
    const int E = p.E, nb = E + 1, tid = threadIdx.x;
    const int64_t P = p.P;
    bool bad = false;
    for (int b = tid; b < nb; b += kCheckThreads) s_cnt[b] = 0;
    for (int b = tid; b <= nb; b += kCheckThreads) s_off[b] = p.offsets[b];
    if (tid == 0) s_present = 0;
    __syncthreads();
    for (int64_t t = tid; t < P; t += kCheckThreads) atomicAdd(&s_cnt[check_bucket(p.expert[t], E)], 1);
    __syncthreads();
    if (tid == 0) {
        bad |= s_off[0] != 0;
        int tiles = 0;   // the padded order's tiles, expert by expert
        for (int b = 1; b < nb; ++b) {
            s_padt[b] = tiles;
            tiles += (s_cnt[b] + kBM - 1) / kBM;
        }
        s_padt[nb] = tiles;
        bad |= tiles > p.max_mtiles || p.hdr[HDR_MOE_TILES] != tiles;
    }
    for (int b = tid; b < nb; b += kCheckThreads) {
        if (s_off[b + 1] - s_off[b] != s_cnt[b]) bad = true;
        if (b >= 1 && s_cnt[b] > 0) atomicAdd(&s_present, 1);
    }
    const bool offs_bad = __syncthreads_or(bad) != 0;

    for (int64_t j = tid; j < P; j += kCheckThreads) {
        const int t = p.perm[j];
        if (t < 0 || t >= P) {
            bad = true;
            continue;
        }
        if (offs_bad) continue;
        int lo = 0, hi = nb - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= j) lo = mid;
            else hi = mid - 1;
        }
        if (check_bucket(p.expert[t], E) != lo) bad = true;
        if (j + 1 < s_off[lo + 1] && p.perm[j + 1] <= t) bad = true;
    }

    const int n = *p.num_segments;
    if (tid == 0 && (n < 0 || n > E || n != s_present || p.hdr[HDR_NSEG] != n)) bad = true;
    for (int s = tid; s < ((n >= 0 && n <= E) ? n : 0); s += kCheckThreads) {
        const int id = p.seg_id[s];
        if (id < 0 || id >= E) {
            bad = true;
            continue;
        }
        if (s > 0 && p.seg_id[s - 1] >= id) bad = true;
        if (p.seg_len[s] != s_cnt[id + 1] || p.seg_len[s] <= 0 || p.seg_rank[s] != 0) bad = true;
        if (!offs_bad && p.seg_start[s] != s_off[id + 1]) bad = true;
    }

    // the padded order (its capacity: max_mtiles tiles of 128 rows)
    if (!offs_bad) {
        const int64_t npad = static_cast<int64_t>(p.max_mtiles) * kBM;
        const int tiles = s_padt[nb];
        for (int64_t i = tid; i < npad; i += kCheckThreads) {
            const int m = static_cast<int>(i / kBM);
            int want = -1;
            if (m < tiles) {
                int lo = 1, hi = nb - 1;   // the expert whose tiles hold m: the last b with s_padt[b] <= m
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_padt[mid] <= m) lo = mid;
                    else hi = mid - 1;
                }
                const int64_t k = i - static_cast<int64_t>(s_padt[lo]) * kBM;
                if (k < s_cnt[lo]) {
                    const int64_t j = s_off[lo] + k;   // its position in perm
                    want = (j >= 0 && j < P) ? p.perm[j] : -2;
                }
                if (i % kBM == 0 && p.mt_expert[m] != lo - 1) bad = true;
            } else if (i % kBM == 0 && p.mt_expert[m] != -1) {
                bad = true;
            }
            if (p.perm_pad[i] != want) bad = true;
        }
    }
    const bool any_bad = __syncthreads_or(bad) != 0;
    if (tid == 0) {
        p.hdr[HDR_CHECK] = any_bad ? 1 : 0;
        if (any_bad) atomicOr(p.counters + CNT_STATUS, LORA_DEV_CHECK);
    }
}

cudaError_t launch_moe_route_check(const RouteParams &p, cudaStream_t stream)
{
    moe_route_check_kernel<<<1, kCheckThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_seg_check(const SegCheckParams &q, cudaStream_t stream)
{
    seg_check_kernel<<<1, kCheckThreads, 0, stream>>>(q);
    return cudaGetLastError();
}

}  // namespace lora
