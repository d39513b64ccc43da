// Tiled schedule of the fused multi-LoRA linear layer on tcgen05.
//
// Page "vLLM-Ascend dynamic LoRA" (pptc.cn/news/149022): §2.3 (tokens grouped
// by adapter into segments, every segment consumed inside ONE operator
// launch), §2.2 (S = x A^T first, then S B^T; never pre-multiplied), §2.4
// (tile M first, then the rank), §4.2 #1 (S accumulated in fp32), §3.4 / §4.1
// (output rows back in the original token order, -1 rows = base only).
//
// Work is a list of jobs executed by a persistent grid (one CTA per SM):
//   shrink job (tile m, chunks c0..c1):  D[128, 16*(c1-c0)] = x_perm[m] A_cat^T
//       over the full K; the epilogue masks every row to its own segment's
//       rank panels, multiplies by scale, rounds to bf16 and parks the panels
//       in an L2-resident scratch, then bumps the tile's ready counter.
//   output job (tile m, tile n):  D[128, 256] = x_perm[m] W[n]^T over K, then
//       extra K-steps  D += S_panel[m, c] B_panel[c, n]^T  for the tile's
//       chunks (S read back through TMA once the ready counter is complete),
//       then + bias, round to bf16, rows scattered to y[perm[row]].
// Shrink jobs come first in the list, so no CTA ever waits on a job that is
// queued behind a waiting job: the grid cannot deadlock (every wait is also
// bounded).
//
// Roles inside a CTA (320 threads):
//   warp 0      TMA producer: W / A / B / S boxes by 2-D tiled loads
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2..5  epilogue: tcgen05.ld -> registers -> global
//   warps 6..9  x loaders: the tile's permuted token rows, 16 bytes per
//               thread by cp.async into the swizzled layout (a row gather
//               costs one LSU request per 16 bytes instead of one TMA
//               instruction per four rows, which the TMA unit issues too
//               slowly to feed the tensor core)
// Smem: one ring of 4 stages, each a 16 KB x slot and a 32 KB W slot under
// one full and one empty barrier (192 KB), 128-byte swizzle for the K-blocks
// of 64, 32-byte swizzle for the 16-wide rank panels.  TMEM: two 256-column
// fp32 accumulators so the epilogue of job j overlaps the mainloop of job
// j+1.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

constexpr int kXSlot = kBM * kBK * 2;         // 16 KB
constexpr int kWSlot = kBN * kBK * 2;         // 32 KB
constexpr int kSPanelBytes = kBM * kChunk * 2;   // 4 KB  (128 rows x 16)
constexpr int kBPanelBytes = kBN * kChunk * 2;   // 8 KB  (256 rows x 16)
constexpr int kAPanelBytes = kChunk * kBK * 2;   // 2 KB  (16 rows x 64)
constexpr int kPanelsPerStage = 2;               // expand step: 2 chunks x (2 S sets x 4 KB + B 8 KB) per W slot
constexpr int kSAreaBytes = 2 * kPanelsPerStage * kSPanelBytes;   // S panels [set][chunk] at the slot's start
constexpr int kTcThreads = 320;   // 10 warps: TMA, MMA, 4 epilogue, 4 x loaders
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;
// The shared memory holds one ring of stages.  A stage is an x slot (the
// loader warps' cp.async row gathers, 16 KB) and a W slot (the producer's
// TMA boxes: W, A panels, or S and B panels, 32 KB) with ONE full barrier,
// which counts the 128 loader threads' copies and the W slot's bytes, and
// one empty barrier.  The MMA thread, whose loop bounds the K steps (the
// tensor pipe queues few MMAs, so every wait and commit between a step's
// MMAs shows), then waits once and commits once per K step.  An expand
// stage has no x rows: its producer arrives for the loader threads.
constexpr int kStages = 4;   // 4 x 48 KB
template <int kStg>
constexpr size_t tc_smem_bytes()
{
    return kStg * (kXSlot + kWSlot) + 1024 /*align*/ + 256 /*barriers*/ + 2 * kBN * 2 /*bias of two tiles*/;
}
static_assert(kSAreaBytes + kPanelsPerStage * kBPanelBytes <= kWSlot, "an expand stage fits in one W slot");

struct Job {
    int kind;   // 0 shrink, 1 output
    int layer;  // the layer of the launch it belongs to
    int m, n, c0, c1;
    int kb0, kb1;   // K blocks of this piece of the job
    int part;       // kPartFull, or a piece of a split output tile: kPartHead (holds K block 0) / kPartTail
    int slot;       // split tile: index of its partial-sum scratch
};

enum { kPartFull = 0, kPartHead = 1, kPartTail = 2 };

// The ring stages of an item after its K steps: its expand steps,
// kPanelsPerStage chunks a stage (an output tile, or the head piece of a
// split one, whose token tile has chunks).  Every role steps through them.
__device__ __forceinline__ int expand_stages(const Job &jb)
{
    return (jb.kind == 1 && jb.c1 > jb.c0 && jb.part != kPartTail)
               ? (jb.c1 - jb.c0 + kPanelsPerStage - 1) / kPanelsPerStage
               : 0;
}

// Item j of the launch: the n_sjobs shrink items of every layer (each
// layer's list alike: the layers share one table), then every layer's
// output tiles.
__device__ __forceinline__ Job decode_job(int j, int n_sjobs, const TcParams &p, int nmt)
{
    Job jb;
    jb.part = kPartFull;
    jb.slot = 0;
    const int nsl = n_sjobs / p.num_layers;   // shrink items of one layer
    if (j < n_sjobs) {
        // shrink item j: K piece jl % S of shrink job jl / S of its layer
        jb.layer = j / nsl;
        const int jl = j - jb.layer * nsl;
        const int S = p.shrink_split, sj = jl / S, h = jl - sj * S;
        const int kb = p.layer[jb.layer].kblocks;
        jb.kind = 0;
        jb.m = p.sjob_tile[sj];
        jb.n = 0;
        jb.c0 = p.sjob_c0[sj];
        jb.c1 = p.sjob_c1[sj];
        jb.kb0 = (kb * h) / S;
        jb.kb1 = (kb * (h + 1)) / S;
        jb.slot = h;   // the S panel set it writes
        return jb;
    }
    int t = j - n_sjobs;
    int l = 0;
    while (l + 1 < p.num_layers && t >= p.layer[l + 1].tile0) ++l;
    const TcLayer &Ly = p.layer[l];
    t -= Ly.tile0;
    jb.layer = l;
    jb.kb0 = 0;
    jb.kb1 = p.mode == kModeExpand ? 0 : Ly.kblocks;
    const int per_group = p.group_m * Ly.num_ntiles;
    const int g = t / per_group, r = t - g * per_group;
    const int m0 = g * p.group_m;
    const int gm = min(p.group_m, nmt - m0);
    jb.kind = 1;
    jb.m = m0 + r % gm;
    jb.n = r / gm;
    if (p.mode == kModeMoe) {   // a plain GEMM tile: no expand steps
        jb.c0 = jb.c1 = 0;
        return jb;
    }
    // the expand steps use the panels of the output slice holding tile n
    int sl = 0;
    for (int k = 1; k < p.num_slices; ++k)
        if (jb.n * kBN >= Ly.slice_start[k]) sl = k;
    jb.c0 = p.tile_chunk_off[jb.m * p.num_slices + sl];
    jb.c1 = p.tile_chunk_off[jb.m * p.num_slices + sl + 1];
    return jb;
}

// The q-th work item of CTA b (false past the last).  Without stream-K the
// CTAs take jobs b, b + G, ...  With stream-K the whole waves are taken that
// way, and the jobs of the last partial wave are shared out: its shrink jobs
// whole (one per CTA, first CTAs), its output tiles as equal runs of K blocks
// over at most sk_pieces(KB) CTAs per tile.  A tile cut between CTAs has one head
// piece (K block 0, last item of its CTA) and tail pieces (first items of the
// next CTAs).  A CTA holds at most one tail piece: each tail stores its
// partial sums in its CTA's own scratch slot and counts itself on the tile's
// counter; the head waits for them, adds them, applies the expand steps and
// writes y.  Nothing is added atomically, so the scratch needs no clearing.
// CTAs per split tile, on average, at most: pieces of about 32 K blocks or
// more, 2 to 4 of them.  Shorter pieces cost more in the partial-sum handoff
// than they save (measured: K = 4096 tiles run faster in 2 pieces than in 4,
// K = 12288 tiles faster in 4 than in 2).
__device__ __forceinline__ int sk_pieces(int KB) { return min(4, max(2, KB / 32)); }

struct SkPlan {
    int nmt;                     // token tiles of this call (kModeMoe: the routing's count)
    int waves, rs, t0, ro, gp;   // whole waves; tail shrink jobs; first tail tile; tail tiles; CTAs sharing them
    int64_t wt;                  // K blocks of the tail tiles
    int64_t dk;                  // K blocks a CTA whose first item is a K piece of a shrink job is ahead by
    int nsj;                     // such CTAs (the first nsj)
};

// First K block (in the tail tiles' K blocks laid end to end) of the range
// of tail-sharing CTA bb: equal runs, plus dk more for each of the first nsj
// CTAs, which end their whole waves early.
__device__ __forceinline__ int64_t sk_start(const SkPlan &s, int bb)
{
    return ((s.wt - s.dk * s.nsj) * bb) / s.gp + s.dk * min(bb, s.nsj);
}

__device__ __forceinline__ SkPlan sk_plan(int n_sjobs, int n_out, int G, int KB, bool streamk, int split)
{
    SkPlan s;
    const int total = n_sjobs + n_out;
    // split only when the last wave would leave a quarter or more of the
    // CTAs idle: otherwise the extra partial-sum epilogues cost more than
    // the idle time they recover
    const int rem = total % G;
    streamk = streamk && rem != 0 && rem * 4 <= G * 3;
    s.waves = streamk ? total / G : (total + G - 1) / G;
    const int jf = s.waves * G;
    s.rs = streamk ? max(0, n_sjobs - jf) : 0;
    s.t0 = streamk ? max(0, jf - n_sjobs) : n_out;
    s.ro = streamk ? n_out - s.t0 : 0;
    s.gp = min(G - s.rs, max(1, s.ro) * sk_pieces(KB));
    s.wt = static_cast<int64_t>(s.ro) * KB;
    // the shrink items (K pieces of 1 / split) are the first wave's first
    // items: those CTAs take the missing K blocks in the last wave
    s.dk = 0;
    s.nsj = 0;
    if (streamk && split > 1 && s.rs == 0 && n_sjobs <= s.gp) {
        const int64_t dk = KB - KB / split;
        if (s.wt > dk * n_sjobs) {
            s.dk = dk;
            s.nsj = n_sjobs;
        }
    }
    return s;
}

__device__ __forceinline__ bool get_item(int q, int b, int G, int n_sjobs, int n_out, const SkPlan &s,
                                         const TcParams &p, Job &jb)
{
    const int total = n_sjobs + n_out;
    if (q < s.waves) {
        const int j = b + q * G;
        if (j >= total) return false;
        jb = decode_job(j, n_sjobs, p, s.nmt);
        return true;
    }
    const int qt = q - s.waves;
    if (b < s.rs) {   // a whole shrink job of the last wave
        if (qt > 0) return false;
        jb = decode_job(s.waves * G + b, n_sjobs, p, s.nmt);
        return true;
    }
    if (s.ro <= 0 || b - s.rs >= s.gp) return false;
    const int KB = p.layer[0].kblocks, bb = b - s.rs;   // stream-K: one layer
    const int64_t r0 = sk_start(s, bb), r1 = sk_start(s, bb + 1);
    int64_t f = r0;
    int t = static_cast<int>(f / KB);
    for (int i = 0; i < qt && f < r1; ++i) {
        ++t;
        f = static_cast<int64_t>(t) * KB;
    }
    if (f >= r1) return false;
    jb = decode_job(n_sjobs + s.t0 + t, n_sjobs, p, s.nmt);
    jb.kb0 = static_cast<int>(f - static_cast<int64_t>(t) * KB);
    jb.kb1 = static_cast<int>(min(r1, static_cast<int64_t>(t + 1) * KB) - static_cast<int64_t>(t) * KB);
    jb.part = jb.kb0 > 0 ? kPartTail : (jb.kb1 < KB ? kPartHead : kPartFull);
    jb.slot = t;
    return true;
}

// The tail pieces of split tile t whose head piece is CTA b are the next
// non-empty tail-sharing CTAs that start inside the tile; a tail's scratch
// slot is its tail-sharing CTA index.  sk_tail_count: how many there are.
// sk_next_tail: the slot of the first tail after slot `after` (the head's
// own index for the first one).
__device__ __forceinline__ int sk_next_tail(int after, const SkPlan &s)
{
    int bb = after + 1;
    while (bb < s.gp && sk_start(s, bb + 1) == sk_start(s, bb)) ++bb;
    return bb;
}

__device__ __forceinline__ int sk_tail_count(int b, int t, const SkPlan &s, int KB)
{
    int n = 0;
    const int64_t end = static_cast<int64_t>(t + 1) * KB;
    for (int bb = b - s.rs + 1; bb < s.gp; ++bb) {
        const int64_t r0 = sk_start(s, bb), r1 = sk_start(s, bb + 1);
        if (r0 >= end) break;
        if (r1 > r0) ++n;
    }
    return n;
}

template <int kStg>
__global__ void __launch_bounds__(kTcThreads, 1) lora_tc_kernel(const __grid_constant__ TcArgs args)
{
    const TcParams &p = args.p;
    const CUtensorMap &tm_s = args.s;
    static_assert(kStg * kWSlot >= kBM * kBN * 4, "a split tile's fp32 partials fit in the W slots");
    static_assert((2 * kStg + 5) * 8 + 16 <= 256, "barriers, TMEM address, abort flag and drain counts fit");
    static_assert(tc_smem_bytes<kStg>() <= 232448, "fits the opt-in shared memory of a CTA");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xring = smem;                                  // the stages' x slots, kStg x 16 KB
    uint8_t *wring = smem + kStg * kXSlot;                  // their W slots, kStg x 32 KB
    uint64_t *full = reinterpret_cast<uint64_t *>(wring + kStg * kWSlot);
    uint64_t *empty = full + kStg;
    uint64_t *acc_full = empty + kStg;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *sk_bar = acc_empty + 2;   // stream-K head: the partial sums have landed in the W ring
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sk_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *drain = const_cast<int *>(abort_flag) + 1;   // for the teardown: [0] stages issued, [1] the last item
    // bias of the output tile of each accumulator slot: [2][kBN] bf16 (16-byte aligned)
    uint32_t *s_bias = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(full) + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t *status = p.counters + CNT_STATUS;
    const long long wait = p.wait_cycles;
    // A programmatic dependent launch: the kernel after this one may place
    // its CTAs on the SMs this grid's CTAs leave, and this grid's CTAs run
    // their prologue while the kernel ahead of them ends (below).
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStg; ++s) {
            mbar_init(&full[s], 128 + 1);   // a cp.async-completion arrive per loader thread, the producer's expect_tx
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 128);
        }
        mbar_init(sk_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&args.maps[0].w);
        tma_prefetch_map(&args.maps[0].a);
        tma_prefetch_map(&args.maps[0].b);
        tma_prefetch_map(&tm_s);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Nothing before this point reads or writes global memory that another
    // kernel produces or consumes: wait for the kernel ahead (its tables,
    // counters, S and outputs) before the first such access.
    pdl_wait();

    // shrink items: every shrink job in p.shrink_split pieces along K
    // LORA_DEBUG build: a segment table (or an expert routing) that failed
    // its check leaves every CTA's work list empty (every CTA reads the same
    // verdict)
    const bool table_bad = kDebugChecks && p.hdr[HDR_CHECK] != 0;
    const int nmt = p.mode == kModeMoe ? min(p.hdr[HDR_MOE_TILES], p.num_mtiles) : p.num_mtiles;
    const int n_sjobs = (p.mode == kModeExpand || p.mode == kModeMoe || table_bad)
                            ? 0 : p.hdr[HDR_NSJOBS] * p.shrink_split * p.num_layers;
    int n_out = 0;   // output tiles of every layer
    if (p.mode != kModeShrink && !table_bad)
        for (int l = 0; l < p.num_layers; ++l) n_out += nmt * p.layer[l].num_ntiles;
    SkPlan sk = sk_plan(n_sjobs, n_out, gridDim.x, p.layer[0].kblocks, p.streamk != 0, p.shrink_split);
    sk.nmt = nmt;
    Job jb;

    if (warp == 0) {
        // ===================== TMA producer: W slots (W, A panels, S / B panels)
        uint32_t it = 0;
        // The S-ready counter of (layer, token tile m) is put back to zero by
        // the last of the layer's num_ntiles output tiles of row m to pass
        // the wait on it: each adds itself to a consumer counter right after
        // the wait (a release: its read of the counter comes first) and reads
        // the result one item later, so the round trip hides behind the
        // loads; the last one takes an acquire fence before the reset, which
        // orders the reset after every consumer's read.
        int32_t *cons = p.counters + CNT_FIXED + p.num_layers * p.num_mtiles;
        int rst_m = -1, rst_old = 0, rst_nt = 0;   // counter index, consumers before me, the layer's tiles per row
        auto settle = [&]() {
            if (rst_m >= 0 && rst_old == rst_nt - 1) {
                fence_acq_rel_gpu();
                p.counters[CNT_FIXED + rst_m] = 0;
                cons[rst_m] = 0;
            }
            rst_m = -1;
        };
        // A stage is refilled only once the MMA has freed it AND its full
        // barrier's previous phase has completed, so this stage's arrives
        // always open a new phase.  In a healthy run the second wait returns
        // at once (the MMA waited for that phase before freeing the stage);
        // after a timeout let a wait go early it keeps an arrive off a phase
        // that still waits for bytes.  A stage that never comes free is
        // skipped.  (The loader warps guard their arrives the same way.)
        auto slot_free = [&](int s, uint32_t round) -> bool {
            int ok = 1;
            if (lane == 0 && round > 0) {
                mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                ok = mbar_wait(&full[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
            }
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        };
        for (int q = 0; get_item(q, blockIdx.x, gridDim.x, n_sjobs, n_out, sk, p, jb); ++q) {
            const TcLayer &Ly = p.layer[jb.layer];
            const TcLayerMaps &mp = args.maps[jb.layer];
            // shrink job: consecutive rank panels of one adapter are
            // consecutive pool rows, loaded as one box of 16..64 rows per run.
            // The runs are found once per job, one lane per chunk: lane c
            // starts a run of run_len panels at pool row run_row, else 0.
            int run_row = 0, run_len = 0;
            // output job: the first B-pool row of the [N, 16] panel of each
            // of the tile's first 32 chunks, one lane per chunk, loaded now
            // for the expand steps
            const int brow_l = (jb.kind == 1 && jb.c0 + lane < jb.c1) ? p.chunk_bpanel[jb.c0 + lane] * Ly.N : 0;
            // kModeMoe: the tile's expert's rows of the stacked expert weights
            const int w_row0 = (p.mode == kModeMoe && jb.kind == 1) ? p.mt_expert[jb.m] * Ly.N : 0;
            if (jb.kind == 0) {
                const int c = jb.c0 + lane;
                const bool in = c < jb.c1;
                const int r = in ? p.chunk_arow[c] : -1;
                const int prev = __shfl_up_sync(0xffffffffu, r, 1);
                const bool start = in && (lane == 0 || prev != r - kChunk);
                const unsigned starts = __ballot_sync(0xffffffffu, start);
                if (start) {
                    // up to the next start or the end of the job, at most 4 panels
                    const unsigned later = starts & ~((2u << lane) - 1u);
                    const int next = later ? __ffs(later) - 1 : jb.c1 - jb.c0;
                    run_row = r;
                    run_len = next - lane;
                }
                // runs longer than 4 panels are split: every 4th panel of a
                // run starts a box (each lane finds its run: the nearest
                // start at or below it)
                const unsigned upto = starts & ((2u << lane) - 1u);
                const int owner_lane = upto ? 31 - __clz(upto) : 0;
                const int owner_row = __shfl_sync(0xffffffffu, run_row, owner_lane);
                const int owner_len = __shfl_sync(0xffffffffu, run_len, owner_lane);
                const int off = lane - owner_lane;   // panel index inside its run
                if (in && off % 4 == 0) {
                    run_row = owner_row + kChunk * off;
                    run_len = min(4, owner_len - off);
                } else {
                    run_len = 0;
                }
            }
            for (int kb = jb.kb0; kb < jb.kb1; ++kb, ++it) {
                const int s = it % kStg;
                if (!slot_free(s, it / kStg)) continue;
                uint8_t *wsl = wring + s * kWSlot;
                if (jb.kind == 1) {
                    if (lane == 0) {
                        mbar_expect_tx(&full[s], kWSlot);
                        tma_load_2d(wsl, &mp.w, &full[s], kb * kBK, jb.n * kBN + w_row0);
                    }
                } else {
                    if (lane == 0) mbar_expect_tx(&full[s], (jb.c1 - jb.c0) * kAPanelBytes);
                    __syncwarp();
                    if (run_len > 0) {
                        const CUtensorMap *m =
                            run_len == 1 ? &mp.a : run_len == 2 ? &mp.a32 : run_len == 3 ? &mp.a48 : &mp.a64;
                        tma_load_2d(wsl + lane * kAPanelBytes, m, &full[s], kb * kBK, run_row);
                    }
                }
                __syncwarp();
            }
            if (jb.kind == 1 && jb.c1 > jb.c0 && jb.part != kPartTail) {
                if (p.mode == kModeLinear) {
                    if (lane == 0) {
                        // every K piece of every shrink job of the tile (this layer's)
                        const int ci = jb.layer * p.num_mtiles + jb.m;
                        wait_flag_geq(p.counters + CNT_FIXED + ci, p.tile_njobs[jb.m] * p.s_sets, abort_flag, status,
                                      LORA_DEV_TIMEOUT, wait);
                        fence_proxy_async_global();
                        settle();
                        rst_old = atom_release_gpu_add(cons + ci, 1);
                        rst_m = ci;
                        rst_nt = Ly.num_ntiles;
                    }
                    __syncwarp();
                }
                for (int cg = jb.c0; cg < jb.c1; cg += kPanelsPerStage, ++it) {
                    const int s = it % kStg;
                    if (!slot_free(s, it / kStg)) continue;
                    uint8_t *wsl = wring + s * kWSlot;   // [S panels [set][chunk] | B panels [chunk]]
                    const int nc = min(kPanelsPerStage, jb.c1 - cg);
                    if (lane == 0) {   // the stage has no x rows: arrive for the loader threads too
                        mbar_expect_tx(&full[s], nc * (p.s_sets * kSPanelBytes + kBPanelBytes));
                        mbar_arrive_n(&full[s], 128);
                    }
                    __syncwarp();
                    const int ci = cg - jb.c0 + lane;   // chunk index inside the tile
                    const int brow_s = __shfl_sync(0xffffffffu, brow_l, ci & 31);
                    if (lane < nc) {
                        const int c = cg + lane;
                        const int brow = ci < 32 ? brow_s : p.chunk_bpanel[c] * Ly.N;
                        for (int h = 0; h < p.s_sets; ++h)
                            tma_load_2d(wsl + (h * kPanelsPerStage + lane) * kSPanelBytes, &tm_s, &full[s], 0,
                                        (jb.layer * p.s_sets + h) * p.s_set_rows + c * kBM);
                        tma_load_2d(wsl + kSAreaBytes + lane * kBPanelBytes, &mp.b, &full[s], 0, brow + jb.n * kBN);
                    }
                    __syncwarp();
                }
            }
        }
        if (lane == 0) {
            settle();
            drain[0] = static_cast<int>(it);
        }
    } else if (warp >= 6) {
        // ===================== x loaders: permuted-row gather (cp.async) =====
        // Thread lt copies 16-byte chunk (lt % 8) of rows lt/8 + 16q, q < 8,
        // into the 128-byte-swizzled x slot; a warp instruction covers four
        // whole 128-byte row segments.  Completion is tracked by the hardware
        // (cp.async.mbarrier.arrive.noinc on the stage's full barrier), so
        // every stage stays in flight; the MMA thread fences the
        // generic-proxy writes for the tensor core's async-proxy reads after
        // its wait.  The loaders step over expand stages (no x rows).
        const int lt = threadIdx.x - 192;
        const int chunk = lt & 7, rb = lt >> 3;
        const uint32_t swz = static_cast<uint32_t>((chunk ^ (rb & 7)) << 4);
        uint32_t it = 0;
        for (int q = 0; get_item(q, blockIdx.x, gridDim.x, n_sjobs, n_out, sk, p, jb); ++q) {
            if (jb.kb1 <= jb.kb0) {
                it += expand_stages(jb);
                continue;
            }
            const TcLayer &Ly = p.layer[jb.layer];
            const uint16_t *src[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                int64_t pp = static_cast<int64_t>(jb.m) * kBM + rb + 16 * q;
                if (pp >= p.M) pp = p.M - 1;
                int64_t row = p.perm[pp];
                if (kDebugChecks && !debug_index_ok(row >= (p.mode == kModeMoe ? -1 : 0) && row < p.out_rows, status))
                    row = 0;
                if (p.mode == kModeMoe) row = row >= 0 ? row / p.topk : 0;   // a pair's token; a gap reads row 0
                src[q] = Ly.x + row * Ly.K + chunk * 8;
            }
            for (int kb = jb.kb0; kb < jb.kb1; ++kb, ++it) {
                const int s = it % kStg;
                const uint32_t round = it / kStg;
                int ok = 1;   // as the producer's slot_free: the full barrier's previous phase has completed
                if (lane == 0 && round > 0) {
                    mbar_wait(&empty[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                    ok = mbar_wait(&full[s], (round - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) continue;
                uint8_t *xs = xring + s * kXSlot + swz;
                const uint32_t nbytes = (kb * kBK + chunk * 8 < Ly.K) ? 16u : 0u;
#pragma unroll
                for (int q = 0; q < 8; ++q) cp_async16(xs + (rb + 16 * q) * 128, src[q] + kb * kBK, nbytes);
                cp_async_mbar_arrive_noinc(&full[s]);
            }
            it += expand_stages(jb);
        }
        cp_async_wait_all();
    } else if (warp == 1) {
        // ===================== MMA issuer ====================================
        // The K steps' operand descriptors: those of slot 0, advanced by the
        // slot's and the 16-wide K step's byte offsets (>> 4) in the start
        // address field (shared-memory offsets stay inside its 14 bits).
        const uint64_t xdesc0 = umma_sdesc(smem_u32(xring), 1024, kSwizzle128);
        const uint64_t wdesc0 = umma_sdesc(smem_u32(wring), 1024, kSwizzle128);
        uint32_t it = 0;
        int last_q = -1;
        for (int q = 0; get_item(q, blockIdx.x, gridDim.x, n_sjobs, n_out, sk, p, jb); ++q) {
            const uint32_t slot = q & 1, use = q >> 1;
            if (use > 0) mbar_wait(&acc_empty[slot], (use - 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
            tc_fence_after();
            const uint32_t d = tmem_base + slot * kAccCols;
            const int n_mma = jb.kind == 0 ? (jb.c1 - jb.c0) * kChunk : kBN;
            const uint32_t idesc = umma_idesc_bf16(kBM, n_mma);
            uint32_t acc = 0;
            for (int kb = jb.kb0; kb < jb.kb1; ++kb, ++it) {
                const int s = it % kStg;
                mbar_wait(&full[s], (it / kStg) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                fence_proxy_async_smem();   // x arrived through the generic proxy (cp.async)
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t xd = xdesc0 + static_cast<uint64_t>((s * kXSlot) >> 4);
                    const uint64_t wd = wdesc0 + static_cast<uint64_t>((s * kWSlot) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {   // 16 K columns of bf16 = 32 bytes
                        umma_bf16(d, xd + 2 * kk, wd + 2 * kk, idesc, acc);
                        acc = 1;
                    }
                    umma_commit(&empty[s]);
                }
                __syncwarp();
            }
            if (jb.kind == 1 && jb.c1 > jb.c0 && jb.part != kPartTail) {
                const uint32_t idesc_e = umma_idesc_bf16(kBM, kBN);
                for (int cg = jb.c0; cg < jb.c1; cg += kPanelsPerStage, ++it) {
                    const int s = it % kStg;
                    mbar_wait(&full[s], (it / kStg) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sa = smem_u32(wring + s * kWSlot);
                        const uint32_t ba = sa + kSAreaBytes;
                        const int nc = min(kPanelsPerStage, jb.c1 - cg);
                        for (int i = 0; i < nc; ++i)
                            for (int h = 0; h < p.s_sets; ++h) {   // (S_0 + S_1) B^T, set by set
                                umma_bf16(d, umma_sdesc(sa + (h * kPanelsPerStage + i) * kSPanelBytes, 256, kSwizzle32),
                                          umma_sdesc(ba + i * kBPanelBytes, 256, kSwizzle32), idesc_e, acc);
                                acc = 1;
                            }
                        umma_commit(&empty[s]);
                    }
                    __syncwarp();
                }
            }
            if (lane == 0) umma_commit(&acc_full[slot]);
            __syncwarp();
            last_q = q;
        }
        if (lane == 0) drain[1] = last_q;
        __syncwarp();
    } else if (warp >= 2) {
        // ===================== epilogue (warps 2..5) =========================
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int et = threadIdx.x - 64;   // 0..127
        for (int q = 0; get_item(q, blockIdx.x, gridDim.x, n_sjobs, n_out, sk, p, jb); ++q) {
            const TcLayer &Ly = p.layer[jb.layer];
            const uint32_t slot = q & 1, use = q >> 1;
            uint32_t *tbias = s_bias + slot * (kBN / 2);   // [kBN / 2] bf16 pairs
            const bool out_bias = jb.kind == 1 && jb.part != kPartTail && p.mode == kModeLinear && Ly.bias;
            if (out_bias) {
                // the tile's 256 bias values, once, while the MMA still runs
                // (the barriers keep the previous tile's readers apart)
                named_bar_sync(1, 128);
                const int col = jb.n * kBN + 2 * et;
                uint32_t bv = 0u;
                if (col + 1 < Ly.N) bv = __ldg(reinterpret_cast<const uint32_t *>(Ly.bias + col));
                else if (col < Ly.N) bv = static_cast<uint32_t>(__ldg(Ly.bias + col));
                tbias[et] = bv;
                named_bar_sync(1, 128);
            }
            // the row's original token, read while the MMA still runs
            const int64_t pp = static_cast<int64_t>(jb.m) * kBM + row;
            // kModeMoe: the output row is the pair itself (-1: a gap of the padded order)
            bool valid = pp < p.M && (p.mode != kModeMoe || p.perm[pp] >= 0);
            int tok = valid ? p.perm[pp] : 0;
            if (kDebugChecks && valid && !debug_index_ok(tok >= 0 && tok < p.out_rows, status)) {
                valid = false;   // this row is neither read by id nor stored
                tok = 0;
            }
            const bool lora_row = p.mode != kModeExpand || pp >= p.offsets[1];
            // the LoRA scale of my row: the call's scale times its adapter's
            // factor (rows outside every segment are masked anyway); the
            // standalone shrink applies the factor alone (an e4m3 pool's A
            // factor; no factor for a bf16 pool: S leaves unscaled)
            float row_sc = p.mode == kModeShrink ? 1.f : Ly.scale;
            if (Ly.adapter_scale && jb.kind == 0 && (p.mode == kModeLinear || p.mode == kModeShrink) && valid) {
                const int id = p.ids[tok];
                row_sc *= (id >= 0 && id < p.num_adapters) ? __ldg(Ly.adapter_scale + id) : 0.f;
            }
            mbar_wait(&acc_full[slot], use & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
            tc_fence_after();
            const uint32_t tbase = tmem_base + slot * kAccCols + (static_cast<uint32_t>(quad * 32) << 16);

            if (jb.kind == 0) {
                // ---- S panels: mask to the row's own segment, scale, bf16 ----
                // (panel set jb.slot of the layer: the K piece of the shrink job)
                uint16_t *panels =
                    p.s_panels + static_cast<int64_t>(jb.layer * p.s_sets + jb.slot) * p.s_set_rows * kChunk;
                for (int c = jb.c0; c < jb.c1; ++c) {
                    uint32_t r[16];
                    tmem_ld16(tbase + (c - jb.c0) * kChunk, r);
                    tmem_ld_wait16(r);
                    const int32_t rng = p.chunk_rng[c];
                    const bool keep = valid && row >= rng_lo(rng) && row < rng_hi(rng);
                    if (p.mode == kModeLinear) {
                        const float sc = keep ? row_sc : 0.f;
                        uint32_t o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            o[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * sc, __uint_as_float(r[2 * e + 1]) * sc);
                        uint4 *dst = reinterpret_cast<uint4 *>(panels + (static_cast<int64_t>(c) * kBM + row) * kChunk);
                        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    } else if (keep) {
                        // standalone shrink: fp32, unscaled, original row, panel
                        // columns (the caller's S starts at zero: K pieces add)
                        float4 *dst = reinterpret_cast<float4 *>(p.s_out + static_cast<int64_t>(tok) * p.s_cols +
                                                                 rng_panel(rng) * kChunk);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const float4 f4 = make_float4(
                                __uint_as_float(r[4 * v]) * row_sc, __uint_as_float(r[4 * v + 1]) * row_sc,
                                __uint_as_float(r[4 * v + 2]) * row_sc, __uint_as_float(r[4 * v + 3]) * row_sc);
                            if (p.shrink_split > 1) atomicAdd(dst + v, f4);
                            else dst[v] = f4;
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&acc_empty[slot]);
                if (p.mode == kModeLinear) {
                    fence_proxy_async_global();
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (et == 0) red_release_gpu_add(p.counters + CNT_FIXED + jb.layer * p.num_mtiles + jb.m, 1);
                }
            } else if (jb.part == kPartTail) {
                // ---- tail piece of a split tile: store my partial sums --------
                // in my CTA's scratch slot, layout [col / 4][row][4]: a warp's
                // float4 accesses cover 512 contiguous bytes
                float4 *part = reinterpret_cast<float4 *>(p.sk_part) +
                               static_cast<int64_t>(blockIdx.x - sk.rs) * (kBN / 4) * kBM;
                // four 16-column TMEM loads per wait (one group at a time: the
                // register budget holds no more)
#pragma unroll 1
                for (int cc = 0; cc < kBN / 16; cc += 4) {
                    uint32_t r[4][16];
#pragma unroll
                    for (int h = 0; h < 4; ++h) tmem_ld16(tbase + (cc + h) * 16, r[h]);
                    tmem_ld_wait16(r[0]);
#pragma unroll
                    for (int h = 1; h < 4; ++h) tmem_regs_after_wait16(r[h]);
                    if (cc + 4 == kBN / 16) {
                        tc_fence_before();
                        mbar_arrive(&acc_empty[slot]);
                    }
#pragma unroll
                    for (int h = 0; h < 4; ++h)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float4 f4 =
                                make_float4(__uint_as_float(r[h][4 * k]), __uint_as_float(r[h][4 * k + 1]),
                                            __uint_as_float(r[h][4 * k + 2]), __uint_as_float(r[h][4 * k + 3]));
                            __stcg(part + ((cc + h) * 4 + k) * kBM + row, f4);
                        }
                }
                __threadfence();
                named_bar_sync(1, 128);
                if (et == 0) red_release_gpu_add(p.sk_cnt + jb.slot * kWinCntStride, 1);
            } else {
                // ---- output tile (whole, or the head piece of a split tile):
                // + the tails' partial sums, + bias, bf16, scatter to the
                // original row ----------------------------------------------
                const int n0 = jb.n * kBN;
                const bool head = jb.part == kPartHead;
                // the head is its CTA's last item: the W ring is idle now, and
                // the first tail's partials (128 KB) come in by four bulk
                // copies; further tails' are added from L2
                const float4 *spart = reinterpret_cast<const float4 *>(wring);
                int ntail = 0, tail0 = 0;
                if (head) {
                    ntail = sk_tail_count(blockIdx.x, jb.slot, sk, Ly.kblocks);
                    tail0 = sk_next_tail(blockIdx.x - sk.rs, sk);
                    if (et == 0) {   // every tail piece has stored its partial sums
                        wait_flag_geq(p.sk_cnt + jb.slot * kWinCntStride, ntail, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                        fence_proxy_async_global();   // their stores -> the bulk copies' reads
                        mbar_expect_tx(sk_bar, kBM * kBN * 4);
                        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.sk_part) +
                                             static_cast<int64_t>(tail0) * kBM * kBN * 4;
                        for (int i = 0; i < 4; ++i) bulk_load(wring + i * kWSlot, src + i * kWSlot, kWSlot, sk_bar);
                    }
                    mbar_wait(sk_bar, 0, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                    // further tails: each thread adds them into its own row of
                    // the shared-memory copy, sixteen loads in flight at a time
                    float4 *sp = reinterpret_cast<float4 *>(wring);
                    for (int i = 1, ts = tail0; i < ntail; ++i) {
                        ts = sk_next_tail(ts, sk);
                        const float4 *xp =
                            reinterpret_cast<const float4 *>(p.sk_part) + static_cast<int64_t>(ts) * (kBN / 4) * kBM;
#pragma unroll 1
                        for (int k0 = 0; k0 < kBN / 4; k0 += 16) {
                            float4 b[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k) b[k] = __ldcg(xp + (k0 + k) * kBM + row);
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const float4 a = sp[(k0 + k) * kBM + row];
                                sp[(k0 + k) * kBM + row] =
                                    make_float4(a.x + b[k].x, a.y + b[k].y, a.z + b[k].z, a.w + b[k].w);
                            }
                        }
                    }
                }
                // one 16-column chunk: + partials, + bias (from shared memory) or
                // the existing y (standalone expand), bf16, store to the row
                auto emit = [&](int cc, const uint32_t (&r)[16]) {
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
                    if (head) {   // the tails' summed partials, from shared memory
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float4 pv = spart[(cc * 4 + k) * kBM + row];
                            v[4 * k] += pv.x;
                            v[4 * k + 1] += pv.y;
                            v[4 * k + 2] += pv.z;
                            v[4 * k + 3] += pv.w;
                        }
                    }
                    const int col = n0 + cc * 16;
                    if (!valid || col >= Ly.N || !lora_row) return;
                    uint16_t *dst = Ly.y + static_cast<int64_t>(tok) * Ly.N + col;
                    if (p.mode == kModeExpand) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(dst);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (col + 8 * h >= Ly.N) break;
                            const uint4 u = src[h];
                            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                v[8 * h + 2 * e] += bf16_lo(w4[e]);
                                v[8 * h + 2 * e + 1] += bf16_hi(w4[e]);
                            }
                        }
                    } else if (out_bias) {
                        const uint4 *bsrc = reinterpret_cast<const uint4 *>(tbias + cc * 8);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint4 u = bsrc[h];
                            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                v[8 * h + 2 * e] += bf16_lo(w4[e]);
                                v[8 * h + 2 * e + 1] += bf16_hi(w4[e]);
                            }
                        }
                    }
                    uint4 *o = reinterpret_cast<uint4 *>(dst);
                    o[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                      pack_bf16x2(v[6], v[7]));
                    if (col + 8 < Ly.N)
                        o[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                                          pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
                };
                // four chunks per TMEM wait
                for (int cc = 0; cc < kBN / 16; cc += 4) {
                    uint32_t r[4][16];
#pragma unroll
                    for (int h = 0; h < 4; ++h) tmem_ld16(tbase + (cc + h) * 16, r[h]);
                    tmem_ld_wait16(r[0]);
#pragma unroll
                    for (int h = 1; h < 4; ++h) tmem_regs_after_wait16(r[h]);
                    if (cc + 4 == kBN / 16) {
                        tc_fence_before();
                        mbar_arrive(&acc_empty[slot]);
                    }
#pragma unroll
                    for (int h = 0; h < 4; ++h) emit(cc + h, r[h]);
                }
                if (head && et == 0) {
                    p.sk_cnt[jb.slot * kWinCntStride] = 0;   // zero again for the next call
                    // the partial sums' bulk copies have landed before the CTA
                    // ends, even if the wait above gave up after a timeout
                    mbar_wait(sk_bar, 0, abort_flag, status, LORA_DEV_TIMEOUT, wait);
                }
            }
        }
    }

    // ---- teardown ---------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // After a timeout let a wait of this CTA go early, its loads and MMAs
    // still in flight are waited for (bounded) before the tensor memory is
    // freed and the CTA ends: the last phase of each stage (the producer's
    // bytes and the loader warps' copies) and the last commit, which covers
    // every MMA.  In a healthy run every one of them has been waited for.
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t it = static_cast<uint32_t>(drain[0]);
            for (uint32_t i = it > kStg ? it - kStg : 0; i < it; ++i)
                mbar_wait(&full[i % kStg], (i / kStg) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
        }
        if (warp == 1 && lane == 0 && drain[1] >= 0)
            mbar_wait(&acc_full[drain[1] & 1], (drain[1] >> 1) & 1, abort_flag, status, LORA_DEV_TIMEOUT, wait);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// Standalone expand: turn the caller's fp32 S [M, s_cols] (original token
// order) into the kernel's bf16 S panels (permuted tile rows, each row masked
// to its own segment's rank panels, multiplied by scale and by its adapter's
// factor).  One CTA per token tile, one thread per tile row.
__global__ void __launch_bounds__(kBM) s_prep_kernel(const float *S, int32_t s_cols, float scale, TcParams p)
{
    const int m = blockIdx.x, row = threadIdx.x;
    if (kDebugChecks && p.hdr[HDR_CHECK] != 0) return;   // LORA_DEBUG: the table failed its check
    const int64_t pp = static_cast<int64_t>(m) * kBM + row;
    const bool valid = pp < p.M;
    const int tok = valid ? p.perm[pp] : 0;
    if (p.layer[0].adapter_scale && valid) {
        const int id = p.ids[tok];
        scale *= (id >= 0 && id < p.num_adapters) ? p.layer[0].adapter_scale[id] : 0.f;
    }
    for (int c = p.tile_chunk_off[m * p.num_slices]; c < p.tile_chunk_off[(m + 1) * p.num_slices]; ++c) {
        const int32_t rng = p.chunk_rng[c];
        const bool keep = valid && row >= rng_lo(rng) && row < rng_hi(rng);
        const float *src = S + static_cast<int64_t>(tok) * s_cols + rng_panel(rng) * kChunk;
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            w[e] = keep ? pack_bf16x2(src[2 * e] * scale, src[2 * e + 1] * scale) : 0u;
        uint4 *dst = reinterpret_cast<uint4 *>(p.s_panels + (static_cast<int64_t>(c) * kBM + row) * kChunk);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

cudaError_t launch_s_prep(const float *S, int32_t s_cols, float scale, const TcParams &p, cudaStream_t stream)
{
    s_prep_kernel<<<p.num_mtiles, kBM, 0, stream>>>(S, s_cols, scale, p);
    return cudaGetLastError();
}

template <int kStg>
static cudaError_t launch_tc_split(const TcArgs &args, int grid, cudaStream_t stream)
{
    constexpr size_t smem = tc_smem_bytes<kStg>();
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(lora_tc_kernel<kStg>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (dev < 64) configured[dev] = 1;
    }
    // a programmatic dependent launch: the CTAs start their prologue as the
    // kernel ahead releases SMs, and wait for it before touching its data
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lora_tc_kernel<kStg>, args);
}

cudaError_t launch_tc(const TcArgs &args, int grid, cudaStream_t stream)
{
    return launch_tc_split<kStages>(args, grid, stream);
}

}  // namespace lora
