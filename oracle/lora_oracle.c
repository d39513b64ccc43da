/*
 * CPU oracle for the fused dynamic multi-LoRA linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * Every result is computed in fp64 from the exact bf16 inputs widened to
 * double, with plain loops in index order (no blocking, no fusion, no
 * reordering).  The only parallelism is OpenMP over independent output rows.
 *
 * Source: "vLLM-Ascend dynamic LoRA" (pptc.cn/news/149022):
 *   §1.1  y = x W^T + (x A^T) B^T, A is [r, K], B is [N, r]
 *   §2.1  per-token lora_id_map, -1 = no LoRA, nullable bias, output [M, N]
 *   §2.2  two steps: S = x A^T, then y_lora = S B^T (never pre-multiplied)
 *   §2.3  bucketing by lora_id into contiguous segments (id, tokens, rank)
 *   §3.4  rows with id -1 carry the base output unchanged
 *   §4.3  ranks padded to a multiple of 16 with zero rows / columns
 * The per-call scalar `scale` multiplying the LoRA term is this project's
 * reading (the page's formula has an implicit scale of 1).
 * A merged output (Q|K|V, gate|up: one adapter pair per output slice, as a
 * merged projection with LoRA needs it; the page's §3.3 names the merged QKV
 * shape) is oracle_lora_linear_slices_rows, the same formula per slice.
 *
 * Adapter storage here is the oracle's own, deliberately naive layout:
 * adapter i's A_i [r_i, K] row-major starts right after A_{i-1}, and
 * B_i [N, r_i] row-major starts right after B_{i-1}, using TRUE ranks.
 *
 * Adapters may also be given as 8-bit floats (e4m3) with one fp64 dequant
 * factor per adapter and factor: A_i = a_deq_i * e4m3(a), B_i = b_deq_i *
 * e4m3(b) (the *_e4m3 functions; this project's extension, the page stores
 * adapters in the model's own precision).  The 8-bit codes are decoded
 * exactly from the format's definition (oracle_e4m3_to_f64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE fp32: widening is a 16-bit shift. */
static double bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* An id is usable when it names an adapter; anything else (including ids
 * below -1 or past the last adapter) is treated as "no LoRA". */
static int32_t effective_id(int32_t id, int32_t num_adapters)
{
    return (id >= 0 && id < num_adapters) ? id : -1;
}

/* Start of adapter i in the oracle's concatenated A (elements). */
static int64_t a_start(const int32_t *rank, int32_t i, int64_t K)
{
    int64_t s = 0;
    for (int32_t j = 0; j < i; ++j) s += (int64_t)rank[j] * K;
    return s;
}

/* Start of adapter i in the oracle's concatenated B (elements). */
static int64_t b_start(const int32_t *rank, int32_t i, int64_t N)
{
    int64_t s = 0;
    for (int32_t j = 0; j < i; ++j) s += N * (int64_t)rank[j];
    return s;
}

/*
 * Segment table (§2.3): a stable counting sort of the tokens by key id+1.
 *   bucket 0 holds the id -1 tokens, bucket b>0 holds adapter b-1;
 *   cnt[b]   = number of tokens in bucket b
 *   off[0]   = 0, off[b+1] = off[b] + cnt[b]          (A+2 entries)
 *   perm[off[b] + (number of earlier tokens in bucket b)] = t
 *   one segment per non-empty adapter bucket, ascending id:
 *     (id, start = off[id+1], len = cnt[id+1], rank = padded rank)
 * The padded rank is r rounded up to a multiple of 16 (§4.3).
 * Returns the number of ids that named no adapter (they are sorted as -1).
 */
int oracle_build_segments(const int32_t *ids, int64_t M, int32_t num_adapters,
                          const int32_t *true_rank, int32_t *perm, int32_t *bucket_offsets,
                          int32_t *seg_id, int32_t *seg_start, int32_t *seg_len,
                          int32_t *seg_rank, int32_t *num_segments)
{
    int64_t nb = (int64_t)num_adapters + 1;
    int64_t *cnt = (int64_t *)calloc((size_t)nb, sizeof(int64_t));
    int64_t *next = (int64_t *)calloc((size_t)nb, sizeof(int64_t));
    int invalid = 0;
    for (int64_t t = 0; t < M; ++t) {
        int32_t e = effective_id(ids[t], num_adapters);
        if (e != ids[t]) invalid++;
        cnt[e + 1]++;
    }
    bucket_offsets[0] = 0;
    for (int64_t b = 0; b < nb; ++b) bucket_offsets[b + 1] = (int32_t)(bucket_offsets[b] + cnt[b]);
    for (int64_t b = 0; b < nb; ++b) next[b] = bucket_offsets[b];
    for (int64_t t = 0; t < M; ++t) {   /* visiting t in order keeps the sort stable */
        int32_t e = effective_id(ids[t], num_adapters);
        perm[next[e + 1]++] = (int32_t)t;
    }
    int32_t ns = 0;
    for (int32_t i = 0; i < num_adapters; ++i) {
        if (cnt[i + 1] == 0) continue;
        seg_id[ns] = i;
        seg_start[ns] = bucket_offsets[i + 1];
        seg_len[ns] = (int32_t)cnt[i + 1];
        seg_rank[ns] = ((true_rank[i] + 15) / 16) * 16;
        ns++;
    }
    *num_segments = ns;
    free(cnt);
    free(next);
    return invalid;
}

/*
 * The layer, for a chosen set of output rows (all rows when rows == NULL):
 *   base[t,n] = sum_k x[t,k] W[n,k] + bias[n]
 *   id -1:      y[t,n] = base[t,n]
 *   id i >= 0:  S[t,j] = sum_k x[t,k] A_i[j,k]              (j < r_i)
 *               y[t,n] = base[t,n] + scale * s_i * sum_j S[t,j] B_i[n,j]
 * where s_i = adapter_scale[i] (1 when adapter_scale is NULL): an optional
 * per-adapter factor on the LoRA term (this project's extension; the
 * page's formula has one implicit scale of 1).
 * y is [nrows, N] fp64, row q holding token rows[q].
 */
void oracle_lora_linear_rows(const uint16_t *x, int64_t M, int64_t K,
                             const uint16_t *W, int64_t N, const uint16_t *bias,
                             const int32_t *ids, int32_t num_adapters, const int32_t *rank,
                             const uint16_t *a_cat, const uint16_t *b_cat, double scale,
                             const double *adapter_scale, const int64_t *rows, int64_t nrows, double *y)
{
    (void)M;
#pragma omp parallel
    {
        double *xr = (double *)malloc((size_t)K * sizeof(double));
        double *S = (double *)malloc(64 * 1024 * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < nrows; ++q) {
            int64_t t = rows ? rows[q] : q;
            for (int64_t k = 0; k < K; ++k) xr[k] = bf16_to_f64(x[t * K + k]);
            double *yr = y + q * N;
            /* base GEMM row, then bias */
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += xr[k] * bf16_to_f64(W[n * K + k]);
                if (bias) acc += bf16_to_f64(bias[n]);
                yr[n] = acc;
            }
            int32_t i = effective_id(ids[t], num_adapters);
            if (i < 0) continue;               /* §3.4: -1 rows pass through */
            int64_t r = rank[i];
            const uint16_t *Ai = a_cat + a_start(rank, i, K);
            const uint16_t *Bi = b_cat + b_start(rank, i, N);
            /* step 1 (§2.2): S = x A_i^T */
            for (int64_t j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += xr[k] * bf16_to_f64(Ai[j * K + k]);
                S[j] = acc;
            }
            /* step 2 (§2.2): y += scale * s_i * S B_i^T */
            double si = adapter_scale ? adapter_scale[i] : 1.0;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t j = 0; j < r; ++j) acc += S[j] * bf16_to_f64(Bi[n * r + j]);
                yr[n] += scale * si * acc;
            }
        }
        free(xr);
        free(S);
    }
}

/*
 * Step 1 alone (§2.2): S[t, j] = sum_k x[t,k] A_{id(t)}[j,k] for j < r_id,
 * and 0 for j >= r_id and for rows whose id is -1.  S is [nrows, s_cols].
 */
void oracle_shrink_rows(const uint16_t *x, int64_t M, int64_t K, const int32_t *ids,
                        int32_t num_adapters, const int32_t *rank, const uint16_t *a_cat,
                        const int64_t *rows, int64_t nrows, int64_t s_cols, double *S)
{
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < nrows; ++q) {
        int64_t t = rows ? rows[q] : q;
        double *Sr = S + q * s_cols;
        for (int64_t j = 0; j < s_cols; ++j) Sr[j] = 0.0;
        int32_t i = effective_id(ids[t], num_adapters);
        if (i < 0) continue;
        const uint16_t *Ai = a_cat + a_start(rank, i, K);
        for (int64_t j = 0; j < rank[i] && j < s_cols; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_f64(x[t * K + k]) * bf16_to_f64(Ai[j * K + k]);
            Sr[j] = acc;
        }
    }
}

/*
 * Step 2 alone (§2.2, §2.3 "added to the y_base rows"), given S:
 *   y[t,n] = y_in[t,n] + scale * s_id * sum_{j < r_id} S[t,j] B_id[n,j]   (id >= 0)
 *   y[t,n] = y_in[t,n]                                                  (id == -1)
 * S is fp32 [M, s_cols] (the given input, widened exactly); y_in is bf16;
 * s_id as in oracle_lora_linear_rows.
 */
void oracle_expand_rows(const float *S, int64_t s_cols, const uint16_t *y_in, int64_t N,
                        const int32_t *ids, int32_t num_adapters, const int32_t *rank,
                        const uint16_t *b_cat, double scale, const double *adapter_scale,
                        const int64_t *rows, int64_t nrows, double *y)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < nrows; ++q) {
        int64_t t = rows ? rows[q] : q;
        double *yr = y + q * N;
        for (int64_t n = 0; n < N; ++n) yr[n] = bf16_to_f64(y_in[t * N + n]);
        int32_t i = effective_id(ids[t], num_adapters);
        if (i < 0) continue;
        int64_t r = rank[i];
        const uint16_t *Bi = b_cat + b_start(rank, i, N);
        double si = adapter_scale ? adapter_scale[i] : 1.0;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < r && j < s_cols; ++j)
                acc += (double)S[t * s_cols + j] * bf16_to_f64(Bi[n * r + j]);
            yr[n] += scale * si * acc;
        }
    }
}

/*
 * Selected single elements y[rows[q], cols[q]] of the layer (same definition
 * as oracle_lora_linear_rows, evaluated element by element; S is recomputed
 * for every element).  Used for bounded samples of large workloads.
 */
void oracle_lora_linear_elems(const uint16_t *x, int64_t K, const uint16_t *W, int64_t N,
                              const uint16_t *bias, const int32_t *ids, int32_t num_adapters,
                              const int32_t *rank, const uint16_t *a_cat, const uint16_t *b_cat,
                              double scale, const double *adapter_scale, const int64_t *rows,
                              const int64_t *cols, int64_t n, double *y)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t q = 0; q < n; ++q) {
        int64_t t = rows[q], c = cols[q];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += bf16_to_f64(x[t * K + k]) * bf16_to_f64(W[c * K + k]);
        if (bias) acc += bf16_to_f64(bias[c]);
        int32_t i = effective_id(ids[t], num_adapters);
        if (i >= 0) {
            int64_t r = rank[i];
            const uint16_t *Ai = a_cat + a_start(rank, i, K);
            const uint16_t *Bi = b_cat + b_start(rank, i, N);
            double lora = 0.0;
            for (int64_t j = 0; j < r; ++j) {
                double s = 0.0;
                for (int64_t k = 0; k < K; ++k) s += bf16_to_f64(x[t * K + k]) * bf16_to_f64(Ai[j * K + k]);
                lora += s * bf16_to_f64(Bi[c * r + j]);
            }
            acc += scale * (adapter_scale ? adapter_scale[i] : 1.0) * lora;
        }
        y[q] = acc;
    }
}

/*
 * The layer with a merged output (Q|K|V, gate|up, ...): the output columns
 * are cut into nslices slices [slice_start[s], slice_start[s+1]) and adapter
 * i has one pair per slice, A_i^s [r_i, K] and B_i^s [N_s, r_i] with
 * N_s = slice_start[s+1] - slice_start[s].  For a token of adapter i and an
 * output column n of slice s:
 *   y[t,n] = base[t,n] + scale * s_i * sum_j S^s[t,j] B_i^s[n - slice_start[s], j],
 *   S^s[t,j] = sum_k x[t,k] A_i^s[j,k]
 * a_cat holds A_i^s row-major, adapter-major then slice; b_cat holds B_i^s
 * row-major, adapter-major then slice.  Rows as in oracle_lora_linear_rows.
 */
void oracle_lora_linear_slices_rows(const uint16_t *x, int64_t M, int64_t K,
                                    const uint16_t *W, int64_t N, const uint16_t *bias,
                                    const int32_t *ids, int32_t num_adapters, const int32_t *rank,
                                    int32_t nslices, const int64_t *slice_start,
                                    const uint16_t *a_cat, const uint16_t *b_cat, double scale,
                                    const double *adapter_scale, const int64_t *rows, int64_t nrows, double *y)
{
    (void)M;
#pragma omp parallel
    {
        double *xr = (double *)malloc((size_t)K * sizeof(double));
        double *S = (double *)malloc(64 * 1024 * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < nrows; ++q) {
            int64_t t = rows ? rows[q] : q;
            for (int64_t k = 0; k < K; ++k) xr[k] = bf16_to_f64(x[t * K + k]);
            double *yr = y + q * N;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += xr[k] * bf16_to_f64(W[n * K + k]);
                if (bias) acc += bf16_to_f64(bias[n]);
                yr[n] = acc;
            }
            int32_t i = effective_id(ids[t], num_adapters);
            if (i < 0) continue;
            int64_t r = rank[i];
            int64_t a0 = 0, b0 = 0;   /* adapter i's first element in a_cat / b_cat */
            for (int32_t j = 0; j < i; ++j) {
                a0 += (int64_t)nslices * rank[j] * K;
                b0 += N * (int64_t)rank[j];
            }
            double si = adapter_scale ? adapter_scale[i] : 1.0;
            for (int32_t s = 0; s < nslices; ++s) {
                const uint16_t *As = a_cat + a0 + (int64_t)s * r * K;
                const uint16_t *Bs = b_cat + b0 + slice_start[s] * r;
                for (int64_t j = 0; j < r; ++j) {
                    double acc = 0.0;
                    for (int64_t k = 0; k < K; ++k) acc += xr[k] * bf16_to_f64(As[j * K + k]);
                    S[j] = acc;
                }
                for (int64_t n = slice_start[s]; n < slice_start[s + 1]; ++n) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < r; ++j) acc += S[j] * bf16_to_f64(Bs[(n - slice_start[s]) * r + j]);
                    yr[n] += scale * si * acc;
                }
            }
        }
        free(xr);
        free(S);
    }
}

/*
 * Mixture-of-experts layer with grouped expert GEMMs (the page "Qwen3-MoE
 * low-latency inference on Atlas A3", mokono.cn/news/2297686, its MoE section:
 * route the tokens to their experts, one grouped matmul over all experts,
 * then put the rows back and sum them with the routing weights):
 *   y[t,n] = sum_{j < topk, e = expert[t,j] valid} weight[t,j] * sum_k x[t,k] W_e[n,k]
 * expert ids outside [0, num_experts) contribute nothing.  W holds the
 * experts' [N, K] weights one after another.  Rows as in
 * oracle_lora_linear_rows.
 */
void oracle_moe_rows(const uint16_t *x, int64_t M, int64_t K, const uint16_t *W, int64_t N, int32_t num_experts,
                     int32_t topk, const int32_t *expert, const float *weight, const int64_t *rows, int64_t nrows,
                     double *y)
{
    (void)M;
#pragma omp parallel
    {
        double *xr = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < nrows; ++q) {
            int64_t t = rows ? rows[q] : q;
            for (int64_t k = 0; k < K; ++k) xr[k] = bf16_to_f64(x[t * K + k]);
            double *yr = y + q * N;
            for (int64_t n = 0; n < N; ++n) yr[n] = 0.0;
            for (int32_t j = 0; j < topk; ++j) {
                int32_t e = expert[t * topk + j];
                if (e < 0 || e >= num_experts) continue;
                double w = (double)weight[t * topk + j];
                const uint16_t *We = W + (int64_t)e * N * K;
                for (int64_t n = 0; n < N; ++n) {
                    double acc = 0.0;
                    for (int64_t k = 0; k < K; ++k) acc += xr[k] * bf16_to_f64(We[n * K + k]);
                    yr[n] += w * acc;
                }
            }
        }
        free(xr);
    }
}

/*
 * e4m3, the 8-bit float with 1 sign bit, 4 exponent bits (bias 7) and 3
 * mantissa bits, no infinities (OCP 8-bit floating point, "E4M3"):
 *   exponent field e = 0:      (-1)^s * (m / 8) * 2^-6          (subnormal)
 *   e = 1..15:                 (-1)^s * (1 + m / 8) * 2^(e - 7)
 *   e = 15 with m = 7:         NaN (the largest finite value is 448)
 */
double oracle_e4m3_to_f64(uint8_t v)
{
    int s = v >> 7, e = (v >> 3) & 15, m = v & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/*
 * oracle_lora_linear_rows with e4m3 adapters: the same layer, with
 *   A_i[j,k] = deq[2i] * e4m3(a8_i[j,k]),  B_i[n,j] = deq[2i+1] * e4m3(b8_i[n,j])
 * (a8_cat / b8_cat in the oracle's concatenated true-rank layout, one byte
 * per element; deq: [num_adapters][2] fp64).
 */
void oracle_lora_linear_rows_e4m3(const uint16_t *x, int64_t M, int64_t K,
                                  const uint16_t *W, int64_t N, const uint16_t *bias,
                                  const int32_t *ids, int32_t num_adapters, const int32_t *rank,
                                  const uint8_t *a8_cat, const uint8_t *b8_cat, const double *deq, double scale,
                                  const double *adapter_scale, const int64_t *rows, int64_t nrows, double *y)
{
    (void)M;
#pragma omp parallel
    {
        double *xr = (double *)malloc((size_t)K * sizeof(double));
        double *S = (double *)malloc(64 * 1024 * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < nrows; ++q) {
            int64_t t = rows ? rows[q] : q;
            for (int64_t k = 0; k < K; ++k) xr[k] = bf16_to_f64(x[t * K + k]);
            double *yr = y + q * N;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += xr[k] * bf16_to_f64(W[n * K + k]);
                if (bias) acc += bf16_to_f64(bias[n]);
                yr[n] = acc;
            }
            int32_t i = effective_id(ids[t], num_adapters);
            if (i < 0) continue;
            int64_t r = rank[i];
            const uint8_t *Ai = a8_cat + a_start(rank, i, K);
            const uint8_t *Bi = b8_cat + b_start(rank, i, N);
            for (int64_t j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) acc += xr[k] * (deq[2 * i] * oracle_e4m3_to_f64(Ai[j * K + k]));
                S[j] = acc;
            }
            double si = adapter_scale ? adapter_scale[i] : 1.0;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t j = 0; j < r; ++j) acc += S[j] * (deq[2 * i + 1] * oracle_e4m3_to_f64(Bi[n * r + j]));
                yr[n] += scale * si * acc;
            }
        }
        free(xr);
        free(S);
    }
}

/* oracle_shrink_rows with e4m3 adapters (A_i as in oracle_lora_linear_rows_e4m3). */
void oracle_shrink_rows_e4m3(const uint16_t *x, int64_t M, int64_t K, const int32_t *ids,
                             int32_t num_adapters, const int32_t *rank, const uint8_t *a8_cat, const double *deq,
                             const int64_t *rows, int64_t nrows, int64_t s_cols, double *S)
{
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < nrows; ++q) {
        int64_t t = rows ? rows[q] : q;
        double *Sr = S + q * s_cols;
        for (int64_t j = 0; j < s_cols; ++j) Sr[j] = 0.0;
        int32_t i = effective_id(ids[t], num_adapters);
        if (i < 0) continue;
        const uint8_t *Ai = a8_cat + a_start(rank, i, K);
        for (int64_t j = 0; j < rank[i] && j < s_cols; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_f64(x[t * K + k]) * (deq[2 * i] * oracle_e4m3_to_f64(Ai[j * K + k]));
            Sr[j] = acc;
        }
    }
}

/* oracle_expand_rows with e4m3 adapters (B_i as in oracle_lora_linear_rows_e4m3). */
void oracle_expand_rows_e4m3(const float *S, int64_t s_cols, const uint16_t *y_in, int64_t N,
                             const int32_t *ids, int32_t num_adapters, const int32_t *rank,
                             const uint8_t *b8_cat, const double *deq, double scale, const double *adapter_scale,
                             const int64_t *rows, int64_t nrows, double *y)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < nrows; ++q) {
        int64_t t = rows ? rows[q] : q;
        double *yr = y + q * N;
        for (int64_t n = 0; n < N; ++n) yr[n] = bf16_to_f64(y_in[t * N + n]);
        int32_t i = effective_id(ids[t], num_adapters);
        if (i < 0) continue;
        int64_t r = rank[i];
        const uint8_t *Bi = b8_cat + b_start(rank, i, N);
        double si = adapter_scale ? adapter_scale[i] : 1.0;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < r && j < s_cols; ++j)
                acc += (double)S[t * s_cols + j] * (deq[2 * i + 1] * oracle_e4m3_to_f64(Bi[n * r + j]));
            yr[n] += scale * si * acc;
        }
    }
}
