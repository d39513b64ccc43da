// Mixture-of-experts finalize (the pages' MoE section: after the grouped
// expert matmul, put every token's rows back and sum them with the routing
// weights).  The routing is the segment builder in routing mode and the
// grouped GEMM is the tiled kernel in kModeMoe; this file holds the last step.
//
//   y[t, n] = bf16( sum_{j < topk, expert[t,j] valid} weight[t,j] * out[t * topk + j, n] )
//
// out holds the experts' bf16 rows in (token, slot) pair order.  Memory-bound:
// one thread per 8 output columns of one token, 16-byte loads and stores,
// coalesced along n; the fp32 sum runs in the slots' order.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

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
