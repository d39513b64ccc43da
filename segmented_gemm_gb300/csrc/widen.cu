// e4m3 adapter pools for the schedules that read bf16 operands through TMA
// (the tiled and split-K schedules, the standalone shrink and expand): the
// adapters a batch uses are widened into the pool's bf16 scratch, at the
// same element offsets, before the fused launch.  Every e4m3 value is a
// bf16 value, so the widening is exact; the per-adapter dequant factors are
// folded into the per-adapter factor array the kernels already apply.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

// 16 codes (one 16-byte load) -> 16 bf16 values (two 16-byte stores).
__device__ __forceinline__ void widen16(const uint8_t *src, uint16_t *dst)
{
    uint32_t o[8];
    e4m3x16_to_bf16(*reinterpret_cast<const uint4 *>(src), o);
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Grid: one group of `parts` CTAs per segment of the table (adapters used
// by the batch); CTA 0 also writes every adapter's factor for this call.
__global__ void __launch_bounds__(256) widen_kernel(const WidenParams p)
{
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < p.A; i += blockDim.x) {
            const float s = p.adapter_scale ? p.adapter_scale[i] : 1.f;
            const float da = p.dequant[2 * i], db = p.dequant[2 * i + 1];
            p.fac[i] = p.mode == kWidenShrink ? da : p.mode == kWidenExpand ? s * db : s * da * db;
        }
    }
    const int seg = blockIdx.x / p.parts, part = blockIdx.x - seg * p.parts;
    if (seg >= *p.num_segments) return;
    const int i = p.seg_id[seg];
    if (kDebugChecks && (i < 0 || i >= p.A)) return;   // LORA_DEBUG: a table the checker has flagged
    const int64_t na = static_cast<int64_t>(p.rank[i]) * p.K / 16;   // 16-code groups (padded rows are zero)
    const int64_t nb = static_cast<int64_t>(p.rank[i]) * p.N / 16;
    const uint8_t *a8 = p.a8 + p.a_off[i];
    const uint8_t *b8 = p.b8 + p.b_off[i];
    uint16_t *aw = p.aw + p.a_off[i];
    uint16_t *bw = p.bw + p.b_off[i];
    const int64_t step = static_cast<int64_t>(p.parts) * blockDim.x;
    for (int64_t v = static_cast<int64_t>(part) * blockDim.x + threadIdx.x; v < na + nb; v += step) {
        if (v < na) widen16(a8 + 16 * v, aw + 16 * v);
        else widen16(b8 + 16 * (v - na), bw + 16 * (v - na));
    }
}

cudaError_t launch_widen(const WidenParams &p, int max_segments, cudaStream_t stream)
{
    widen_kernel<<<max(1, max_segments) * p.parts, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace lora
