// Segment builder kernel ("vLLM-Ascend dynamic LoRA", §2.3): one CTA of 512
// threads runs the build of seg_build_body.cuh.  The decode-sized fused
// kernel runs the same body in one of its own CTAs instead.
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"
#include "seg_build_body.cuh"

namespace lora {

using SegBuild16 = SegBuild<16>;

__global__ void __launch_bounds__(SegBuild16::kSegThreads, 1) seg_build_kernel(SegParams p)
{
    // Let a fused kernel that follows start its prologue and weight stream
    // now; it waits for this grid before reading anything built here.
    pdl_launch_dependents();

    extern __shared__ int sm[];
    SegBuild16::run(p, sm);
    // Launched as the programmatic dependent of the decode-sized fused
    // kernel (which reads none of these tables, and whose inputs this grid
    // only reads), it runs beside that kernel and finishes only after it, so
    // stream order holds for what follows.  A no-op for an ordinary launch.
    if (threadIdx.x == 0) pdl_wait();
}

size_t seg_build_smem_bytes(int32_t A) { return SegBuild16::smem_bytes(A); }

cudaError_t launch_seg_build(const SegParams &p, bool pdl, cudaStream_t stream)
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
    // pdl: right after the decode-sized fused kernel, beside which it runs.
    // Before a fused kernel it is an ordinary launch: a programmatic one
    // there measured slower, its waiting block delaying the fused kernel's
    // clusters.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(SegBuild16::kSegThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, seg_build_kernel, p);
}

}  // namespace lora
