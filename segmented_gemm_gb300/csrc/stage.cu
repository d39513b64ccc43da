// Moving a step's inputs and outputs across the host link with the SMs.
//
// A GB300 board's host memory sits behind a coherent chip-to-chip link, and
// pinned host memory is mapped into the GPU's address space, so kernels can
// load from and store to it.  lora_copy_async copies a few buffers in one
// small kernel (no copy-engine transfer: a step's chain stays kernels only,
// and the kernel takes part in programmatic launch like the fused layers);
// lora_device_pointer gives the device-side address of a buffer, which the
// fused layer can take as y (its output rows are plain stores).
#include <cuda_runtime.h>

#include "internal.h"
#include "lora.h"
#include "ptx.cuh"

namespace lora {

struct CopyList {
    uint4 *dst[LORA_MAX_COPIES];
    const uint4 *src[LORA_MAX_COPIES];
    int64_t end[LORA_MAX_COPIES];   // running total of 16-byte units up to and including copy i
    int32_t n;
};

constexpr int kCopyThreads = 256;

// One 16-byte unit per thread and pass; every unit of a pass is in flight at
// once, which is what hides the link's latency.
__global__ void __launch_bounds__(kCopyThreads) stage_copy_kernel(CopyList c)
{
    pdl_launch_dependents();   // the launch behind this one may start its prologue
    pdl_wait();                // every kernel ahead has finished with these buffers
    const int64_t total = c.end[c.n - 1];
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kCopyThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x; i < total; i += stride) {
        int s = 0;
        while (i >= c.end[s]) ++s;
        const int64_t j = i - (s ? c.end[s - 1] : 0);
        c.dst[s][j] = c.src[s][j];
    }
}

// The address a kernel on the current device uses for ptr: ptr itself for
// this device's memory or managed memory, the mapped alias for pinned host
// memory; nullptr for anything else (pageable host memory, another device's
// memory, an unknown pointer).
static void *device_alias(const void *ptr)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    switch (a.type) {
    case cudaMemoryTypeDevice:
        return a.device == dev ? const_cast<void *>(ptr) : nullptr;
    case cudaMemoryTypeManaged:
        return const_cast<void *>(ptr);
    case cudaMemoryTypeHost:
        return a.devicePointer;
    default:
        return nullptr;
    }
}

}  // namespace lora

using namespace lora;

extern "C" int lora_device_pointer(const void *ptr, void **dev_ptr)
{
    if (!ptr || !dev_ptr) return LORA_ERR_NULL;
    void *d = device_alias(ptr);
    if (!d) return LORA_ERR_ACCESS;
    *dev_ptr = d;
    return LORA_OK;
}

extern "C" int lora_copy_async(const lora_copy_t *copies, int32_t n, lora_stream_t stream)
{
    if (n < 0 || n > LORA_MAX_COPIES) return LORA_ERR_SHAPE;
    if (n > 0 && !copies) return LORA_ERR_NULL;
    CopyList c{};
    int64_t units = 0;
    for (int32_t i = 0; i < n; ++i) {
        const lora_copy_t &k = copies[i];
        if (k.bytes < 0) return LORA_ERR_SHAPE;
        if (k.bytes == 0) continue;
        if (!k.dst || !k.src) return LORA_ERR_NULL;
        if ((reinterpret_cast<uintptr_t>(k.dst) | reinterpret_cast<uintptr_t>(k.src) |
             static_cast<uintptr_t>(k.bytes)) % 16)
            return LORA_ERR_ALIGN;
        void *d = device_alias(k.dst), *s = device_alias(k.src);
        if (!d || !s) return LORA_ERR_ACCESS;
        c.dst[c.n] = static_cast<uint4 *>(d);
        c.src[c.n] = static_cast<const uint4 *>(s);
        units += k.bytes / 16;
        c.end[c.n] = units;
        ++c.n;
    }
    if (c.n == 0) return LORA_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return LORA_ERR_CUDA;
    const int64_t want = (units + kCopyThreads - 1) / kCopyThreads;
    const int64_t cap = 8ll * (sms > 0 ? sms : 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap));
    cfg.blockDim = dim3(kCopyThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stage_copy_kernel, c) == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}
