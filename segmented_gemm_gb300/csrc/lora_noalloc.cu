// lora_linear_noalloc: the fused layer for callers that cannot allocate
// device memory (for instance an inference-engine hook that receives no
// workspace and is not allowed to call cudaMalloc while it runs).  The
// scratch that lora_linear keeps in the caller's workspace lives here in a
// statically allocated device array instead.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "lora.h"

namespace lora {

// The library's scratch for lora_linear_noalloc.  Every GPU that loads the
// library holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LORA_NOALLOC_SCRATCH_BYTES];

// Device address of the array, looked up once per device.  In host code the
// array's name is only a host-side stand-in, so kernels must be given this
// address, never &g_noalloc_scratch.
static void *noalloc_scratch_address(int *rc)
{
    static void *addr[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *rc = LORA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            *rc = LORA_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    *rc = LORA_OK;
    return addr[dev];
}

}  // namespace lora

using namespace lora;

// The tiled schedule's optional split-tile scratch (one 128 KB slot per
// output tile it may split) is larger than the whole array, so calls here
// with M > 128 always run that schedule without splitting a partial last
// wave along K.
static_assert(static_cast<size_t>(kStreamKMaxTiles) * kBM * kBN * 4 > LORA_NOALLOC_SCRATCH_BYTES,
              "the split-tile scratch would fit: clear its counters before each call");

extern "C" int lora_linear_noalloc(const lora_bf16_t *x, int64_t M, const lora_bf16_t *W, const lora_bf16_t *bias,
                                   const int32_t *lora_id_map, const lora_pool_t *pool, float scale, lora_bf16_t *y,
                                   lora_stream_t stream)
{
    // the pool and M are checked before any layout arithmetic depends on them
    int rc = check_pool(pool);
    if (rc) return rc;
    if (M < 0 || M > kMaxTokens) return LORA_ERR_SHAPE;
    if (M == 0) return LORA_OK;
    // the call is refused when the minimal layout (everything but the
    // optional split-tile scratch) does not fit the array
    const WsLayout L = make_ws_layout(M, pool->N, pool->num_adapters);
    if (L.total_min > LORA_NOALLOC_SCRATCH_BYTES) return LORA_ERR_CAPACITY;
    if (!x || !W || !y || !lora_id_map) return LORA_ERR_NULL;
    void *ws = noalloc_scratch_address(&rc);
    if (rc != LORA_OK) return rc;
    // The array keeps whatever the previous call (of any shape) left in it:
    // clear the parts that this call's layout needs to start at zero.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(ws);
    const size_t zero_regions[][2] = {{L.counters, L.n_counters * 4},
                                      {L.wcnt, static_cast<size_t>(L.max_win_str) * kWinCntStride * 4},
                                      {L.acc_str, L.acc_str_bytes},
                                      {L.acc_out, L.acc_out_bytes},
                                      {L.acc_shr, L.acc_shr_bytes}};
    for (const auto &r : zero_regions)
        if (r[1] > 0 && cudaMemsetAsync(base + r[0], 0, r[1], s) != cudaSuccess) return LORA_ERR_CUDA;
    return lora_linear(x, M, W, bias, lora_id_map, pool, scale, nullptr, y, ws, LORA_NOALLOC_SCRATCH_BYTES, stream);
}
