// The grouped expert GEMM on two token tiles of one expert per work item
// (moe_pair.cu), as lora_moe_gemm launches it.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lora {

struct MoePairParams {
    const uint16_t *x;          // bf16 [M, K]: the tokens
    uint16_t *out;              // bf16 [M * topk, N]: one row per (token, slot) pair
    const int32_t *perm_pad;    // [max_mtiles * 128]: the pair at each row of the padded order, -1 in the gaps
    const int32_t *mt_expert;   // [max_mtiles]: the expert of each 128-row tile of the padded order
    const int32_t *hdr;         // the routing's header (its tile count, the debug build's check verdict)
    int32_t *status;            // LORA_DEV_* bits
    int64_t out_rows;           // M * topk
    int32_t K, N, topk, kblocks, num_ntiles, max_mtiles;
    long long wait_cycles;      // the bounded waits' long budget
};

// Token tiles the kernel's item list holds; lora_moe_gemm uses the tiled
// kernel's expert mode for larger routings.
constexpr int kMoePairMaxTiles = 4096;

cudaError_t launch_moe_pair(const CUtensorMap &w, const MoePairParams &p, cudaStream_t stream);

}  // namespace lora
