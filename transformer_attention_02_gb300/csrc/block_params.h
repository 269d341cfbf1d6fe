// Host-visible parameters of the attention block's kernels (projection GEMM
// and LayerNorm) and their launchers, defined in block_kernels.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {
namespace gemm {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kATileBytes = kBM * kBK * 2;                      // 16 KiB
constexpr int kBTileBytes = kBN * kBK * 2;                      // 32 KiB
constexpr int kStageBytes = kATileBytes + kBTileBytes;
// barriers: full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain
constexpr int bFull = 0, bEmpty = kStages, bAccFull = 2 * kStages, bAccEmpty = bAccFull + 2,
              bDrain = bAccEmpty + 2, kNumBars = bDrain + 1;
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kTmemSlotOff = kBarOff + 8 * kNumBars;
constexpr int kAbortOff = kTmemSlotOff + 4;
constexpr int kSmemBytes = kAbortOff + 4 + 1024;                // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemCols = 512;

struct GemmParams {
    int M, N, K;
    const uint16_t* bias;         // [N] or null
    const uint16_t* residual;     // [M, ldr] or null
    uint16_t* out;                // [M, ldo]
    int ldo, ldr;
    int tiles_m, tiles_n, n_tiles, k_steps;
    int group_rows;               // tile rows walked together (L2 reuse of the W column panels)
    unsigned long long timeout_ns;
    unsigned int* status;
};

// Launches gemm_bf16_kernel with `grid` persistent CTAs (attr_set caches, per
// device, that its shared-memory attribute has been set). ATTN_OK or ATTN_ERR_CUDA.
int launch(bool& attr_set, const CUtensorMap& a, const CUtensorMap& w, const GemmParams& p, int grid,
           cudaStream_t stream);

}  // namespace gemm

// LayerNorm of each of M rows of H bf16 values (H a multiple of 8, at most
// 8192): y = (x - mean) / sqrt(var + eps) * gamma + beta, FP32 statistics.
// attr_set caches, per context and kernel instance, that the kernel's
// shared-memory attribute has been set.
int launch_layernorm(bool (&attr_set)[3], const uint16_t* x, const uint16_t* gamma, const uint16_t* beta, uint16_t* y,
                     int M, int H, float eps, int num_sms, cudaStream_t stream);

}  // namespace attn
