// Definition of launch_fwd and the macro that instantiates one family of
// forward-kernel variants (both head dimensions, all four mask kinds) in a
// translation unit of its own.
#pragma once

#include "../../include/attn.h"
#include "attn_kernel.cuh"
#include "attn_launch.h"

namespace attn {

template <int D, bool CAUSAL, bool ADDITIVE, bool BF16, bool ROPE, bool PACK>
int launch_fwd(bool& attr_set, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& to, const FwdParams& p, int grid, cudaStream_t stream) {
    auto kernel = attn_fwd_kernel<D, CAUSAL, ADDITIVE, BF16, ROPE, PACK>;
    constexpr int smem = TileCfg<D>::kSmemBytes;
    if (!attr_set) {
        // The in-kernel register split assumes exactly launch_regs(ROPE) per thread at launch.
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return ATTN_ERR_CUDA;
        if (fa.numRegs != launch_regs(ROPE)) return ATTN_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set = true;
    }
    kernel<<<grid, kernel_threads(ROPE), smem, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

#define ATTN_INSTANTIATE_ONE(D, CAUSAL, ADDITIVE, BF16, ROPE, PACK)                                              \
    template int attn::launch_fwd<D, CAUSAL, ADDITIVE, BF16, ROPE, PACK>(                                        \
        bool&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,                      \
        const attn::FwdParams&, int, cudaStream_t);

#define ATTN_INSTANTIATE_FWD(BF16, ROPE, PACK)                  \
    ATTN_INSTANTIATE_ONE(64, false, false, BF16, ROPE, PACK)    \
    ATTN_INSTANTIATE_ONE(64, true, false, BF16, ROPE, PACK)     \
    ATTN_INSTANTIATE_ONE(64, false, true, BF16, ROPE, PACK)     \
    ATTN_INSTANTIATE_ONE(64, true, true, BF16, ROPE, PACK)      \
    ATTN_INSTANTIATE_ONE(128, false, false, BF16, ROPE, PACK)   \
    ATTN_INSTANTIATE_ONE(128, true, false, BF16, ROPE, PACK)    \
    ATTN_INSTANTIATE_ONE(128, false, true, BF16, ROPE, PACK)    \
    ATTN_INSTANTIATE_ONE(128, true, true, BF16, ROPE, PACK)
