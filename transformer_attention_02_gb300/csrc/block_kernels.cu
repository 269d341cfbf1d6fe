// Kernels of the attention block other than the attention itself: the
// projection GEMM (gemm_kernel.cuh) and the LayerNorm ("ATB orchestration
// blog" section 2, the fused attention block: LayerNorm -> QKV projection ->
// FlashAttention -> output projection -> residual add).
#include "../../include/attn.h"
#include <algorithm>

#include "gemm_kernel.cuh"

namespace attn {

namespace gemm {

int launch(bool& attr_set, const CUtensorMap& a, const CUtensorMap& w, const GemmParams& p, int grid,
           cudaStream_t stream) {
    if (!attr_set) {
        if (cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set = true;
    }
    gemm_bf16_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, w, p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace gemm

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One warp per row; the row (at most 32 chunks of 8 values per lane) stays in
// registers between the two statistics passes and the output pass. Mean and
// biased variance in FP32, the variance taken around the mean (two passes).
template <int kMaxPerLane>
__global__ void __launch_bounds__(256) layernorm_kernel(const uint4* __restrict__ x, const uint4* __restrict__ gamma,
                                                        const uint4* __restrict__ beta, uint4* __restrict__ y, int M,
                                                        int chunks, float inv_h, float eps) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < M; row += warps) {
        const uint4* xr = x + (size_t)row * chunks;
        uint4 v[kMaxPerLane];
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < chunks) {
                v[i] = xr[c];
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) sum += __uint_as_float(w[j] << 16) + __uint_as_float(w[j] & 0xffff0000u);
            }
        }
        const float mean = warp_sum(sum) * inv_h;
        float sq = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            if (lane + 32 * i < chunks) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a = __uint_as_float(w[j] << 16) - mean, b = __uint_as_float(w[j] & 0xffff0000u) - mean;
                    sq += a * a + b * b;
                }
            }
        }
        const float rstd = rsqrtf(warp_sum(sq) * inv_h + eps);
        uint4* yr = y + (size_t)row * chunks;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < chunks) {
                const uint4 g4 = __ldg(gamma + c), b4 = __ldg(beta + c);
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, bw[4] = {b4.x, b4.y, b4.z, b4.w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a = (__uint_as_float(w[j] << 16) - mean) * rstd * __uint_as_float(gw[j] << 16) +
                                    __uint_as_float(bw[j] << 16);
                    const float b = (__uint_as_float(w[j] & 0xffff0000u) - mean) * rstd *
                                        __uint_as_float(gw[j] & 0xffff0000u) +
                                    __uint_as_float(bw[j] & 0xffff0000u);
                    o[j] = ptx::pack_bf16x2(a, b);
                }
                yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

}  // namespace

int launch_layernorm(const uint16_t* x, const uint16_t* gamma, const uint16_t* beta, uint16_t* y, int M, int H,
                     float eps, int num_sms, cudaStream_t stream) {
    const int chunks = H / 8;
    const long long warps_needed = M;
    const unsigned grid = (unsigned)std::max(1LL, std::min((warps_needed + 7) / 8, 16LL * num_sms));
    const auto* x4 = reinterpret_cast<const uint4*>(x);
    const auto* g4 = reinterpret_cast<const uint4*>(gamma);
    const auto* b4 = reinterpret_cast<const uint4*>(beta);
    auto* y4 = reinterpret_cast<uint4*>(y);
    const float inv_h = 1.0f / (float)H;
    if (chunks <= 32 * 8)
        layernorm_kernel<8><<<grid, 256, 0, stream>>>(x4, g4, b4, y4, M, chunks, inv_h, eps);
    else if (chunks <= 32 * 16)
        layernorm_kernel<16><<<grid, 256, 0, stream>>>(x4, g4, b4, y4, M, chunks, inv_h, eps);
    else
        layernorm_kernel<32><<<grid, 256, 0, stream>>>(x4, g4, b4, y4, M, chunks, inv_h, eps);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
