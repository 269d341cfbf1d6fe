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
// biased variance in FP32, the variance taken around the mean (two passes);
// the output is (x - mean) * (rstd * gamma) + beta. Each block first widens
// gamma and beta to FP32 in shared memory, one {gamma, gamma, beta, beta}
// vector per pair of columns, laid out [pair of the chunk][chunk] so that a
// warp's 16-byte reads of consecutive chunks are conflict-free.
template <int kMaxPerLane>
__global__ void __launch_bounds__(256) layernorm_kernel(const uint4* __restrict__ x, const uint4* __restrict__ gamma,
                                                        const uint4* __restrict__ beta, uint4* __restrict__ y, int M,
                                                        int chunks, float inv_h, float eps) {
    extern __shared__ float4 ln_gb[];                   // [4][chunks]
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        const uint4 g4 = __ldg(gamma + c), b4 = __ldg(beta + c);
        const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            ln_gb[j * chunks + c] = make_float4(__uint_as_float(gw[j] << 16), __uint_as_float(gw[j] & 0xffff0000u),
                                                __uint_as_float(bw[j] << 16), __uint_as_float(bw[j] & 0xffff0000u));
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < M; row += warps) {
        const uint4* xr = x + (size_t)row * chunks;
        uint4 v[kMaxPerLane];
        // Two bf16 values per 32-bit word, processed as an FP32 pair with the
        // packed (f32x2) instructions.
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < chunks) {
                v[i] = xr[c];
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    ptx::add2(s0, s1, s0, s1, __uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
            }
        }
        const float mean = warp_sum(s0 + s1) * inv_h;
        float q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            if (lane + 32 * i < chunks) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float d0, d1;
                    ptx::add2(d0, d1, __uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u), -mean, -mean);
                    ptx::fma2(q0, q1, d0, d1, d0, d1, q0, q1);
                }
            }
        }
        const float rstd = rsqrtf(warp_sum(q0 + q1) * inv_h + eps);
        uint4* yr = y + (size_t)row * chunks;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < chunks) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 gb = ln_gb[j * chunks + c];
                    float d0, d1, a0, a1, y0, y1;
                    ptx::add2(d0, d1, __uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u), -mean, -mean);
                    ptx::fma2(a0, a1, gb.x, gb.y, rstd, rstd, 0.f, 0.f);
                    ptx::fma2(y0, y1, d0, d1, a0, a1, gb.z, gb.w);
                    o[j] = ptx::pack_bf16x2(y0, y1);
                }
                yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// Rows of 1025-4096 values: one block of eight warps per SM (up to 255
// registers per thread) with each lane's part of the row unpacked to FP32
// registers (at most 128 values), so the bf16 pairs are widened once instead
// of once per pass; the variance pass centres the values in place and the
// output pass is two pair FMAs per pair, (x - mean) * (rstd * gamma) + beta,
// the same arithmetic as layernorm_kernel. Each warp loads its next row's
// chunks while it processes the current one.
template <int kPerLane>
__global__ void __launch_bounds__(256, 1) layernorm_rows_kernel(const uint4* __restrict__ x,
                                                               const uint4* __restrict__ gamma,
                                                               const uint4* __restrict__ beta, uint4* __restrict__ y,
                                                               int M, int chunks, float inv_h, float eps) {
    extern __shared__ float4 ln_gb[];                   // [4][chunks]
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    uint4 nxt[kPerLane];
    auto fetch = [&](int r) {
        const uint4* xr = x + (size_t)r * chunks;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i)
            if (lane + 32 * i < chunks) nxt[i] = xr[lane + 32 * i];
    };
    if (row < M) fetch(row);                            // in flight while gamma and beta are widened
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        const uint4 g4 = __ldg(gamma + c), b4 = __ldg(beta + c);
        const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            ln_gb[j * chunks + c] = make_float4(__uint_as_float(gw[j] << 16), __uint_as_float(gw[j] & 0xffff0000u),
                                                __uint_as_float(bw[j] << 16), __uint_as_float(bw[j] & 0xffff0000u));
    }
    __syncthreads();
    for (; row < M; row += warps) {
        float v[8 * kPerLane];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            if (lane + 32 * i < chunks) {
                const uint32_t w[4] = {nxt[i].x, nxt[i].y, nxt[i].z, nxt[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                    v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
                    ptx::add2(s0, s1, s0, s1, v[8 * i + 2 * j], v[8 * i + 2 * j + 1]);
                }
            }
        }
        if (row + warps < M) fetch(row + warps);
        const float mean = warp_sum(s0 + s1) * inv_h;
        float q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            if (lane + 32 * i < chunks) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float& d0 = v[8 * i + 2 * j];
                    float& d1 = v[8 * i + 2 * j + 1];
                    ptx::add2(d0, d1, d0, d1, -mean, -mean);
                    ptx::fma2(q0, q1, d0, d1, d0, d1, q0, q1);
                }
            }
        }
        const float rstd = rsqrtf(warp_sum(q0 + q1) * inv_h + eps);
        uint4* yr = y + (size_t)row * chunks;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < chunks) {
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 gb = ln_gb[j * chunks + c];
                    float a0, a1, y0, y1;
                    ptx::fma2(a0, a1, gb.x, gb.y, rstd, rstd, 0.f, 0.f);
                    ptx::fma2(y0, y1, v[8 * i + 2 * j], v[8 * i + 2 * j + 1], a0, a1, gb.z, gb.w);
                    o[j] = ptx::pack_bf16x2(y0, y1);
                }
                yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

}  // namespace

int launch_layernorm(bool (&attr_set)[3], const uint16_t* x, const uint16_t* gamma, const uint16_t* beta, uint16_t* y,
                     int M, int H, float eps, int num_sms, cudaStream_t stream) {
    const int chunks = H / 8;
    const size_t smem = (size_t)H * 8;                 // gamma and beta in FP32
    // Two blocks of eight warps per SM, each looping over rows.
    const unsigned grid = (unsigned)std::max(1LL, std::min(((long long)M + 7) / 8, 2LL * num_sms));
    const auto* x4 = reinterpret_cast<const uint4*>(x);
    const auto* g4 = reinterpret_cast<const uint4*>(gamma);
    const auto* b4 = reinterpret_cast<const uint4*>(beta);
    auto* y4 = reinterpret_cast<uint4*>(y);
    const float inv_h = 1.0f / (float)H;
    auto run = [&](auto kernel, bool& set) -> int {
        if (!set) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 8 * 8192) != cudaSuccess)
                return ATTN_ERR_CUDA;
            set = true;
        }
        kernel<<<grid, 256, smem, stream>>>(x4, g4, b4, y4, M, chunks, inv_h, eps);
        return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    };
    if (chunks <= 32 * 4) return run(layernorm_kernel<8>, attr_set[0]);
    if (chunks <= 32 * 16) {
        // rows of 1025-4096 values: one block of eight warps per SM, each warp looping over rows
        if (!attr_set[1]) {
            if (cudaFuncSetAttribute(layernorm_rows_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 8 * 8192) !=
                cudaSuccess)
                return ATTN_ERR_CUDA;
            attr_set[1] = true;
        }
        const unsigned g1 = (unsigned)std::max(1LL, std::min(((long long)M + 7) / 8, (long long)num_sms));
        layernorm_rows_kernel<16><<<g1, 256, smem, stream>>>(x4, g4, b4, y4, M, chunks, inv_h, eps);
        return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
    return run(layernorm_kernel<32>, attr_set[2]);
}

}  // namespace attn
