// Projection GEMM of the attention block on the 5th-generation tensor cores:
//   out[m, n] = sum_k A[m, k] W[n, k]  (+ bias[n])  (+ residual[m, n])
// A (M x K) and W (N x K) row-major bf16, FP32 accumulation in tensor memory,
// bf16 out ("ATB orchestration blog" section 2, the fused attention block's
// Linear steps; the bias and the residual add are fused into the epilogue).
//
// Persistent kernel, one CTA of 192 threads per SM, tiles of 128 x 256
// outputs walked in a grouped order (a group of tile rows at a time, column by
// column, so that a wave of CTAs shares its A rows and W columns in L2):
//   warp 0     TMA producer: 64-wide K slices of A (128 x 64) and W (256 x 64)
//              into a ring of kStages 48 KiB stages (128-byte swizzle);
//   warp 1     MMA issuer: four tcgen05.mma (M=128, N=256, K=16) per stage
//              into one of two 256-column TMEM accumulators, so that the
//              epilogue of one tile overlaps the products of the next;
//   warps 2-5  epilogue: each thread owns one output row, reads 32 accumulator
//              columns at a time (tcgen05.ld 32x32b), adds the bias and the
//              residual, rounds to bf16 and stores.
// Every wait is bounded (same status word and abort protocol as the
// attention kernel).
#pragma once

#include "attn_kernel.cuh"
#include "block_params.h"

namespace attn {
namespace gemm {

// Tile t of the grouped order -> (tile row, tile column): groups of
// group_rows tile rows, each walked column by column.
__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& tm, int& tn) {
    const int per_group = p.group_rows * p.tiles_n;
    const int group = t / per_group;
    const int first = group * p.group_rows;
    const int rows = min(p.group_rows, p.tiles_m - first);
    const int r = t - group * per_group;
    tm = first + r % rows;
    tn = r / rows;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem_ptr = smem_raw + pad;
    const uint32_t smem = raw + pad;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bars = smem + kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem_ptr + kAbortOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_ptr + kTmemSlotOff);

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < kNumBars; ++i) ptx::mbar_init(bar(i), (i == bAccEmpty || i == bAccEmpty + 1) ? 4u : 1u);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_shared();
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const SyncCtx sc{abort_flag, p.status, p.timeout_ns};
    const bool leader = lane == 0;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        uint32_t fill = 0;
        bool alive = true;
        for (int t = blockIdx.x; t < p.n_tiles && alive; t += gridDim.x) {
            int tm, tn;
            tile_coords(t, p, tm, tn);
            for (int ks = 0; ks < p.k_steps; ++ks, ++fill) {
                const uint32_t s = fill % kStages;
                if (fill >= (uint32_t)kStages && !warp_wait(bar(bEmpty + s), ((fill / kStages) - 1) & 1u, sc)) {
                    alive = false;
                    break;
                }
                if (leader) {
                    const uint32_t dst = smem + s * kStageBytes;
                    ptx::mbar_arrive_expect_tx(bar(bFull + s), kStageBytes);
                    ptx::tma_load_2d(dst, &tmA, bar(bFull + s), ks * kBK, tm * kBM);
                    ptx::tma_load_2d(dst + kATileBytes, &tmW, bar(bFull + s), ks * kBK, tn * kBN);
                }
                __syncwarp();
            }
        }
        for (uint32_t s = 0; s < (uint32_t)kStages; ++s)
            if (fill > s) drain_phase(bar(bFull + s), ((s + kStages * ((fill - 1 - s) / kStages)) / kStages) & 1u, sc);
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdesc = ptx::idesc_f16(kBM, kBN, true, false, false);
        uint32_t use = 0;
        int it = 0;
        bool issued = false, alive = true;
        for (int t = blockIdx.x; t < p.n_tiles && alive; t += gridDim.x, ++it) {
            const int acc = it & 1;
            if (it >= 2 && !warp_wait(bar(bAccEmpty + acc), ((it >> 1) - 1) & 1u, sc)) break;
            ptx::tc_fence_after_sync();
            const uint32_t d = tmem + (uint32_t)(acc * kBN);
            for (int ks = 0; ks < p.k_steps; ++ks, ++use) {
                const uint32_t s = use % kStages;
                if (!warp_wait(bar(bFull + s), (use / kStages) & 1u, sc)) {
                    alive = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                if (leader) {
                    const uint64_t ad = ptx::sdesc_kmajor_sw128(smem + s * kStageBytes);
                    const uint64_t bd = ptx::sdesc_kmajor_sw128(smem + s * kStageBytes + kATileBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        ptx::mma_ss(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), kIdesc,
                                    (ks > 0 || kk > 0) ? 1u : 0u);
                    ptx::tc_commit(bar(bEmpty + s));
                }
                issued = true;
                __syncwarp();
            }
            if (!alive) break;
            if (leader) ptx::tc_commit(bar(bAccFull + acc));
            __syncwarp();
        }
        if (issued) {
            if (leader) ptx::tc_commit(bar(bDrain));
            __syncwarp();
            drain_phase(bar(bDrain), 0, sc);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int quarter = warp & 3;                             // TMEM lanes 32*quarter ..
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        int it = 0;
        for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++it) {
            int tm, tn;
            tile_coords(t, p, tm, tn);
            const int acc = it & 1;
            if (!warp_wait(bar(bAccFull + acc), (it >> 1) & 1u, sc)) break;
            ptx::tc_fence_after_sync();
            const int row = tm * kBM + quarter * 32 + lane;
            const bool row_ok = row < p.M;
            const int n0 = tn * kBN;
            const uint32_t taddr = tmem + lane_base + (uint32_t)(acc * kBN);
            for (int c = 0; c < kBN; c += 32) {
                uint32_t v[32];
                ptx::tmem_ld32(taddr + (uint32_t)c, v);
                const int col = n0 + c;
                const bool col_ok = col < p.N;                     // N is a multiple of 32
                uint4 res[4] = {};
                if (p.residual && row_ok && col_ok) {
                    const uint4* rp = reinterpret_cast<const uint4*>(p.residual + (size_t)row * p.ldr + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) res[i] = rp[i];
                }
                ptx::tmem_ld_wait();
                ptx::reg_fence32(v);
                if (row_ok && col_ok) {
                    float bias[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) bias[i] = 0.f;
                    if (p.bias) {
                        const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4 w = __ldg(bp + i);
                            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                bias[8 * i + 2 * j] = __uint_as_float(ws[j] << 16);
                                bias[8 * i + 2 * j + 1] = __uint_as_float(ws[j] & 0xffff0000u);
                            }
                        }
                    }
                    uint32_t outw[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float a = __uint_as_float(v[2 * i]) + bias[2 * i];
                        float b = __uint_as_float(v[2 * i + 1]) + bias[2 * i + 1];
                        if (p.residual) {
                            const uint32_t rw = (&res[i / 4].x)[i % 4];
                            a += __uint_as_float(rw << 16);
                            b += __uint_as_float(rw & 0xffff0000u);
                        }
                        outw[i] = ptx::pack_bf16x2(a, b);
                    }
                    uint4* op = reinterpret_cast<uint4*>(p.out + (size_t)row * p.ldo + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        op[i] = make_uint4(outw[4 * i], outw[4 * i + 1], outw[4 * i + 2], outw[4 * i + 3]);
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (leader) ptx::mbar_arrive(bar(bAccEmpty + acc));
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace gemm
}  // namespace attn
