// Fused attention forward for sm_103a: Q K^T -> scale -> mask -> online
// softmax -> P V in one persistent, warp-specialised kernel.
//
// What is computed ("CANN-ATB图优化-…融合算子" Pattern 2; "ATB engineering
// guide" §4.1 pattern 2 and §5.1; "ops-transformer：…实战" §2.2, §2.4, §3.2):
//   o[b,i,h,:] = sum_j softmax_j(s_ij) v[b,j,h/G,:],
//   s_ij = scale <q[b,i,h,:], k[b,j,h/G,:]> + mask[b,i,j]   (G = Hq / Hkv)
//   lse[b,h,i] = log sum_j exp(s_ij)
// with the softmax computed block by block: each row keeps a running maximum
// and a running sum in FP32 registers, and the score matrix lives only in
// tensor memory (TMEM), never in device memory.
//
// Work decomposition ("ops-transformer：…实战" §3.2 and §5.2: B and H are
// independent, the sequence is split into blocks, all cores kept busy):
// a work tile is (b, h, 256 query rows). A persistent grid of one CTA per SM
// walks the tiles; with a causal mask the longest tiles come first and the
// query heads that share a K/V head are adjacent so their K/V stay in L2.
//
// Roles inside a CTA (320 threads):
//   warps 0-3  softmax warpgroup 0: query rows [m0, m0+128)      (TMEM lanes 0-127)
//   warps 4-7  softmax warpgroup 1: query rows [m0+128, m0+256)
//   warp  8    MMA issuer (one thread) + TMEM allocation
//   warp  9    TMA producer (one thread) + barrier initialisation
// Pipelining ("ops-transformer：…实战" §2.3): while one warpgroup exponentiates
// its scores, the tensor cores work on the other warpgroup's tile, and the TMA
// warp streams the next K/V tiles into a ring of shared-memory slots.
//
// TMEM (512 columns, FP32): S0 [0,128), S1 [128,256), O0 [256,256+D),
// O1 [256+D,256+2D). P_t (bf16, two per column) overwrites the first 64
// columns of S_t once the softmax warpgroup holds S_t in registers; the second
// product reads P straight from TMEM.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace attn {

struct FwdParams {
    void* o;                  // (B, Sq, Hq, D) 16-bit
    float* lse;               // (B, Hq, Sq)
    const float* mask;        // (B, Sq, Sk) FP32 or null
    int B, Hq, Hkv, Sq, Sk;
    int group;                // Hq / Hkv
    int n_mblk;               // ceil(Sq / 256)
    int n_tiles;              // B * Hq * n_mblk
    float scale_log2;         // scale * log2(e)
    int mask_vec4;            // mask rows may be read with 16-byte loads
    int debug_stall;          // wait on a barrier nothing signals (timeout test)
    unsigned long long timeout_ns;
    unsigned int* status;     // device status word, bit 0 = a wait timed out
};

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kBlockM = 128;        // query rows per softmax warpgroup
constexpr int kBlockN = 128;        // keys per K/V tile
constexpr int kRowsPerTile = 2 * kBlockM;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O only when the max grows by > 2^8
constexpr unsigned long long kDrainLimitNs = 1000000000ull;
constexpr unsigned int kStatusTimeout = 1u;

template <int D>
struct TileCfg {
    static_assert(D == 64 || D == 128, "head dimension must be 64 or 128");
    static constexpr int kBoxCols = 64;                       // one 128-byte swizzle span
    static constexpr int kBoxes = D / kBoxCols;
    static constexpr int kBoxBytes = 128 * kBoxCols * 2;      // 128 rows x 128 bytes
    static constexpr int kTileBytes = kBoxes * kBoxBytes;     // 128 rows x D
    static constexpr int kSlots = (D == 128) ? 4 : 8;         // K/V ring (K and V alternate)
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = 2 * kTileBytes;
    static constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
    // barrier indices
    static constexpr int bQFull = 0;        // [2]
    static constexpr int bQEmpty = 2;
    static constexpr int bSFull = 3;        // [2]
    static constexpr int bPFull = 5;        // [2]
    static constexpr int bPVDone = 7;       // [2]
    static constexpr int bOFull = 9;        // [2]
    static constexpr int bDrain = 11;
    static constexpr int bStall = 12;
    static constexpr int bKVFull = 13;      // [kSlots]
    static constexpr int bKVEmpty = 13 + kSlots;
    static constexpr int kNumBars = 13 + 2 * kSlots;
    static constexpr int kTmemSlotOff = kBarOff + 8 * kNumBars;
    static constexpr int kAbortOff = kTmemSlotOff + 4;
    static constexpr int kSmemUsed = kAbortOff + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;       // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr int s_col(int t) { return t * 128; }
    static constexpr int kOCol0 = 256;
    static_assert(kOCol0 + 2 * D <= 512, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct TileInfo {
    int b, h, hk, m0, n_blocks;
};

template <bool CAUSAL>
__device__ __forceinline__ TileInfo tile_info(int tile, const FwdParams& p) {
    const int bh_count = p.B * p.Hq;
    const int mb_rank = tile / bh_count;
    const int bh = tile - mb_rank * bh_count;
    const int mb = CAUSAL ? (p.n_mblk - 1 - mb_rank) : mb_rank;
    TileInfo t;
    t.b = bh / p.Hq;
    t.h = bh - t.b * p.Hq;
    t.hk = t.h / p.group;
    t.m0 = mb * kRowsPerTile;
    int kv_end = p.Sk;
    if (CAUSAL) {
        const int last_row = min(t.m0 + kRowsPerTile - 1, p.Sq - 1);
        kv_end = min(p.Sk, max(0, last_row + (p.Sk - p.Sq) + 1));
    }
    t.n_blocks = (kv_end + kBlockN - 1) / kBlockN;
    return t;
}

struct SyncCtx {
    volatile uint32_t* abort_flag;
    unsigned int* status;
    unsigned long long timeout_ns;
};

// Bounded wait on an mbarrier phase. Returns false (and raises the CTA's abort
// flag and the device status bit) when the limit runs out, or false at once
// when another thread of the CTA has already aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const SyncCtx& sc) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*sc.abort_flag) return false;
        if (ptx::global_timer_ns() - t0 > sc.timeout_ns) {
            *sc.abort_flag = 1u;
            atomicOr(sc.status, kStatusTimeout);
            return false;
        }
    }
}

// Wait used only while shutting down: ignores the abort flag, has its own limit.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, const SyncCtx& sc) {
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::global_timer_ns() - t0 > kDrainLimitNs) {
            atomicOr(sc.status, kStatusTimeout);
            return;
        }
    }
}

// ------------------------------------------------------------ TMA producer
template <int D, bool CAUSAL>
__device__ void role_tma(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                         const FwdParams& p, uint32_t smem, const SyncCtx& sc) {
    using C = TileCfg<D>;
    const uint32_t bars = smem + C::kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t kv_fill = 0, q_loads = 0;
    bool alive = true;
    for (int tile = blockIdx.x; tile < p.n_tiles && alive; tile += gridDim.x) {
        const TileInfo ti = tile_info<CAUSAL>(tile, p);
        if (ti.n_blocks == 0) continue;
        if (q_loads > 0 && !wait_phase(bar(C::bQEmpty), (q_loads - 1) & 1u, sc)) { alive = false; break; }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_arrive_expect_tx(bar(C::bQFull + t), C::kTileBytes);
            for (int c = 0; c < C::kBoxes; ++c)
                ptx::tma_load_4d(smem + C::kQOff + t * C::kTileBytes + c * C::kBoxBytes, tmQ,
                                 bar(C::bQFull + t), c * C::kBoxCols, ti.h, ti.m0 + t * kBlockM, ti.b);
        }
        ++q_loads;
        for (int j = 0; j < ti.n_blocks && alive; ++j) {
            for (int kv = 0; kv < 2; ++kv) {
                const uint32_t slot = kv_fill % C::kSlots;
                if (kv_fill >= (uint32_t)C::kSlots &&
                    !wait_phase(bar(C::bKVEmpty + slot), ((kv_fill / C::kSlots) - 1) & 1u, sc)) {
                    alive = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(bar(C::bKVFull + slot), C::kTileBytes);
                const CUtensorMap* map = kv ? tmV : tmK;
                for (int c = 0; c < C::kBoxes; ++c)
                    ptx::tma_load_4d(smem + C::kKVOff + slot * C::kTileBytes + c * C::kBoxBytes, map,
                                     bar(C::bKVFull + slot), c * C::kBoxCols, ti.hk, j * kBlockN, ti.b);
                ++kv_fill;
            }
        }
    }
    // Shut down: wait until every copy this thread started has landed.
    for (uint32_t s = 0; s < (uint32_t)C::kSlots; ++s) {
        if (kv_fill > s) {
            const uint32_t last = s + C::kSlots * ((kv_fill - 1 - s) / C::kSlots);
            drain_phase(bar(C::bKVFull + s), (last / C::kSlots) & 1u, sc);
        }
    }
    if (q_loads > 0) {
        drain_phase(bar(C::bQFull + 0), (q_loads - 1) & 1u, sc);
        drain_phase(bar(C::bQFull + 1), (q_loads - 1) & 1u, sc);
    }
}

// -------------------------------------------------------------- MMA issuer
template <int D, bool CAUSAL, bool BF16>
__device__ void role_mma(const FwdParams& p, uint32_t smem, uint32_t tmem, const SyncCtx& sc) {
    using C = TileCfg<D>;
    const uint32_t bars = smem + C::kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    constexpr uint32_t kIdescQK = ptx::idesc_f16(128, kBlockN, BF16, false, false);
    constexpr uint32_t kIdescPV = ptx::idesc_f16(128, D, BF16, false, true);
    uint32_t kv_use = 0, q_uses = 0;
    uint32_t p_cnt[2] = {0, 0}, pv_cnt[2] = {0, 0};
    bool issued = false;
    bool alive = true;
    if (p.debug_stall) alive = wait_phase(bar(C::bStall), 0, sc);   // nothing ever arrives
    for (int tile = blockIdx.x; tile < p.n_tiles && alive; tile += gridDim.x) {
        const TileInfo ti = tile_info<CAUSAL>(tile, p);
        if (ti.n_blocks == 0) continue;
        if (!wait_phase(bar(C::bQFull + 0), q_uses & 1u, sc) ||
            !wait_phase(bar(C::bQFull + 1), q_uses & 1u, sc)) { alive = false; break; }
        ++q_uses;
        ptx::tc_fence_after_sync();
        for (int j = 0; j < ti.n_blocks; ++j) {
            // ---- S_t = Q_t K_j^T
            const uint32_t ks = kv_use % C::kSlots;
            if (!wait_phase(bar(C::bKVFull + ks), (kv_use / C::kSlots) & 1u, sc)) { alive = false; break; }
            ++kv_use;
            ptx::tc_fence_after_sync();
            const uint32_t k_base = smem + C::kKVOff + ks * C::kTileBytes;
            for (int t = 0; t < 2 && alive; ++t) {
                // S_t still holds P_t of the previous block until that P.V is done.
                if (pv_cnt[t] > 0) {
                    if (!wait_phase(bar(C::bPVDone + t), (pv_cnt[t] - 1) & 1u, sc)) { alive = false; break; }
                    ptx::tc_fence_after_sync();
                }
                const uint32_t q_base = smem + C::kQOff + t * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
                    ptx::mma_ss(tmem + C::s_col(t), ptx::sdesc_kmajor_sw128(q_base + off),
                                ptx::sdesc_kmajor_sw128(k_base + off), kIdescQK, kk > 0 ? 1u : 0u);
                }
                issued = true;
                ptx::tc_commit(bar(C::bSFull + t));
            }
            if (!alive) break;
            ptx::tc_commit(bar(C::bKVEmpty + ks));
            if (j == ti.n_blocks - 1) ptx::tc_commit(bar(C::bQEmpty));
            // ---- O_t += P_t V_j
            const uint32_t vs = kv_use % C::kSlots;
            if (!wait_phase(bar(C::bKVFull + vs), (kv_use / C::kSlots) & 1u, sc)) { alive = false; break; }
            ++kv_use;
            const uint32_t v_base = smem + C::kKVOff + vs * C::kTileBytes;
            for (int t = 0; t < 2 && alive; ++t) {
                if (!wait_phase(bar(C::bPFull + t), p_cnt[t] & 1u, sc)) { alive = false; break; }
                ++p_cnt[t];
                ptx::tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    ptx::mma_ts(tmem + C::kOCol0 + t * D, tmem + C::s_col(t) + kk * 8,
                                ptx::sdesc_mnmajor_sw128(v_base + kk * 16 * 128, C::kBoxBytes), kIdescPV,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::tc_commit(bar(C::bPVDone + t));
                ++pv_cnt[t];
                if (j == ti.n_blocks - 1) ptx::tc_commit(bar(C::bOFull + t));
            }
            if (!alive) break;
            ptx::tc_commit(bar(C::bKVEmpty + vs));
        }
    }
    // Shut down: every MMA this thread issued must finish before TMEM is freed.
    if (issued) {
        ptx::tc_commit(bar(C::bDrain));
        drain_phase(bar(C::bDrain), 0, sc);
    }
}

// ------------------------------------------------ softmax / epilogue warpgroup
template <int D, bool CAUSAL, bool ADDITIVE, bool BF16>
__device__ void role_softmax(const FwdParams& p, uint32_t smem, uint32_t tmem, int wg, const SyncCtx& sc) {
    using C = TileCfg<D>;
    const uint32_t bars = smem + C::kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    const int warp = threadIdx.x >> 5;
    const int r = threadIdx.x & 127;                          // row inside the 128-row tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::s_col(wg);
    const uint32_t tO = tmem + lane_base + C::kOCol0 + wg * D;
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr float kLog2e = 1.4426950408889634f;
    uint32_t s_phase = 0, o_phase = 0;

    for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x) {
        const TileInfo ti = tile_info<CAUSAL>(tile, p);
        const int row = ti.m0 + wg * kBlockM + r;
        const bool row_ok = row < p.Sq;
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + (((size_t)ti.b * p.Sq + row) * p.Hq + ti.h) * D;
        float* lse_out = p.lse + ((size_t)ti.b * p.Hq + ti.h) * p.Sq + row;
        if (ti.n_blocks == 0) {                               // no visible key anywhere in the tile
            if (row_ok) {
                uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
                *lse_out = -INFINITY;
            }
            continue;
        }
        // keys [0, kv_lim) are visible to this row
        int kv_lim = p.Sk;
        if (CAUSAL) kv_lim = min(p.Sk, max(0, row + (p.Sk - p.Sq) + 1));
        const float* mrow = nullptr;
        if (ADDITIVE && row_ok) mrow = p.mask + ((size_t)ti.b * p.Sq + row) * p.Sk;

        float m_used = -INFINITY;     // max used for the exponentials (log2 units)
        float l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < ti.n_blocks; ++j) {
            ok = wait_phase(bar(C::bSFull + wg), s_phase, sc);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            s_phase ^= 1u;
            ptx::tc_fence_after_sync();
            uint32_t sr[kBlockN];
#pragma unroll
            for (int c = 0; c < kBlockN / 32; ++c) ptx::tmem_ld32(tS + 32 * c, sr + 32 * c);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < kBlockN / 32; ++c) ptx::reg_fence32(sr + 32 * c);

            const int key0 = j * kBlockN;
            const int vis = kv_lim - key0;                    // columns >= vis are hidden
            // x = s * scale * log2(e) (+ mask * log2(e)): logits in log2 units
            float x[kBlockN];
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) x[c] = __uint_as_float(sr[c]) * p.scale_log2;
            if (ADDITIVE && mrow != nullptr) {
                if (p.mask_vec4 && key0 + kBlockN <= p.Sk) {
                    const float4* m4 = reinterpret_cast<const float4*>(mrow + key0);
#pragma unroll
                    for (int c = 0; c < kBlockN / 4; ++c) {
                        const float4 mv = __ldg(m4 + c);
                        x[4 * c + 0] = fmaf(mv.x, kLog2e, x[4 * c + 0]);
                        x[4 * c + 1] = fmaf(mv.y, kLog2e, x[4 * c + 1]);
                        x[4 * c + 2] = fmaf(mv.z, kLog2e, x[4 * c + 2]);
                        x[4 * c + 3] = fmaf(mv.w, kLog2e, x[4 * c + 3]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        if (key0 + c < p.Sk) x[c] = fmaf(__ldg(mrow + key0 + c), kLog2e, x[c]);
                }
            }
            if (vis < kBlockN) {
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (c >= vis) x[c] = -INFINITY;
            }
            float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
            for (int c = 4; c < kBlockN; c += 4) {
                mx0 = fmaxf(mx0, x[c + 0]);
                mx1 = fmaxf(mx1, x[c + 1]);
                mx2 = fmaxf(mx2, x[c + 2]);
                mx3 = fmaxf(mx3, x[c + 3]);
            }
            const float m_new = fmaxf(m_used, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)));
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_used = m_new;
            } else {
                const bool need = m_new > m_used + kRescaleThreshold;
                rescale = __any_sync(0xffffffffu, need);
                if (need) {
                    alpha = ptx::ex2(m_used - m_new);
                    l_sum *= alpha;
                    m_used = m_new;
                }
            }
            const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
            uint32_t pk[kBlockN / 2];
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int c = 0; c < kBlockN / 2; ++c) {
                const float p0 = ptx::ex2(x[2 * c] - m_ref);
                const float p1 = ptx::ex2(x[2 * c + 1] - m_ref);
                ls0 += p0;
                ls1 += p1;
                pk[c] = BF16 ? ptx::pack_bf16x2(p0, p1) : ptx::pack_f16x2(p0, p1);
            }
            l_sum += ls0 + ls1;
            ptx::tmem_st32(tS + 0, pk);
            ptx::tmem_st32(tS + 32, pk + 32);
            if (rescale) {
                // O_t holds the previous blocks' sum and no P.V is running on it:
                // this S_t was computed only after that P.V had completed.
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    ptx::tmem_ld32(tO + 32 * c, ov);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence32(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    ptx::tmem_st32(tO + 32 * c, ov);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar(C::bPFull + wg));
        }
        if (!ok) return;
        // ---- epilogue: O / l -> 16-bit, LSE -> FP32
        ok = wait_phase(bar(C::bOFull + wg), o_phase, sc);
        if (!__all_sync(0xffffffffu, ok)) return;
        o_phase ^= 1u;
        ptx::tc_fence_after_sync();
        const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            ptx::tmem_ld32(tO + 32 * c, ov);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(ov);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = __uint_as_float(ov[2 * i]) * inv_l;
                const float b = __uint_as_float(ov[2 * i + 1]) * inv_l;
                w[i] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
            }
            if (row_ok) {
                uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
                dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
            }
        }
        if (row_ok) *lse_out = l_sum > 0.f ? (m_used + log2f(l_sum)) * kLn2 : -INFINITY;
    }
}

// ------------------------------------------------------------------ kernel
template <int D, bool CAUSAL, bool ADDITIVE, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using C = TileCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    // Swizzled TMA tiles and the MMA descriptors both assume 1024-byte alignment.
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem_ptr = smem_raw + pad;
    const uint32_t smem = raw + pad;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem_ptr + C::kAbortOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_ptr + C::kTmemSlotOff);

    if (warp == kTmaWarp && lane == 0) {
        const uint32_t bars = smem + C::kBarOff;
        for (int i = 0; i < C::kNumBars; ++i) {
            const bool many = (i == C::bPFull || i == C::bPFull + 1);
            ptx::mbar_init(bars + 8u * i, many ? kBlockM : 1u);
        }
        *abort_flag = 0u;
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_shared();
        ptx::prefetch_tensormap(&tmQ);
        ptx::prefetch_tensormap(&tmK);
        ptx::prefetch_tensormap(&tmV);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const SyncCtx sc{abort_flag, p.status, p.timeout_ns};

    if (warp < 8) {
        role_softmax<D, CAUSAL, ADDITIVE, BF16>(p, smem, tmem, warp >> 2, sc);
    } else if (warp == kMmaWarp) {
        if (lane == 0) role_mma<D, CAUSAL, BF16>(p, smem, tmem, sc);
        __syncwarp();
    } else if (warp == kTmaWarp) {
        if (lane == 0) role_tma<D, CAUSAL>(&tmQ, &tmK, &tmV, p, smem, sc);
        __syncwarp();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace attn
