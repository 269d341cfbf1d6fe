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
// a work tile is (b, h, 256 query rows). The grid has one CTA per tile; at
// most one fits on an SM, and a running CTA takes over the tiles of CTAs that
// have not started (cluster launch control), so the grid behaves as a
// persistent one with a dynamic schedule. With a causal mask the longest tiles
// come first and the query heads that share a K/V head are grouped so that
// their K/V stay in L2 (tile_info).
//
// Roles inside a CTA (384 threads; 512 in the rotary variant):
//   warps 0-3  softmax warpgroup 0: query rows [m0, m0+128)      (TMEM lanes 0-127)
//   warps 4-7  softmax warpgroup 1: query rows [m0+128, m0+256)
//   warp  8    MMA issuer (one thread) + TMEM allocation
//   warp  9    TMA producer of K/V (one thread) + barrier initialisation
//   warp 10    producer of the shared-memory tile ring (the CTA's work tiles)
//              and TMA producer of Q, a tile ahead for the lower sub-tile; in
//              the D=128 masked variants it also stores the output staged in
//              the Q buffers
//   warp 11    idle (it completes the third warpgroup for the register split)
//   warps 12-15 rotary variant only: rotate each Q sub-tile as it lands, 32
//              rows per warp
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
    int n_splits;             // key ranges per (b, h, query block); 1 = keys not split
    int split_blocks;         // 128-key blocks per key range
    int n_tiles;              // B * Hq * n_mblk * n_splits
    float* o_part;            // split keys: FP32 O of each key range (n_splits, B, Hq, Sq, D), else null
    float* lse_part;          // split keys: FP32 LSE of each key range (n_splits, B, Hq, Sq)
    float scale_log2;         // scale * log2(e)
    int mask_vec4;            // mask rows may be read with 32-byte (2) or 16-byte (1) loads, else 0
    int flags;                // kFlagOVec8 | kFlagDebugStall
    int head_group;           // tile order: (b, head) slices per group (see tile_info)
    unsigned long long timeout_ns;
    unsigned int* status;     // device status word, bit 0 = a wait timed out
    const float* rope;        // rotary table (max_pos, D/2, {cos, sin}) FP32 (rotating variant only)
    int q_pos0;               // position of query row 0 (rotating variant only)
    // Kept last: inserting it earlier shifted the 64-bit fields after it and
    // measurably changed the code generated for the unpacked kernels.
    int pack_shift;           // > 0: the 2^pack_shift query heads of a K/V head share each tile's rows
};
// Kept at 128 bytes, with the 64-bit fields where they are: appending two int
// fields (136 bytes) made the kernel 5% slower on the Llama-2-7B-shaped
// prefill, with the same code otherwise.
static_assert(sizeof(FwdParams) <= 128, "FwdParams size");
constexpr int kFlagOVec8 = 1;         // O rows may be written with 32-byte stores
constexpr int kFlagDebugStall = 2;    // the MMA issuer waits on a barrier nothing signals (timeout test)

constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kQWarp = 10;
constexpr int kRotateWarp0 = 12;            // rotary variant: warps 12-15 rotate the Q sub-tiles
// Threads and register split. Three warpgroups (four in the rotary variant),
// launched at 168 registers per thread (384 x 168 = 64512), then the softmax
// warpgroups grow to 192 and the MMA/TMA/Q warpgroup shrinks to 120:
// 128 x (192 + 192 + 120) = 64512. Rotary variant: launched at 128
// (512 x 128 = 65536), softmax 184, MMA/TMA/Q 96, rotation 48:
// 128 x (184 + 184 + 96 + 48) = 65536. The host refuses to launch unless the
// compiled kernel uses exactly launch_regs(ROPE), so the split always fits.
__host__ __device__ constexpr int kernel_threads(bool rope) { return rope ? 512 : 384; }
__host__ __device__ constexpr int launch_regs(bool rope) { return rope ? 128 : 168; }
__host__ __device__ constexpr uint32_t softmax_regs(bool rope) { return rope ? 184u : 192u; }
__host__ __device__ constexpr uint32_t control_regs(bool rope) { return rope ? 96u : 120u; }
constexpr uint32_t kRotateRegs = 48;
static_assert(128 * (2 * softmax_regs(false) + control_regs(false)) <= kernel_threads(false) * launch_regs(false),
              "register split");
static_assert(128 * (2 * softmax_regs(true) + control_regs(true) + kRotateRegs) <=
                  kernel_threads(true) * launch_regs(true),
              "register split (rotary variant)");
constexpr int kBlockM = 128;        // query rows per softmax warpgroup
constexpr int kBlockN = 128;        // keys per K/V tile
constexpr int kRowsPerTile = 2 * kBlockM;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O only when the max grows by > 2^8
constexpr int kTileSlots = 8;               // entries of the shared-memory tile ring
// Arrivals that free a tile-ring entry: the K/V producer, the MMA issuer, the
// eight softmax warps and, in the rotary variant, the four rotating warps.
__host__ __device__ constexpr uint32_t tile_consumers(bool rope) { return 1 + 1 + 8 + (rope ? 4u : 0u); }
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
    // Q sub-tile buffers, taken in turn by the sub-tiles (see q_slot).
    static constexpr int kQBufs = 3;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = kQBufs * kTileBytes;
    static constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
    // barrier indices
    static constexpr int bQFull = 0;                  // [kQBufs]
    static constexpr int bQEmpty = kQBufs;            // [kQBufs]
    static constexpr int bSFull = 2 * kQBufs;         // [2]
    static constexpr int bPFull = bSFull + 2;         // [2]
    static constexpr int bOFull = bPFull + 2;         // [2]
    static constexpr int bDrain = bOFull + 2;
    static constexpr int bStall = bDrain + 1;
    static constexpr int bKVFull = bStall + 1;        // [kSlots]
    static constexpr int bKVEmpty = bKVFull + kSlots;
    static constexpr int bQRdy = bKVEmpty + kSlots;   // [kQBufs] rotary variant: Q rotated (four arrivals)
    static constexpr int bTileFull = bQRdy + kQBufs;  // [kTileSlots] tile ring entry published
    static constexpr int bTileEmpty = bTileFull + kTileSlots;   // [kTileSlots] entry freed by every consumer
    static constexpr int bClc = bTileEmpty + kTileSlots;      // cluster-launch-control response landed
    static constexpr int bOStaged = bClc + 1;         // [2][2] sub-tile's O staged (one arrival per warp)
    static constexpr int kNumBars = bOStaged + 4;
    // tile ring: kTileSlots entries of 32 bytes, read and written as 16-byte vectors
    static constexpr int kTileOff = (kBarOff + 8 * kNumBars + 31) / 32 * 32;
    static constexpr int kClcOff = kTileOff + kTileSlots * 32;   // 16-byte cluster-launch-control response
    static constexpr int kTmemSlotOff = kClcOff + 16;
    static constexpr int kAbortOff = kTmemSlotOff + 4;
    static constexpr int kSmemUsed = kAbortOff + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;       // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr int s_col(int t) { return t * 128; }
    static constexpr int kOCol0 = 256;
    static_assert(kOCol0 + 2 * D <= 512, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kKVOff % 1024 == 0 && kBarOff % 1024 == 0, "swizzled tiles need 1024-byte alignment");
    static_assert(kTileOff % 32 == 0, "tile ring entries are accessed as 16-byte vectors");
    static_assert(kClcOff % 16 == 0, "the launch-control response is a 16-byte value");
    static_assert(kTmemSlotOff % 4 == 0 && kAbortOff % 4 == 0, "4-byte words");
};

struct TileInfo {
    int b, h, hk, m0;  // h: the (first) query head; m0: the first query row
    int split;      // key range index
    int kb0;        // first 128-key block of the key range
    int nb[2];      // KV blocks needed by query sub-tile t (rows m0+128t .. m0+128t+127)
    int n;          // max(nb[0], nb[1]): KV blocks streamed for the tile
};

// Work tiles in launch order (the dynamic schedule hands them out in this
// order, so it is also the order in which they start). A slice is one (b, head)
// pair (b, K/V head with head packing); a slice has n_mblk query blocks and
// n_splits key ranges. The slices are cut into groups of head_group
// consecutive slices, about a fixed budget of K/V bytes each, and a group's
// tiles run together so that its K/V stays in L2 while all of its query blocks
// read it; within a group the query blocks run from the last (longest, with a
// causal mask) to the first. With a causal mask the three shortest query-block
// levels of every slice are left out of the groups and run at the very end,
// longest first over all slices, so that the last tiles to start are short.
// The query heads sharing a K/V head are adjacent slices, so they run side by side.
// With head packing (pack_shift > 0, decode and short prefills) a tile belongs
// to one K/V head: each 128-row sub-tile holds 128 >> pack_shift query rows of
// all 2^pack_shift query heads of the group (row r of the sub-tile is query
// row r >> pack_shift of head h + (r & (group - 1))), so the group's heads
// share every K/V block instead of streaming it once each.
template <bool CAUSAL, bool PACK>
__device__ __forceinline__ TileInfo tile_info(int tile, const FwdParams& p) {
    const int ps = PACK ? p.pack_shift : 0;
    const int heads = PACK ? p.Hkv : p.Hq;
    const int sub_rows = kBlockM >> ps;
    const int slices = p.B * heads;
    const int tail_levels = CAUSAL ? min(3, p.n_mblk) : 0;     // the three shortest levels run last
    const int head_levels = p.n_mblk - tail_levels;            // levels run inside the groups
    const int grouped = slices * head_levels * p.n_splits;      // tiles of the group phase
    int mb, split, bh;
    if (tile < grouped) {
        const int per_slice = head_levels * p.n_splits;
        const int g0 = tile / (p.head_group * per_slice) * p.head_group;   // first slice of the group
        const int gs = min(p.head_group, slices - g0);                      // slices in the group
        const int local = tile - g0 * per_slice;
        const int per_level = gs * p.n_splits;
        const int level = local / per_level;
        const int rem = local - level * per_level;
        split = rem / gs;
        bh = g0 + (rem - split * gs);
        mb = CAUSAL ? (p.n_mblk - 1 - level) : level;
    } else {
        const int local = tile - grouped;
        const int per_level = slices * p.n_splits;
        const int level = local / per_level;
        const int rem = local - level * per_level;
        split = rem / slices;
        bh = rem - split * slices;
        mb = CAUSAL ? (tail_levels - 1 - level) : (head_levels + level);
    }
    TileInfo t;
    t.b = bh / heads;
    const int hh = bh - t.b * heads;
    t.h = PACK ? hh * p.group : hh;
    t.hk = PACK ? hh : hh / p.group;
    t.m0 = mb * 2 * sub_rows;
    t.split = split;
    t.kb0 = split * p.split_blocks;
    const int range_begin = t.kb0 * kBlockN;
    const int range_end = min(p.Sk, range_begin + p.split_blocks * kBlockN);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int first = t.m0 + s * sub_rows;
        const int last = min(first + sub_rows - 1, p.Sq - 1);
        int kv_end = range_begin;
        if (first < p.Sq) kv_end = CAUSAL ? min(range_end, max(0, last + (p.Sk - p.Sq) + 1)) : range_end;
        t.nb[s] = kv_end > range_begin ? (kv_end - range_begin + kBlockN - 1) / kBlockN : 0;
    }
    t.n = max(t.nb[0], t.nb[1]);
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

// All 32 lanes wait on the same phase; the verdict is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const SyncCtx& sc) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, sc));
}

// ------------------------------------------------------------- tile ring
// The Q warp computes each work tile once (tile_info's integer divisions stay
// off every other role's path, the MMA issuer's above all) and publishes it in
// a ring of kTileSlots shared-memory entries of 32 bytes: tile_full[slot]
// completes when the entry is written; every consumer (the K/V producer, the
// MMA issuer, each softmax warp and, in the rotary variant, each rotating
// warp) copies the entry and frees it at once with one arrival on
// tile_empty[slot]. After the last tile the producer publishes an end marker
// (nb = -1).
__device__ __forceinline__ void store_tile_entry(uint8_t* entry, const TileInfo& t) {
    int4* e = reinterpret_cast<int4*>(entry);
    e[0] = make_int4(t.b, t.h, t.hk, t.m0);
    e[1] = make_int4(t.split, t.kb0, t.nb[0], t.nb[1]);
}

__device__ __forceinline__ TileInfo load_tile_entry(const uint8_t* entry) {
    const int4* e = reinterpret_cast<const int4*>(entry);
    const int4 a = e[0], c = e[1];
    TileInfo t;
    t.b = a.x;
    t.h = a.y;
    t.hk = a.z;
    t.m0 = a.w;
    t.split = c.x;
    t.kb0 = c.y;
    t.nb[0] = c.z;
    t.nb[1] = c.w;
    t.n = max(c.z, c.w);
    return t;
}

// A warp copies entry k of the tile ring and frees it (one arrival, lane 0).
// Returns false when the wait was aborted; t.n < 0 marks the end of the work.
__device__ __forceinline__ bool fetch_tile_warp(uint32_t full_bar, uint32_t empty_bar, const uint8_t* ring, uint32_t k,
                                                TileInfo& t, const SyncCtx& sc) {
    const uint32_t slot = k % kTileSlots;
    if (!warp_wait(full_bar + 8u * slot, (k / kTileSlots) & 1u, sc)) return false;
    t = load_tile_entry(ring + 32 * slot);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(empty_bar + 8u * slot);
    return true;
}

// ------------------------------------------------------------ TMA producer
// The whole warp runs this loop (so that addresses and coordinates stay
// warp-uniform); lane 0 issues the copies. The K/V tiles enter the ring in the
// order the MMA issuer takes them: K_0, then per block V_j and K_{j+1}. The
// work tiles come from the tile ring.
template <int D>
__device__ void role_tma(const CUtensorMap* tmK, const CUtensorMap* tmV, uint32_t smem, const uint8_t* smem_ptr,
                         const SyncCtx& sc) {
    using C = TileCfg<D>;
    const bool leader = (threadIdx.x & 31) == 0;
    const uint32_t bars = smem + C::kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t kv_fill = 0;
    auto load = [&](const CUtensorMap* map, const TileInfo& t, int blk) -> bool {
        const uint32_t slot = kv_fill % C::kSlots;
        if (kv_fill >= (uint32_t)C::kSlots &&
            !warp_wait(bar(C::bKVEmpty + slot), ((kv_fill / C::kSlots) - 1) & 1u, sc))
            return false;
        if (leader) {
            ptx::mbar_arrive_expect_tx(bar(C::bKVFull + slot), C::kTileBytes);
            for (int c = 0; c < C::kBoxes; ++c)
                ptx::tma_load_4d(smem + C::kKVOff + slot * C::kTileBytes + c * C::kBoxBytes, map,
                                 bar(C::bKVFull + slot), c * C::kBoxCols, t.hk, (t.kb0 + blk) * kBlockN, t.b);
        }
        ++kv_fill;
        return true;
    };
    const uint8_t* ring = smem_ptr + C::kTileOff;
    bool alive = true;
    for (uint32_t k = 0; alive; ++k) {
        TileInfo ti;
        if (!fetch_tile_warp(bar(C::bTileFull), bar(C::bTileEmpty), ring, k, ti, sc) || ti.n < 0) break;
        if (ti.n > 0) alive = load(tmK, ti, 0);
        for (int j = 0; j < ti.n && alive; ++j) {
            alive = load(tmV, ti, j);
            if (alive && j + 1 < ti.n) alive = load(tmK, ti, j + 1);
        }
    }
    // Shut down: wait until every copy this warp started has landed.
    for (uint32_t s = 0; s < (uint32_t)C::kSlots; ++s) {
        if (kv_fill > s) {
            const uint32_t last = s + C::kSlots * ((kv_fill - 1 - s) / C::kSlots);
            drain_phase(bar(C::bKVFull + s), (last / C::kSlots) & 1u, sc);
        }
    }
}

// ------------------------------------------------- rotary position embedding
// Rotation of the query rows at tile load ("ATB engineering guide" §4.1,
// fusion pattern 5; interleaved pairs as in its §8.4): the pair
// (x[2i], x[2i+1]) of the row at position pos turns by the angle of the
// table's entry (pos, i):
//   (x[2i], x[2i+1]) -> (x[2i] cos - x[2i+1] sin, x[2i+1] cos + x[2i] sin),
// in FP32, rounded once to the 16-bit input type the tensor core reads.
template <bool BF16>
__device__ __forceinline__ uint32_t rotate_pair(uint32_t w, float c, float s) {
    float x0, x1;
    if (BF16) {
        x0 = __uint_as_float(w << 16);
        x1 = __uint_as_float(w & 0xffff0000u);
    } else {
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
            : "=f"(x0), "=f"(x1)
            : "r"(w));
    }
    const float y0 = x0 * c - x1 * s, y1 = x1 * c + x0 * s;
    return BF16 ? ptx::pack_bf16x2(y0, y1) : ptx::pack_f16x2(y0, y1);
}

// One warp rotates rows [r_begin, r_end) of a 128 x D sub-tile held as
// 128-byte-swizzled 64-column boxes; the sub-tile's row r is query row
// row0 + r. Each lane owns one 16-byte chunk of the row (four pairs) and
// visits every kRowsPerPass-th row. It reads the {cos, sin} of its four pairs
// from the table once, at its first row, and then advances them by the fixed
// angle of kRowsPerPass positions with the angle-addition formulas
//   cos(a + d) = cos a cos d - sin a sin d,  sin(a + d) = sin a cos d + cos a sin d,
// so the loop touches only shared memory (no table fetch on its critical
// path). Over the at most 64 steps of a sub-tile the FP32 recurrence drifts by
// a few 2^-24 per step, far below the 16-bit spacing of the results. Rows at
// or past Sq (zero fill of the load) are skipped. The writes are made visible
// to the tensor core's (async) proxy before the caller signals.
template <int D, bool BF16>
__device__ __forceinline__ void rope_rotate_rows(uint8_t* tile, int r_begin, int r_end, int row0, const FwdParams& p) {
    using C = TileCfg<D>;
    constexpr int kChunks = D / 8;                 // 16-byte chunks per row
    constexpr int kRowsPerPass = 32 / kChunks;
    const int lane = threadIdx.x & 31;
    const int g = lane % kChunks;                  // chunk of the row: pairs 4g .. 4g+3
    const int box = g / 8, k = g % 8;
    const int r_stop = min(r_end, p.Sq - row0);
    int r = r_begin + lane / kChunks;
    if (r < r_stop) {
        const float4* table = reinterpret_cast<const float4*>(p.rope) + 2 * g;
        const float4* at = table + (size_t)(p.q_pos0 + row0 + r) * (D / 4);
        float4 a0 = __ldg(at), a1 = __ldg(at + 1);                       // {cos, sin} of the four pairs
        float4 d0 = make_float4(1.f, 0.f, 1.f, 0.f), d1 = d0;
        if (r + kRowsPerPass < r_stop) {                                 // step: position kRowsPerPass
            d0 = __ldg(table + kRowsPerPass * (D / 4));
            d1 = __ldg(table + kRowsPerPass * (D / 4) + 1);
        }
        uint8_t* col = tile + box * C::kBoxBytes;
#pragma unroll 2
        for (; r < r_stop; r += kRowsPerPass) {
            uint4* ptr = reinterpret_cast<uint4*>(col + r * 128 + ((k ^ (r & 7)) << 4));
            uint4 w = *ptr;
            w.x = rotate_pair<BF16>(w.x, a0.x, a0.y);
            w.y = rotate_pair<BF16>(w.y, a0.z, a0.w);
            w.z = rotate_pair<BF16>(w.z, a1.x, a1.y);
            w.w = rotate_pair<BF16>(w.w, a1.z, a1.w);
            *ptr = w;
            a0 = make_float4(a0.x * d0.x - a0.y * d0.y, a0.y * d0.x + a0.x * d0.y,
                             a0.z * d0.z - a0.w * d0.w, a0.w * d0.z + a0.z * d0.w);
            a1 = make_float4(a1.x * d1.x - a1.y * d1.y, a1.y * d1.x + a1.x * d1.y,
                             a1.z * d1.z - a1.w * d1.w, a1.w * d1.z + a1.z * d1.w);
        }
    }
    ptx::fence_proxy_async_shared();
    __syncwarp();
}

// Variants whose upper sub-tile's O leaves through its Q buffer (role_softmax).
template <int D, bool ADDITIVE, bool PACK>
__host__ __device__ constexpr bool kStagesO() {
    return ADDITIVE && !PACK && D == 128;
}

// Q buffer of sub-tile t (0 lower, 1 upper) of the nq-th tile with key blocks,
// and which use of that buffer it is. Sub-tiles take the three buffers in turn
// (lower, upper, next lower, ...): the next tile's lower sub-tile goes into the
// buffer the previous tile's upper sub-tile has freed, a whole tile ahead, and
// its upper sub-tile into the buffer the current lower sub-tile frees after its
// last Q K^T, one key block before the current tile ends.
__device__ __forceinline__ uint32_t q_slot(uint32_t nq, int t, uint32_t& use) {
    const uint32_t i = 2u * nq + (uint32_t)t;
    use = i / 3u;
    return i - 3u * use;
}

// Rotary variant, warps 12-15: warp 12 + q rotates rows 32q .. 32q+31 of every
// Q sub-tile once its load has landed, in the order the Q warp loads them, and
// signals "Q ready" (four arrivals per use). The four warps sit on the four
// SM sub-partitions, so each shares its issue slots with two softmax warps.
template <int D, bool BF16>
__device__ void role_rope_q(const FwdParams& p, uint32_t smem, uint8_t* smem_ptr, const SyncCtx& sc) {
    using C = TileCfg<D>;
    const bool leader = (threadIdx.x & 31) == 0;
    const int r0 = ((threadIdx.x >> 5) & 3) * 32;
    const uint32_t bars = smem + C::kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    const uint8_t* ring = smem_ptr + C::kTileOff;
    uint32_t nq = 0;
    for (uint32_t k = 0;; ++k) {
        TileInfo ti;
        if (!fetch_tile_warp(bar(C::bTileFull), bar(C::bTileEmpty), ring, k, ti, sc) || ti.n < 0) return;
        if (ti.n == 0) continue;
        for (int t = 0; t < 2; ++t) {
            uint32_t use;
            const uint32_t buf = q_slot(nq, t, use);
            if (!warp_wait(bar(C::bQFull + buf), use & 1u, sc)) return;
            rope_rotate_rows<D, BF16>(smem_ptr + C::kQOff + buf * C::kTileBytes, r0, r0 + 32,
                                      ti.m0 + t * kBlockM, p);
            if (leader) ptx::mbar_arrive(bar(C::bQRdy + buf));
        }
        ++nq;
    }
}

// ------------------------------------------------------------- Q producer
// Produces the tile ring and loads the Q sub-tiles of each work tile. An entry
// is published (and, past the CTA's own tile, taken over from an unstarted
// CTA) only when this warp is about to load that tile's Q, one tile before the
// CTA starts it: the later a tile is assigned, the better the dynamic schedule
// balances the SMs. Every other role needs entry k only when it reaches tile k,
// after this warp has loaded Q for it. The sub-tiles take the Q buffers in turn
// (q_slot): the next tile's lower sub-tile is fetched as soon as the previous
// tile's upper one is done, and its upper sub-tile while the current tile's
// last key block runs. (In the rotary variant warps 12-15 rotate each
// sub-tile after it lands.)
template <int D, bool CAUSAL, bool ADDITIVE, bool BF16, bool ROPE, bool PACK>
__device__ void role_qload(const CUtensorMap* tmQ, const CUtensorMap* tmO, const FwdParams& p, uint32_t smem,
                           uint8_t* smem_ptr, const SyncCtx& sc) {
    using C = TileCfg<D>;
    const bool leader = (threadIdx.x & 31) == 0;
    const uint32_t bars = smem + C::kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint8_t* ring = smem_ptr + C::kTileOff;
    // ---- tile ring producer: this CTA's own tile, then the tiles of CTAs that
    // had not started yet (taken over through cluster launch control), then
    // the end marker.
    uint32_t produced = 0;
    uint32_t clc_uses = 0;
    bool own = true, drained = false;
    // Index of the next tile for this CTA: 1 (tile set), 0 (none left), -1 (aborted).
    auto next_tile_index = [&](int& tile) -> int {
        if (own) {
            own = false;
            tile = (int)blockIdx.x;
            return 1;
        }
        if (drained) return 0;
        const uint32_t resp = smem + C::kClcOff;
        if (leader) {
            ptx::mbar_arrive_expect_tx(bar(C::bClc), 16);
            ptx::clc_try_cancel(resp, bar(C::bClc));
        }
        if (!warp_wait(bar(C::bClc), clc_uses & 1u, sc)) {
            // Aborting: the response must still land before the CTA may exit.
            drain_phase(bar(C::bClc), clc_uses & 1u, sc);
            return -1;
        }
        ++clc_uses;
        uint32_t x = 0;
        const bool got = ptx::clc_query(resp, x);
        __syncwarp();                              // every lane has read the response
        if (!got || x >= (uint32_t)p.n_tiles) {
            drained = true;                        // no CTA left to take over
            return 0;
        }
        tile = (int)x;
        return 1;
    };
    // Publishes the next entry. Returns 1 (t = the tile), 0 (end marker) or -1 (aborted).
    auto produce = [&](TileInfo& t) -> int {
        const uint32_t slot = produced % kTileSlots;
        if (produced >= (uint32_t)kTileSlots &&
            !warp_wait(bar(C::bTileEmpty + slot), ((produced / kTileSlots) - 1) & 1u, sc))
            return -1;
        int tile = 0;
        const int found = next_tile_index(tile);
        if (found < 0) return -1;
        if (found) t = tile_info<CAUSAL, PACK>(tile, p);
        if (!found) {
            t.b = t.h = t.hk = t.m0 = t.split = t.kb0 = 0;
            t.nb[0] = t.nb[1] = t.n = -1;
        }
        if (leader) {
            store_tile_entry(ring + 32 * slot, t);
            ptx::mbar_arrive(bar(C::bTileFull + slot));
        }
        ++produced;
        return found;
    };
    // The next tile with at least one key block (1), the end (0) or an abort (-1).
    auto next_work = [&](TileInfo& t) -> int {
        int r;
        do {
            r = produce(t);
        } while (r > 0 && t.n == 0);
        return r;
    };

    uint32_t uses[C::kQBufs] = {};              // loads issued into each buffer
    uint32_t nq = 0;                            // work tiles with at least one block
    // Staged output (see role_softmax): a buffer that held a sub-tile with
    // blocks receives that sub-tile's O from its warpgroup; before the buffer
    // is loaded again this warp waits for it (bOStaged: each warpgroup's
    // stagings alternate between two barriers of its own, and at most two of
    // them are ever pending) and stores it by TMA. The store has read the
    // buffer when wait_group.read returns, so the next load may then
    // overwrite it.
    constexpr bool kStaging = kStagesO<D, ADDITIVE, PACK>();
    const bool stage_o = kStaging && p.o_part == nullptr;
    constexpr int kSt = kStaging ? C::kQBufs : 1;
    int st_idx[kSt], st_wg[kSt], st_b[kSt], st_h[kSt], st_m[kSt];
#pragma unroll
    for (int b = 0; b < kSt; ++b) st_idx[b] = st_wg[b] = st_b[b] = st_h[b] = st_m[b] = -1;
    int n_staged[2] = {0, 0};
    auto store_staged = [&](int buf) -> bool {
        const int idx = st_idx[buf];
        if (!warp_wait(bar(C::bOStaged + 2 * st_wg[buf] + (idx & 1)), ((uint32_t)idx >> 1) & 1u, sc)) return false;
        if (leader) {
            for (int c = 0; c < C::kBoxes; ++c)
                ptx::tma_store_4d(tmO, smem + C::kQOff + buf * C::kTileBytes + c * C::kBoxBytes, c * C::kBoxCols,
                                  st_h[buf], st_m[buf], st_b[buf]);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read<0>();
        }
        __syncwarp();
        st_idx[buf] = -1;
        return true;
    };
    auto load = [&](int buf, int row0, const TileInfo& ti, bool upper) -> bool {
        if (uses[buf] > 0 && !warp_wait(bar(C::bQEmpty + buf), (uses[buf] - 1) & 1u, sc)) return false;
        if (kStaging && st_idx[buf] >= 0 && !store_staged(buf)) return false;
        if (kStaging && stage_o && ti.nb[upper ? 1 : 0] > 0) {
            st_wg[buf] = upper ? 1 : 0;
            st_idx[buf] = n_staged[upper ? 1 : 0]++;
            st_b[buf] = ti.b;
            st_h[buf] = ti.h;
            st_m[buf] = row0;
        }
        if (leader) {
            ptx::mbar_arrive_expect_tx(bar(C::bQFull + buf), C::kTileBytes);
            for (int c = 0; c < C::kBoxes; ++c)
                ptx::tma_load_4d(smem + C::kQOff + buf * C::kTileBytes + c * C::kBoxBytes, tmQ,
                                 bar(C::bQFull + buf), c * C::kBoxCols, ti.h, row0, ti.b);
        }
        ++uses[buf];
        return true;
    };
    TileInfo ti;
    while (next_work(ti) > 0) {
        uint32_t use;
        const int b0 = (int)q_slot(nq, 0, use), b1 = (int)q_slot(nq, 1, use);
        if (!load(b0, ti.m0, ti, false) || !load(b1, ti.m0 + (kBlockM >> (PACK ? p.pack_shift : 0)), ti, true))
            break;
        ++nq;
    }
    if constexpr (kStaging) {
        // The last tiles' staged O, each warpgroup's in staging order.
        for (int pass = 0; pass < C::kQBufs; ++pass) {
            int next = -1;
#pragma unroll
            for (int b = 0; b < C::kQBufs; ++b)
                if (st_idx[b] >= 0 && (next < 0 || st_wg[b] < st_wg[next] ||
                                       (st_wg[b] == st_wg[next] && st_idx[b] < st_idx[next])))
                    next = b;
            if (next < 0 || !store_staged(next)) break;
        }
        if (leader) ptx::bulk_wait_group<0>();    // every store issued here has completed
        __syncwarp();
    }
    // Shut down: wait until every copy this warp started has landed.
    for (int b = 0; b < C::kQBufs; ++b)
        if (uses[b] > 0) drain_phase(bar(C::bQFull + b), (uses[b] - 1) & 1u, sc);
}

// -------------------------------------------------------------- MMA issuer
// Issue order per KV block j of a tile with n blocks (ping-pong between the two
// query tiles, so that each softmax warpgroup works while the tensor cores run
// the other tile's two products):
//     prologue:  S0 = Q0 K0^T, S1 = Q1 K0^T
//     block j:   O0 += P0 V_j, S0 = Q0 K_{j+1}^T, O1 += P1 V_j, S1 = Q1 K_{j+1}^T
// S_t and P_t share TMEM columns. The write of S_t for block j+1 is issued by
// this thread after the product that reads P_t of block j, and the tensor core
// executes the MMAs of one issuing thread in issue order, so that read happens
// first. Each commit covers every MMA issued before it, so "S_t ready" also
// means that the previous O_t += P_t V has completed (the softmax may rescale
// O_t and overwrite P_t after it).
// Lane 0 alone runs the loop and issues every MMA and every commit (a commit
// covers the MMAs of its own thread): a single thread needs no warp votes, and
// the tensor core's queue is short, so every cycle the issuer spends between
// two groups of MMAs can leave it idle. For the same reason the next K/V slot
// is probed (without blocking) before a group is issued, and the wait after
// the group is skipped when the probe already saw the slot full.
template <int D, bool BF16, bool ROPE>
__device__ void role_mma(const FwdParams& p, uint32_t smem, const uint8_t* smem_ptr, uint32_t tmem, const SyncCtx& sc) {
    using C = TileCfg<D>;
    const bool leader = (threadIdx.x & 31) == 0;
    const uint32_t bars = smem + C::kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    constexpr uint32_t kIdescQK = ptx::idesc_f16(128, kBlockN, BF16, false, false);
    constexpr uint32_t kIdescPV = ptx::idesc_f16(128, D, BF16, false, true);
    // Base descriptors; a k-step advances the 16-byte-unit start address field.
    const uint64_t q_desc0 = ptx::sdesc_kmajor_sw128(smem + C::kQOff);
    uint32_t q_buf[2] = {0, 1};                  // Q buffers of the current tile's sub-tiles
    const uint64_t kv_desc0 = ptx::sdesc_kmajor_sw128(smem + C::kKVOff);
    const uint64_t v_desc0 = ptx::sdesc_mnmajor_sw128(smem + C::kKVOff, C::kBoxBytes);
    uint32_t kv_use = 0, nq = 0;
    uint32_t p_cnt[2] = {0, 0};
    bool issued = false;
    bool alive = true;
    constexpr int kQReady = ROPE ? C::bQRdy : C::bQFull;   // Q usable once loaded (and rotated)

    // Next K or V tile of the ring; `seen` = a probe already saw it full.
    auto acquire = [&](uint32_t& slot, bool seen = false) -> bool {
        slot = kv_use % C::kSlots;
        const bool ok = seen || wait_phase(bar(C::bKVFull + slot), (kv_use / C::kSlots) & 1u, sc);
        ++kv_use;
        if (ok) ptx::tc_fence_after_sync();
        return ok;
    };
    auto probe_next = [&]() -> bool {
        return ptx::mbar_test_wait(bar(C::bKVFull + (int)(kv_use % C::kSlots)), (kv_use / C::kSlots) & 1u);
    };
    auto commit = [&](int b) {
        if (leader) ptx::tc_commit(bar(b));
    };
    // S_t = Q K^T from Q buffer qb and the K tile in ring slot k_slot.
    auto issue_qk = [&](int t, uint32_t qb, uint32_t k_slot) {
        const uint64_t qd = q_desc0 + (uint64_t)((qb * C::kTileBytes) >> 4);
        const uint64_t kd = kv_desc0 + (uint64_t)((k_slot * C::kTileBytes) >> 4);
        if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (uint64_t)((((kk >> 2) * C::kBoxBytes) + (kk & 3) * 32) >> 4);
                ptx::mma_ss(tmem + C::s_col(t), qd + off, kd + off, kIdescQK, kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit(bar(C::bSFull + t));
        }
    };
    auto issue_pv = [&](int t, uint32_t v_slot, bool accumulate) {
        const uint64_t vd = v_desc0 + (uint64_t)((v_slot * C::kTileBytes) >> 4);
        if (leader) {
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk) {
                ptx::mma_ts(tmem + C::kOCol0 + t * D, tmem + C::s_col(t) + kk * 8,
                            vd + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
            }
        }
    };
    auto wait_p = [&](int t) -> bool {
        const bool ok = wait_phase(bar(C::bPFull + t), p_cnt[t] & 1u, sc);
        ++p_cnt[t];
        if (ok) ptx::tc_fence_after_sync();
        return ok;
    };

    if (!leader) return;
    if (p.flags & kFlagDebugStall) alive = wait_phase(bar(C::bStall), 0, sc);   // nothing ever arrives
    // Sizes of tile-ring entry k (the issuer reads only the block counts).
    const uint8_t* ring = smem_ptr + C::kTileOff;
    auto fetch = [&](uint32_t k, int& nb0, int& nb1) -> bool {
        const uint32_t slot = k % kTileSlots;
        if (!wait_phase(bar(C::bTileFull + slot), (k / kTileSlots) & 1u, sc)) return false;
        const int4 c = reinterpret_cast<const int4*>(ring + 32 * slot)[1];
        nb0 = c.z;
        nb1 = c.w;
        ptx::mbar_arrive(bar(C::bTileEmpty + slot));
        return true;
    };
    for (uint32_t k = 0; alive; ++k) {
        int n0 = 0, n1 = 0;             // block counts of the tile's sub-tiles
        if (!fetch(k, n0, n1) || n1 < 0) break;      // n1 < 0: end marker
        const int n = max(n0, n1);      // n0, n1 are n or n - 1
        if (n == 0) continue;           // no key block for any row: nothing to issue
        // Q buffers of this tile (q_slot). Both are waited for even when a
        // sub-tile has no block, to keep the parities in step; each is released
        // after its sub-tile's last Q K^T.
        uint32_t use0, use1;
        q_buf[0] = q_slot(nq, 0, use0);
        q_buf[1] = q_slot(nq, 1, use1);
        uint32_t ks, vs;
        if (!wait_phase(bar(kQReady + q_buf[0]), use0 & 1u, sc) || !acquire(ks)) { alive = false; break; }
        if (n0 > 0) issue_qk(0, q_buf[0], ks);
        issued = true;
        if (!wait_phase(bar(kQReady + q_buf[1]), use1 & 1u, sc)) { alive = false; break; }
        ptx::tc_fence_after_sync();
        ++nq;
        if (n1 > 0) issue_qk(1, q_buf[1], ks);
        commit(C::bKVEmpty + ks);
        if (n0 <= 1) commit(C::bQEmpty + q_buf[0]);
        if (n1 <= 1) commit(C::bQEmpty + q_buf[1]);
        bool v_seen = false;
        for (int j = 0; j < n; ++j) {
            const bool more = j + 1 < n;
            if (!acquire(vs, v_seen)) { alive = false; break; }
            const bool k_seen = more && probe_next();
            if (j < n0) {
                if (!wait_p(0)) { alive = false; break; }
                issue_pv(0, vs, j > 0);
                if (j == n0 - 1) commit(C::bOFull + 0);
            }
            if (more) {
                if (!acquire(ks, k_seen)) { alive = false; break; }
                if (j + 1 < n0) {
                    issue_qk(0, q_buf[0], ks);
                    if (j + 2 == n0) commit(C::bQEmpty + q_buf[0]);
                }
            }
            if (j < n1) {
                if (!wait_p(1)) { alive = false; break; }
                issue_pv(1, vs, j > 0);
                if (j == n1 - 1) commit(C::bOFull + 1);
            }
            commit(C::bKVEmpty + vs);
            if (more) {
                v_seen = probe_next();
                if (j + 1 < n1) issue_qk(1, q_buf[1], ks);
                commit(C::bKVEmpty + ks);
                if (j + 2 == n1) commit(C::bQEmpty + q_buf[1]);
            }
        }
    }
    // Shut down: every MMA lane 0 issued must finish before TMEM is freed.
    if (issued) {
        commit(C::bDrain);
        drain_phase(bar(C::bDrain), 0, sc);
    }
}

// ------------------------------------------------ softmax / epilogue warpgroup
template <int D, bool CAUSAL, bool ADDITIVE, bool BF16, bool PACK>
__device__ void role_softmax(const FwdParams& p, uint32_t smem, uint8_t* smem_ptr, uint32_t tmem, int wg,
                             const SyncCtx& sc) {
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
    // With an additive mask and D = 128 (16-bit output, no split keys, no head
    // packing), each warpgroup writes its O into its sub-tile's Q buffer, free
    // once "O ready" has arrived, and the Q warp stores it by TMA (role_qload):
    // the epilogue then skips the row-strided global stores, which compete
    // with the mask rows' loads for the L1 (those loads bound the masked
    // kernel). Without a mask, or at D = 64, the direct stores are as fast or
    // faster.
    const bool stage = kStagesO<D, ADDITIVE, PACK>() && p.o_part == nullptr;
    uint32_t nq = 0, n_staged = 0;                            // tiles with blocks; O staged so far

    const uint8_t* ring = smem_ptr + C::kTileOff;
    for (uint32_t k = 0;; ++k) {
        TileInfo ti;
        if (!fetch_tile_warp(bar(C::bTileFull), bar(C::bTileEmpty), ring, k, ti, sc)) return;
        if (ti.n < 0) break;                                  // end marker
        uint32_t use_unused;
        const uint32_t qbuf = q_slot(nq, wg, use_unused);     // this sub-tile's Q buffer
        if (ti.n > 0) ++nq;
        const int nb = ti.nb[wg];
        const int ps = PACK ? p.pack_shift : 0;
        const int row = ti.m0 + ((wg * kBlockM + r) >> ps);                   // query row
        const int hd = PACK ? ti.h + (r & ((1 << ps) - 1)) : ti.h;            // query head
        const bool row_ok = row < p.Sq;
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + (((size_t)ti.b * p.Sq + row) * p.Hq + hd) * D;
        float* lse_out = p.lse + ((size_t)ti.b * p.Hq + hd) * p.Sq + row;
        // With split keys this tile's result goes to the FP32 partial buffers.
        const bool part = p.o_part != nullptr;
        const size_t prow_index = (((size_t)ti.split * p.B + ti.b) * p.Hq + hd) * p.Sq + row;
        float* prow = part ? p.o_part + prow_index * D : nullptr;
        if (part) lse_out = p.lse_part + prow_index;
        if (nb == 0) {                                        // no visible key for any row here
            if (row_ok) {
                uint4 z = make_uint4(0, 0, 0, 0);
                if (part) {
#pragma unroll
                    for (int c = 0; c < D / 4; ++c) reinterpret_cast<uint4*>(prow)[c] = z;
                } else {
#pragma unroll
                    for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
                }
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
        const float sl = p.scale_log2;
        for (int j = 0; j < nb; ++j) {
            // Each warp waits on its own; the warpgroup agrees on whether to go
            // on at the one named barrier of the block (before the hand-off of
            // P), where a warp whose wait ran out votes to stop.
            const int key0 = (ti.kb0 + j) * kBlockN;
            // x: raw scores, or (additive mask) logits in log2 units
            float x[kBlockN];
            if (ADDITIVE) {
                // The row's mask values for this block are fetched before the wait
                // for S, so that their latency overlaps it instead of sitting on the
                // softmax's path in every block; S is then read in 32-column pieces
                // and combined in place (the mask and S fit in the register budget).
                const bool whole = key0 + kBlockN <= p.Sk;
                if (mrow != nullptr && whole && p.mask_vec4 == 2) {
#pragma unroll
                    for (int c = 0; c < kBlockN / 8; ++c) ptx::ld_global_nc_v8(mrow + key0 + 8 * c, x + 8 * c);
                } else if (mrow != nullptr && whole && p.mask_vec4 == 1) {
                    const float4* m4 = reinterpret_cast<const float4*>(mrow + key0);
#pragma unroll
                    for (int c = 0; c < kBlockN / 4; ++c) {
                        const float4 mv = ptx::ld_global_nc_v4(reinterpret_cast<const float*>(m4 + c));
                        x[4 * c + 0] = mv.x;
                        x[4 * c + 1] = mv.y;
                        x[4 * c + 2] = mv.z;
                        x[4 * c + 3] = mv.w;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        x[c] = (mrow != nullptr && key0 + c < p.Sk) ? __ldg(mrow + key0 + c) : 0.f;
                }
            }
            const bool landed = __all_sync(0xffffffffu, wait_phase(bar(C::bSFull + wg), s_phase, sc));
            s_phase ^= 1u;
            if (landed) {
                ptx::tc_fence_after_sync();
                const int vis = kv_lim - key0;                    // columns >= vis are hidden
                if (ADDITIVE) {
#pragma unroll
                    for (int c = 0; c < kBlockN / 32; ++c) {
                        uint32_t sr[32];
                        ptx::tmem_ld32(tS + 32 * c, sr);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence32(sr);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            x[32 * c + i] = fmaf(x[32 * c + i], kLog2e, __uint_as_float(sr[i]) * sl);
                    }
                } else {
                    uint32_t sr[kBlockN];
#pragma unroll
                    for (int c = 0; c < kBlockN / 32; ++c) ptx::tmem_ld32(tS + 32 * c, sr + 32 * c);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < kBlockN / 32; ++c) ptx::reg_fence32(sr + 32 * c);
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c) x[c] = __uint_as_float(sr[c]);
                }
                if (vis < kBlockN) {
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        if (c >= vis) x[c] = -INFINITY;
                }
                float mA = fmaxf(x[0], x[1]), mB = fmaxf(x[2], x[3]);
                float mC = fmaxf(x[4], x[5]), mD = fmaxf(x[6], x[7]);
#pragma unroll
                for (int c = 8; c < kBlockN; c += 8) {
                    mA = ptx::max3(mA, x[c + 0], x[c + 1]);
                    mB = ptx::max3(mB, x[c + 2], x[c + 3]);
                    mC = ptx::max3(mC, x[c + 4], x[c + 5]);
                    mD = ptx::max3(mD, x[c + 6], x[c + 7]);
                }
                float m_blk = fmaxf(fmaxf(mA, mB), fmaxf(mC, mD));
                if (!ADDITIVE) m_blk *= sl;                       // scale > 0 keeps the order
                const float m_new = fmaxf(m_used, m_blk);
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
                if (rescale) {
                    // O_t holds the sum over the previous blocks and no product is
                    // running on it: "S_t ready" covered the previous O_t += P_t V.
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
                const float nm = (m_used == -INFINITY) ? 0.f : -m_used;
                uint32_t pk[kBlockN / 2];
                float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
                for (int c = 0; c < kBlockN / 2; ++c) {
                    float a, b;
                    if (ADDITIVE)
                        ptx::add2(a, b, x[2 * c], x[2 * c + 1], nm, nm);
                    else
                        ptx::fma2(a, b, x[2 * c], x[2 * c + 1], sl, sl, nm, nm);
                    a = ptx::ex2(a);
                    b = ptx::ex2(b);
                    if (c & 1)
                        ptx::add2(l2, l3, l2, l3, a, b);
                    else
                        ptx::add2(l0, l1, l0, l1, a, b);
                    pk[c] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
                }
                l_sum += (l0 + l1) + (l2 + l3);
                ptx::tmem_st32(tS + 0, pk);
                ptx::tmem_st32(tS + 32, pk + 32);
                ptx::tmem_st_wait();
                ptx::tc_fence_before_sync();
            }
            // All 128 rows of P_t are in TMEM once the warpgroup has met; one
            // thread then tells the MMA issuer (one arrival instead of 128).
            ok = ptx::named_barrier_and(1 + wg, kBlockM, landed);
            if (!ok) break;
            if (r == 0) ptx::mbar_arrive(bar(C::bPFull + wg));
        }
        if (!ok) return;
        // ---- epilogue: O / l -> 16-bit, LSE -> FP32
        ok = ptx::named_barrier_and(1 + wg, kBlockM, wait_phase(bar(C::bOFull + wg), o_phase, sc));
        if (!ok) return;
        o_phase ^= 1u;
        ptx::tc_fence_after_sync();
        const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
        uint32_t ov[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tO + 32 * c, ov + 32 * c);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) ptx::reg_fence32(ov + 32 * c);
        if (part) {
            // FP32 O of this key range, normalised by its own sum (32-byte stores).
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(__uint_as_float(ov[8 * c + i]) * inv_l);
                if (row_ok) ptx::st_global_v8(prow + 8 * c, w);
            }
        } else if (stage) {
            // Row r in the Q buffer's layout: 64-column boxes of 128-byte rows,
            // 16-byte chunk k of row r at ((k ^ (r % 8)) * 16).
            uint8_t* qt = smem_ptr + C::kQOff + qbuf * C::kTileBytes + r * 128;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a = __uint_as_float(ov[32 * c + 2 * i]) * inv_l;
                    const float b = __uint_as_float(ov[32 * c + 2 * i + 1]) * inv_l;
                    w[i] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int g = 4 * c + i;                        // 16-byte chunk of the row
                    *reinterpret_cast<uint4*>(qt + (g / 8) * C::kBoxBytes + (((g % 8) ^ (r & 7)) << 4)) =
                        make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
            ptx::fence_proxy_async_shared();                        // visible to the TMA store
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar(C::bOStaged + 2 * wg + (int)(n_staged & 1u)));
            ++n_staged;
        } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = __uint_as_float(ov[32 * c + 2 * i]) * inv_l;
                const float b = __uint_as_float(ov[32 * c + 2 * i + 1]) * inv_l;
                w[i] = BF16 ? ptx::pack_bf16x2(a, b) : ptx::pack_f16x2(a, b);
            }
            if (row_ok) {
                if (p.flags & kFlagOVec8) {
                    ptx::st_global_v8(orow + 32 * c, w);
                    ptx::st_global_v8(orow + 32 * c + 16, w + 8);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
                    dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
                }
            }
        }
        }
        if (row_ok) *lse_out = l_sum > 0.f ? (m_used + log2f(l_sum)) * kLn2 : -INFINITY;
    }
}

// ------------------------------------------------------------------ kernel
template <int D, bool CAUSAL, bool ADDITIVE, bool BF16, bool ROPE, bool PACK>
__global__ void __launch_bounds__(kernel_threads(ROPE), 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p) {
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
            uint32_t count = 1;
            if (i >= C::bQRdy && i < C::bQRdy + C::kQBufs) count = 4;
            if (i >= C::bTileEmpty && i < C::bTileEmpty + kTileSlots) count = tile_consumers(ROPE);
            if (i >= C::bOStaged && i < C::bOStaged + 4) count = 4;
            ptx::mbar_init(bars + 8u * i, count);
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
        ptx::setmaxnreg_inc<softmax_regs(ROPE)>();
        role_softmax<D, CAUSAL, ADDITIVE, BF16, PACK>(p, smem, smem_ptr, tmem, warp >> 2, sc);
    } else if (warp < kRotateWarp0) {
        ptx::setmaxnreg_dec<control_regs(ROPE)>();
        if (warp == kMmaWarp)
            role_mma<D, BF16, ROPE>(p, smem, smem_ptr, tmem, sc);
        else if (warp == kTmaWarp)
            role_tma<D>(&tmK, &tmV, smem, smem_ptr, sc);
        else if (warp == kQWarp)
            role_qload<D, CAUSAL, ADDITIVE, BF16, ROPE, PACK>(&tmQ, &tmO, p, smem, smem_ptr, sc);
        __syncwarp();
    } else {
        ptx::setmaxnreg_dec<kRotateRegs>();
        role_rope_q<D, BF16>(p, smem, smem_ptr, sc);
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
