// C ABI of the fused attention forward (declared in include/attn.h).
//
// The host side follows the launch layer described in "ops-transformer：
// Transformer算子融合与推理加速实战" §3.2: check the arguments, derive the
// tiling from the shapes, pack the pointers and sizes into one launch-parameter
// struct and launch the kernel. Every check happens before anything is
// enqueued, so a rejected call has no side effect; shape errors surface here,
// at the interface (§6.2 of the same page).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "../../include/attn.h"
#include "attn_kernel.cuh"
#include "attn_launch.h"
#include "block_params.h"

namespace {

constexpr int kAbiVersion = 5;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
constexpr int kMaxContexts = 64;

std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_debug_stall{0};

// Run-time status word of each device: bit 0 = a bounded wait ran out.
__device__ unsigned int g_device_status;

// Cached state of one CUDA context (the primary context of a device, or a
// context the caller created and made current). A __device__ symbol's address,
// a function's attributes and the loaded module all belong to a context, so the
// cache is keyed by the context's process-unique id, never reused.
struct DeviceInfo {
    unsigned long long ctx_id = 0;      // 0: free entry
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    unsigned int* status = nullptr;     // device address of g_device_status
    void* noalloc_scratch = nullptr;    // device address of the allocation-free scratch array
    bool smem_attr_set[2][4][2][3] = {};   // [D is 128][mask kind][bf16][plain, rotary, packed]
    bool gemm_attr_set = false;
    bool ln_attr_set[3] = {};
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxContexts];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

template <typename Fn>
bool fetch_driver_fn(const char* name, int version, Fn* out) {
    if (*out) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    *out = reinterpret_cast<Fn>(fn);
    return true;
}

// Process-unique id of the current context; makes the current device's
// primary context current first when no context is (as the runtime would).
int context_id_for(int dev, unsigned long long* id) {
    if (!fetch_driver_fn("cuCtxGetCurrent", 4000, &g_ctx_current) || !fetch_driver_fn("cuCtxGetId", 12000, &g_ctx_id))
        return ATTN_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
    if (ctx == nullptr) {
        if (cudaSetDevice(dev) != cudaSuccess || g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
            return ATTN_ERR_CUDA;
    }
    return g_ctx_id(ctx, id) == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Cached properties of the current context (sm_103 check, SM count, status
// word). The caller holds g_mutex.
int device_info_locked(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned long long id = 0;
    int rc = context_id_for(dev, &id);
    if (rc != ATTN_OK) return rc;
    DeviceInfo* d = nullptr;
    for (DeviceInfo& e : g_devices) {
        if (e.ctx_id == id) { d = &e; break; }
        if (!d && e.ctx_id == 0) d = &e;
    }
    if (d == nullptr) return ATTN_ERR_UNSUPPORTED;           // more live contexts than the cache holds
    if (d->ctx_id != id) *d = DeviceInfo{};
    d->ctx_id = id;
    if (!d->ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        d->supported = (major == 10 && minor == 3);
        d->num_sms = sms;
        if (d->supported) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return ATTN_ERR_CUDA;
            d->status = static_cast<unsigned int*>(addr);
            if (!fetch_driver_fn("cuTensorMapEncodeTiled", 12000, &g_encode)) return ATTN_ERR_CUDA;
        }
        d->ready = true;
    }
    *out = d;
    return d->supported ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
}

int device_info(DeviceInfo** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    return device_info_locked(out);
}

}  // namespace

int attn::current_context_id(unsigned long long* id) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    return context_id_for(dev, id);
}

namespace {

// 4-D map over a (B, S, H, D) 16-bit tensor, innermost first: (D, H, S, B).
// One box = 64 head-dim columns (128 bytes, the swizzle span) x 128 rows of S.
// token_stride: elements from one (b, s) to the next (0: H * D, contiguous).
// box_heads x box_rows = 128: one box is a whole 128-row sub-tile, heads
// fastest (box_heads > 1 packs the query heads of a K/V group, see tile_info).
int encode_bshd(CUtensorMap* map, const void* base, int B, int S, int H, int D, bool bf16, long long token_stride = 0,
                int box_heads = 1) {
    const long long ts = token_stride > 0 ? token_stride : (long long)H * D;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)ts * 2, (cuuint64_t)S * ts * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)box_heads, (cuuint32_t)(128 / box_heads), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

__global__ void fill_empty_rows_kernel(uint16_t* o, size_t n_o, float* lse, size_t n_lse) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_o; i += stride) o[i] = 0;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_lse; i += stride) lse[i] = -INFINITY;
}

// Merge of the key ranges of a split computation, one warp per query row:
//   lse = log sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s
// where o_s is the softmax-weighted V of range s (normalised within the range).
// A row whose ranges are all empty (lse_s = -inf) gets o = 0, lse = -inf.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ lse_part,
                                                              uint16_t* __restrict__ o, float* __restrict__ lse,
                                                              int n_splits, int B, int Hq, int Sq) {
    constexpr int kPer = D / 32;                      // O elements per lane
    const long long rows = (long long)B * Hq * Sq;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    // row = (b * Hq + h) * Sq + i, the order of the partial buffers
    const int i = (int)(row % Sq);
    const long long bh = row / Sq;
    const int h = (int)(bh % Hq);
    const int b = (int)(bh / Hq);
    float m = -INFINITY;
    for (int s = lane; s < n_splits; s += 32) m = fmaxf(m, lse_part[(long long)s * rows + row]);
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float total = 0.f;
    if (m != -INFINITY) {
        for (int s = 0; s < n_splits; ++s) {
            const float ls = lse_part[(long long)s * rows + row];
            if (ls == -INFINITY) continue;
            const float w = expf(ls - m);
            total += w;
            const float* src = o_part + ((long long)s * rows + row) * D + lane * kPer;
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, src[e], acc[e]);
        }
    }
    const float inv = total > 0.f ? 1.f / total : 0.f;
    uint16_t* dst = o + (((long long)b * Sq + i) * Hq + h) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
        const float a = acc[e] * inv, c = acc[e + 1] * inv;
        const uint32_t packed = BF16 ? attn::ptx::pack_bf16x2(a, c) : attn::ptx::pack_f16x2(a, c);
        *reinterpret_cast<uint32_t*>(dst + e) = packed;
    }
    if (lane == 0) lse[row] = total > 0.f ? m + logf(total) : -INFINITY;
}

template <int D, bool BF16, bool ROPE, bool PACK>
int launch_d(DeviceInfo& dev, int mask_kind, const CUtensorMap& tq, const CUtensorMap& tk,
             const CUtensorMap& tv, const CUtensorMap& to, const attn::FwdParams& p, int grid, cudaStream_t stream) {
    bool* attr = dev.smem_attr_set[D == 128][mask_kind][BF16 ? 1 : 0] + (ROPE ? 1 : PACK ? 2 : 0);
    switch (mask_kind) {
        case ATTN_MASK_NONE:
            return attn::launch_fwd<D, false, false, BF16, ROPE, PACK>(*attr, tq, tk, tv, to, p, grid, stream);
        case ATTN_MASK_CAUSAL:
            return attn::launch_fwd<D, true, false, BF16, ROPE, PACK>(*attr, tq, tk, tv, to, p, grid, stream);
        case ATTN_MASK_ADDITIVE:
            return attn::launch_fwd<D, false, true, BF16, ROPE, PACK>(*attr, tq, tk, tv, to, p, grid, stream);
        default: return attn::launch_fwd<D, true, true, BF16, ROPE, PACK>(*attr, tq, tk, tv, to, p, grid, stream);
    }
}

template <bool BF16, bool ROPE, bool PACK>
int launch_any(DeviceInfo& dev, int D, int mask_kind, const CUtensorMap& tq, const CUtensorMap& tk,
               const CUtensorMap& tv, const CUtensorMap& to, const attn::FwdParams& p, int grid,
               cudaStream_t stream) {
    return D == 128 ? launch_d<128, BF16, ROPE, PACK>(dev, mask_kind, tq, tk, tv, to, p, grid, stream)
                    : launch_d<64, BF16, ROPE, PACK>(dev, mask_kind, tq, tk, tv, to, p, grid, stream);
}

// ------------------------------------------------ rotary position embedding
// Table of the rotation angles (max_pos, D/2, {cos, sin}) in FP32: entry
// (pos, i) holds cos and sin of pos * base^(-2i/D), computed in double.
__global__ void rope_table_kernel(float* table, int max_pos, int D, double base) {
    const long long n = (long long)max_pos * (D / 2);
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
        const long long pos = e / (D / 2);
        const int i = (int)(e % (D / 2));
        double sn, cs;
        sincos((double)pos * pow(base, -2.0 * i / D), &sn, &cs);
        table[2 * e] = (float)cs;
        table[2 * e + 1] = (float)sn;
    }
}

// Rotates every head vector of a (B, S, H, D) 16-bit tensor: row s sits at
// position pos0 + s; y may equal x. One warp per token (b, s): its H*D/8
// 16-byte chunks (four pairs each) are contiguous, and when D/8 divides 32 a
// lane always meets the same chunk of the head vector, so it fetches its two
// table entries (L2-resident) once per token. kUnroll chunks are loaded
// before any is stored, to keep bytes in flight (loads and stores may alias).
// Bandwidth-bound: one read and one write of the tensor.
template <bool BF16>
__global__ void __launch_bounds__(256) rope_apply_kernel(const uint4* x, uint4* y, long long n_tokens, int S,
                                                         int chunks_per_token, int chunks_per_row,
                                                         const float4* table, int pos0) {
    constexpr int kUnroll = 4;
    const int lane = threadIdx.x & 31;
    const long long n_warps = ((long long)gridDim.x * blockDim.x) >> 5;
    const bool fixed_chunk = (32 % chunks_per_row) == 0;
    for (long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < n_tokens; t += n_warps) {
        const float4* row = table + (long long)(pos0 + (int)(t % S)) * (2 * chunks_per_row);
        const uint4* xs = x + t * chunks_per_token;
        uint4* ys = y + t * chunks_per_token;
        float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
        if (fixed_chunk) {
            const int g = lane % chunks_per_row;
            c0 = row[2 * g];
            c1 = row[2 * g + 1];
        }
        for (int j0 = lane; j0 < chunks_per_token; j0 += 32 * kUnroll) {
            uint4 w[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + 32 * u;
                if (j < chunks_per_token) w[u] = xs[j];
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + 32 * u;
                if (j >= chunks_per_token) break;
                if (!fixed_chunk) {
                    const int g = j % chunks_per_row;
                    c0 = row[2 * g];
                    c1 = row[2 * g + 1];
                }
                uint4 r;
                r.x = attn::rotate_pair<BF16>(w[u].x, c0.x, c0.y);
                r.y = attn::rotate_pair<BF16>(w[u].y, c0.z, c0.w);
                r.z = attn::rotate_pair<BF16>(w[u].z, c1.x, c1.y);
                r.w = attn::rotate_pair<BF16>(w[u].w, c1.z, c1.w);
                ys[j] = r;
            }
        }
    }
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

constexpr int kMaxSplits = 1024;
// K/V bytes per group of slices in the tile order: small enough that a group's
// K/V stays in L2 (about 126 MB on GB300) beside the streamed Q and O.
constexpr double kOrderGroupKVBytes = 32.0 * (1 << 20);
constexpr size_t kWorkspaceAlign = 256;

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// SM count of the current device (148 when it cannot be read, e.g. no GPU).
int current_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
        cudaGetLastError();
        return 148;
    }
    return sms;
}

// Head packing (see tile_info): the query heads of a K/V group share each
// tile's rows when the group is a power of two and the whole query sequence
// of the group fits in one tile (decode, short prefills), except with the
// rotary embedding, whose in-kernel rotation assumes one head per tile.
// Returns log2 of the packed heads, or 0.
int pack_shift_for(int Hq, int Hkv, int Sq, bool rope) {
    if (rope || Hkv <= 0 || Hq % Hkv != 0) return 0;
    const int g = Hq / Hkv;
    if (g < 2 || (g & (g - 1)) != 0 || g > 128 || (long long)Sq * g > attn::kRowsPerTile) return 0;
    int s = 0;
    while ((1 << s) < g) ++s;
    return s;
}

// Number of key ranges for a split computation: the requested count, or (0)
// as many as fill one wave of work tiles on the device's SMs without
// exceeding it (1 when the unsplit tiles already cover every SM); never more
// than there are 128-key blocks, and every range holds the same number of
// blocks (the last may be short).
int resolve_splits(int B, int Hq, int Hkv, int Sq, int Sk, int num_splits, bool rope, int* split_blocks) {
    const int n_kb = ceil_div(Sk, attn::kBlockN);
    if (n_kb == 0) { *split_blocks = 1; return 1; }
    const int ps = pack_shift_for(Hq, Hkv, Sq, rope);
    const long long heads = ps ? Hkv : Hq;
    const long long base_tiles = std::max(1LL, (long long)B * heads * ceil_div(Sq, attn::kRowsPerTile >> ps));
    int want = num_splits;
    if (want == 0) want = num_splits == 0 && base_tiles < current_sm_count() ? (int)(current_sm_count() / base_tiles) : 1;
    want = std::min(std::min(want, n_kb), kMaxSplits);
    *split_blocks = ceil_div(n_kb, want);
    return ceil_div(n_kb, *split_blocks);
}

size_t workspace_layout(int B, int Hq, int Sq, int D, int splits, size_t* lse_off) {
    const size_t rows = (size_t)B * Hq * Sq;
    const size_t o_bytes = (size_t)splits * rows * D * sizeof(float);
    *lse_off = (o_bytes + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign;
    return *lse_off + (size_t)splits * rows * sizeof(float);
}

// Rotary embedding arguments of attn_fwd_rope / attn_fwd_rope_f16.
struct RopeArgs {
    const float* table;   // (max_pos, D/2, {cos, sin}) FP32
    int max_pos;
    int q_pos0, k_pos0;   // positions of query row 0 and key 0
    void* k_rot;          // receives the rotated keys, or null: k already holds rotated keys
};

bool rope_args_ok(const RopeArgs& r, int Sq, int Sk) {
    if (!r.table || !aligned(r.table, 16) || r.max_pos <= 0) return false;
    if (r.q_pos0 < 0 || (long long)r.q_pos0 + Sq > r.max_pos) return false;
    if (r.k_rot) {
        if (r.k_pos0 < 0 || (long long)r.k_pos0 + Sk > r.max_pos) return false;
        if (!aligned(r.k_rot, 16)) return false;
    }
    return true;
}

// Grid of a bandwidth-bound element-wise kernel: enough 256-thread blocks to
// cover the work, at most 8 per SM.
unsigned elementwise_grid(long long work, int num_sms) {
    const long long blocks = (work + 255) / 256;
    return (unsigned)std::max(1LL, std::min(blocks, 8LL * num_sms));
}

// Enqueues the key / tensor rotation pass over a (B, S, H, D) tensor.
int launch_rope_apply(const void* x, void* y, int B, int S, int H, int D, const float* table, int pos0, bool bf16,
                      int num_sms, cudaStream_t stream) {
    const long long n_tokens = (long long)B * S;
    const int per_token = H * (D / 8), per_row = D / 8;
    const unsigned grid = (unsigned)std::max(1LL, std::min((n_tokens + 7) / 8, 8LL * num_sms));   // 8 warps a block
    const auto* t4 = reinterpret_cast<const float4*>(table);
    const auto* x4 = static_cast<const uint4*>(x);
    auto* y4 = static_cast<uint4*>(y);
    if (bf16)
        rope_apply_kernel<true><<<grid, 256, 0, stream>>>(x4, y4, n_tokens, S, per_token, per_row, t4, pos0);
    else
        rope_apply_kernel<false><<<grid, 256, 0, stream>>>(x4, y4, n_tokens, S, per_token, per_row, t4, pos0);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Host-side checks of the arguments every forward entry point shares (all but
// the workspace, which depends on the entry point). Nothing is enqueued.
int check_fwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int Hq,
                   int Hkv, int Sq, int Sk, int D, int mask_kind, const float* mask, int num_splits,
                   const RopeArgs* rope) {
    if (B < 0 || Hq < 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
    if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_CAUSAL_ADDITIVE) return ATTN_ERR_INVALID_ARG;
    const bool additive = mask_kind == ATTN_MASK_ADDITIVE || mask_kind == ATTN_MASK_CAUSAL_ADDITIVE;
    // A pointer may be null only when its tensor has no elements.
    const bool q_empty = (long long)B * Sq * Hq == 0, kv_empty = (long long)B * Sk == 0;
    if ((!q && !q_empty) || (!o && !q_empty) || (!lse && !q_empty)) return ATTN_ERR_INVALID_ARG;
    if ((!k && !kv_empty) || (!v && !kv_empty)) return ATTN_ERR_INVALID_ARG;
    if (additive && !mask && !q_empty && !kv_empty) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return ATTN_ERR_INVALID_ARG;
    if (additive && !aligned(mask, 4)) return ATTN_ERR_INVALID_ARG;
    if (Sq > (1 << 30) || Sk > (1 << 30)) return ATTN_ERR_INVALID_ARG;
    if (rope && !rope_args_ok(*rope, Sq, Sk)) return ATTN_ERR_INVALID_ARG;
    if (num_splits < 0) return ATTN_ERR_INVALID_ARG;
    const int pack_shift = pack_shift_for(Hq, Hkv, Sq, rope != nullptr);
    const long long tile_heads = pack_shift ? Hkv : Hq;
    const long long rows_per_tile = attn::kRowsPerTile >> pack_shift;
    const long long n_mblk = ((long long)Sq + rows_per_tile - 1) / rows_per_tile;
    int split_blocks = 1;
    const int splits = resolve_splits(B, Hq, Hkv, Sq, Sk, num_splits, rope != nullptr, &split_blocks);
    if ((long long)B * tile_heads * n_mblk * splits > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

int attn_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                  int Sq, int Sk, int D, float scale, int mask_kind, const float* mask, cudaStream_t stream,
                  bool bf16, int num_splits = 1, void* workspace = nullptr, size_t workspace_bytes = 0,
                  const RopeArgs* rope = nullptr, long long q_stride = 0, long long kv_stride = 0) {
    // ---- arguments (host only, nothing enqueued yet)
    int rc = check_fwd_args(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mask_kind, mask, num_splits, rope);
    if (rc != ATTN_OK) return rc;
    const bool additive = mask_kind == ATTN_MASK_ADDITIVE || mask_kind == ATTN_MASK_CAUSAL_ADDITIVE;
    const int pack_shift = pack_shift_for(Hq, Hkv, Sq, rope != nullptr);
    const long long tile_heads = pack_shift ? Hkv : Hq;
    const long long rows_per_tile = attn::kRowsPerTile >> pack_shift;
    const long long n_mblk = ((long long)Sq + rows_per_tile - 1) / rows_per_tile;
    int split_blocks = 1;
    const int splits = resolve_splits(B, Hq, Hkv, Sq, Sk, num_splits, rope != nullptr, &split_blocks);
    if (B == 0 || Hq == 0 || Sq == 0) return ATTN_OK;        // nothing to compute
    size_t lse_off = 0;
    if (splits > 1) {
        if (!workspace || !aligned(workspace, kWorkspaceAlign)) return ATTN_ERR_INVALID_ARG;
        if (workspace_bytes < workspace_layout(B, Hq, Sq, D, splits, &lse_off)) return ATTN_ERR_INVALID_ARG;
    }
    if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt((float)D);

    DeviceInfo* dev = nullptr;
    rc = device_info(&dev);
    if (rc != ATTN_OK) return rc;

    if (Sk == 0) {                                            // every row sees no key
        const size_t n_o = (size_t)B * Sq * Hq * D, n_lse = (size_t)B * Hq * Sq;
        fill_empty_rows_kernel<<<dev->num_sms, 256, 0, stream>>>(static_cast<uint16_t*>(o), n_o, lse, n_lse);
        return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }

    if (rope && rope->k_rot) {                               // rotate each key once
        rc = launch_rope_apply(k, rope->k_rot, B, Sk, Hkv, D, rope->table, rope->k_pos0, bf16, dev->num_sms, stream);
        if (rc != ATTN_OK) return rc;
        k = rope->k_rot;
    }

    CUtensorMap tq, tk, tv, to;
    if (encode_bshd(&tq, q, B, Sq, Hq, D, bf16, q_stride, 1 << pack_shift) != ATTN_OK ||
        encode_bshd(&tk, k, B, Sk, Hkv, D, bf16, kv_stride) != ATTN_OK ||
        encode_bshd(&tv, v, B, Sk, Hkv, D, bf16, kv_stride) != ATTN_OK ||
        encode_bshd(&to, o, B, Sq, Hq, D, bf16) != ATTN_OK)       // O is always (B, Sq, Hq, D), contiguous
        return ATTN_ERR_CUDA;

    attn::FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.mask = additive ? mask : nullptr;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Sq = Sq;
    p.Sk = Sk;
    p.group = Hq / Hkv;
    p.n_mblk = (int)n_mblk;
    p.n_splits = splits;
    p.split_blocks = splits > 1 ? split_blocks : ceil_div(Sk, attn::kBlockN);
    p.n_tiles = (int)(B * tile_heads * n_mblk * splits);
    p.pack_shift = pack_shift;
    // Tile order (see tile_info): groups of slices holding about
    // kOrderGroupKVBytes of K/V each.
    {
        const long long slices = (long long)B * tile_heads;
        const long long share = pack_shift ? 1 : Hq / Hkv;         // query-head slices per K/V head
        const double kv_head_bytes = 4.0 * Sk * D;                 // K and V of one K/V head, 16-bit
        const long long kv_heads = std::max(1LL, (long long)(kOrderGroupKVBytes / kv_head_bytes));
        p.head_group = (int)std::max(1LL, std::min(slices, kv_heads * share));
    }
    if (splits > 1) {
        p.o_part = static_cast<float*>(workspace);
        p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + lse_off);
    }
    p.scale_log2 = scale * 1.4426950408889634f;
    p.mask_vec4 = !additive ? 0 : (aligned(mask, 32) && Sk % 8 == 0) ? 2 : (aligned(mask, 16) && Sk % 4 == 0) ? 1 : 0;
    p.flags = (aligned(o, 32) ? attn::kFlagOVec8 : 0) | (g_debug_stall.load() ? attn::kFlagDebugStall : 0);
    p.timeout_ns = g_timeout_ns.load();
    p.status = dev->status;
    p.rope = rope ? rope->table : nullptr;
    p.q_pos0 = rope ? rope->q_pos0 : 0;

    // One CTA per work tile. At most one CTA fits on an SM; the running CTAs
    // take over the tiles of CTAs that have not started yet (cluster launch
    // control), so the grid behaves as a persistent one with a dynamic,
    // longest-first schedule.
    const int grid = p.n_tiles;
    if (rope)
        rc = bf16 ? launch_any<true, true, false>(*dev, D, mask_kind, tq, tk, tv, to, p, grid, stream)
                  : launch_any<false, true, false>(*dev, D, mask_kind, tq, tk, tv, to, p, grid, stream);
    else if (pack_shift)
        rc = bf16 ? launch_any<true, false, true>(*dev, D, mask_kind, tq, tk, tv, to, p, grid, stream)
                  : launch_any<false, false, true>(*dev, D, mask_kind, tq, tk, tv, to, p, grid, stream);
    else
        rc = bf16 ? launch_any<true, false, false>(*dev, D, mask_kind, tq, tk, tv, to, p, grid, stream)
                  : launch_any<false, false, false>(*dev, D, mask_kind, tq, tk, tv, to, p, grid, stream);
    if (rc != ATTN_OK || splits == 1) return rc;

    // ---- merge the key ranges
    const long long rows = (long long)B * Hq * Sq;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    auto* o16 = static_cast<uint16_t*>(o);
    if (D == 128) {
        if (bf16) splitkv_combine_kernel<128, true><<<blocks, 256, 0, stream>>>(p.o_part, p.lse_part, o16, lse, splits, B, Hq, Sq);
        else splitkv_combine_kernel<128, false><<<blocks, 256, 0, stream>>>(p.o_part, p.lse_part, o16, lse, splits, B, Hq, Sq);
    } else {
        if (bf16) splitkv_combine_kernel<64, true><<<blocks, 256, 0, stream>>>(p.o_part, p.lse_part, o16, lse, splits, B, Hq, Sq);
        else splitkv_combine_kernel<64, false><<<blocks, 256, 0, stream>>>(p.o_part, p.lse_part, o16, lse, splits, B, Hq, Sq);
    }
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
             int Sk, int D, float scale, int mask_kind, const float* mask, attn_stream_t stream) {
    return attn_fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask,
                         reinterpret_cast<cudaStream_t>(stream), true);
}

int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                 int Sq, int Sk, int D, float scale, int mask_kind, const float* mask, attn_stream_t stream) {
    return attn_fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask,
                         reinterpret_cast<cudaStream_t>(stream), false);
}

size_t attn_splitkv_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int num_splits) {
    if (B < 0 || Hq < 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || (D != 64 && D != 128) || num_splits < 0) return 0;
    int split_blocks = 1;
    const int splits = resolve_splits(B, Hq, Hkv, Sq, Sk, num_splits, false, &split_blocks);
    if (splits <= 1) return 0;
    size_t lse_off = 0;
    return workspace_layout(B, Hq, Sq, D, splits, &lse_off);
}

int attn_splitkv_num_splits(int B, int Hq, int Hkv, int Sq, int Sk, int num_splits) {
    if (B < 0 || Hq < 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || num_splits < 0) return 0;
    int split_blocks = 1;
    return resolve_splits(B, Hq, Hkv, Sq, Sk, num_splits, false, &split_blocks);
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Sq, int Sk, int D, float scale, int mask_kind, const float* mask, int num_splits,
                     void* workspace, size_t workspace_bytes, attn_stream_t stream) {
    return attn_fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask,
                         reinterpret_cast<cudaStream_t>(stream), true, num_splits, workspace, workspace_bytes);
}

int attn_fwd_splitkv_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                         int Sq, int Sk, int D, float scale, int mask_kind, const float* mask, int num_splits,
                         void* workspace, size_t workspace_bytes, attn_stream_t stream) {
    return attn_fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask,
                         reinterpret_cast<cudaStream_t>(stream), false, num_splits, workspace, workspace_bytes);
}

int attn_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                  int Sk, int D, float scale, int mask_kind, const float* mask, const float* rope_table, int max_pos,
                  int q_pos0, int k_pos0, void* k_rot, int num_splits, void* workspace, size_t workspace_bytes,
                  attn_stream_t stream) {
    const RopeArgs r{rope_table, max_pos, q_pos0, k_pos0, k_rot};
    return attn_fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask,
                         reinterpret_cast<cudaStream_t>(stream), true, num_splits, workspace, workspace_bytes, &r);
}

int attn_fwd_rope_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int Sq, int Sk, int D, float scale, int mask_kind, const float* mask, const float* rope_table,
                      int max_pos, int q_pos0, int k_pos0, void* k_rot, int num_splits, void* workspace,
                      size_t workspace_bytes, attn_stream_t stream) {
    const RopeArgs r{rope_table, max_pos, q_pos0, k_pos0, k_rot};
    return attn_fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask,
                         reinterpret_cast<cudaStream_t>(stream), false, num_splits, workspace, workspace_bytes, &r);
}

int attn_rope_table(float* table, int max_pos, int D, double base, attn_stream_t stream) {
    if (max_pos < 0 || D <= 0 || D % 2 != 0 || !(base > 1.0) || !std::isfinite(base)) return ATTN_ERR_INVALID_ARG;
    if ((long long)max_pos * D > (1LL << 31)) return ATTN_ERR_INVALID_ARG;
    if (max_pos == 0) return ATTN_OK;
    if (!table || !aligned(table, 16)) return ATTN_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != ATTN_OK) return rc;
    const long long n = (long long)max_pos * (D / 2);
    rope_table_kernel<<<elementwise_grid(n, dev->num_sms), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        table, max_pos, D, base);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"

namespace {

int rope_apply_impl(const void* x, void* y, int B, int S, int H, int D, const float* table, int max_pos, int pos0,
                    cudaStream_t stream, bool bf16) {
    if (B < 0 || S < 0 || H < 0 || D <= 0 || D % 8 != 0 || max_pos < 0 || pos0 < 0) return ATTN_ERR_INVALID_ARG;
    if ((long long)pos0 + S > max_pos || (long long)H * (D / 8) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    const long long n_chunks = (long long)B * S * H * (D / 8);
    if (n_chunks == 0) return ATTN_OK;
    if (!x || !y || !table || !aligned(x, 16) || !aligned(y, 16) || !aligned(table, 16)) return ATTN_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != ATTN_OK) return rc;
    return launch_rope_apply(x, y, B, S, H, D, table, pos0, bf16, dev->num_sms, stream);
}

}  // namespace

extern "C" {

int attn_rope_apply(const void* x, void* y, int B, int S, int H, int D, const float* rope_table, int max_pos, int pos0,
                    attn_stream_t stream) {
    return rope_apply_impl(x, y, B, S, H, D, rope_table, max_pos, pos0, reinterpret_cast<cudaStream_t>(stream), true);
}

int attn_rope_apply_f16(const void* x, void* y, int B, int S, int H, int D, const float* rope_table, int max_pos,
                        int pos0, attn_stream_t stream) {
    return rope_apply_impl(x, y, B, S, H, D, rope_table, max_pos, pos0, reinterpret_cast<cudaStream_t>(stream), false);
}

}  // extern "C"

// ------------------------------------------------------------ attention block
namespace {

// 2-D map over a row-major (rows x cols) bf16 matrix: boxes of 64 columns
// (128 bytes, the swizzle span) x box_rows rows; out-of-range reads are zero.
int encode_rows(CUtensorMap* map, const void* base, long long rows, long long cols, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

bool linear_args_ok(const void* a, const void* w, const void* bias, const void* residual, const void* out, int M, int N,
                    int K) {
    if (M < 0 || N <= 0 || K <= 0 || N % 32 != 0 || K % 8 != 0) return false;
    if ((long long)M * N > (1LL << 40) || (long long)M * K > (1LL << 40)) return false;
    if (M == 0) return true;
    if (!a || !w || !out) return false;
    return aligned(a, 16) && aligned(w, 16) && aligned(out, 16) && aligned(bias, 16) && aligned(residual, 16);
}

// Enqueues out = a w^T (+ bias) (+ residual); arguments already checked.
int linear_impl(DeviceInfo& dev, const void* a, const void* w, const void* bias, const void* residual, void* out, int M,
                int N, int K, cudaStream_t stream) {
    if (M == 0) return ATTN_OK;
    CUtensorMap ta, tw;
    if (encode_rows(&ta, a, M, K, attn::gemm::kBM) != ATTN_OK || encode_rows(&tw, w, N, K, attn::gemm::kBN) != ATTN_OK)
        return ATTN_ERR_CUDA;
    attn::gemm::GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.bias = static_cast<const uint16_t*>(bias);
    p.residual = static_cast<const uint16_t*>(residual);
    p.out = static_cast<uint16_t*>(out);
    p.ldo = N;
    p.ldr = N;
    p.tiles_m = ceil_div(M, attn::gemm::kBM);
    p.tiles_n = ceil_div(N, attn::gemm::kBN);
    p.n_tiles = p.tiles_m * p.tiles_n;
    p.k_steps = ceil_div(K, attn::gemm::kBK);
    // Raster order for L2 reuse (129 MB on GB300): when W fits in about a third
    // of L2 it stays resident whatever the order, so small groups stream each
    // A row panel once; otherwise a group's A row panels (about 32 MiB) stay
    // resident while the W column panels stream past them.
    const double w_bytes = 2.0 * N * K, a_panel = 2.0 * attn::gemm::kBM * K;
    int group = 8;
    if (w_bytes > 40e6) group = std::max(8, (int)((32 << 20) / a_panel));
    p.group_rows = std::max(1, std::min(group, p.tiles_m));
    p.timeout_ns = g_timeout_ns.load();
    p.status = dev.status;
    const int grid = p.n_tiles < dev.num_sms ? p.n_tiles : dev.num_sms;
    return attn::gemm::launch(dev.gemm_attr_set, ta, tw, p, grid, stream);
}

bool layernorm_args_ok(const void* x, const void* gamma, const void* beta, const void* y, int M, int H) {
    if (M < 0 || H < 8 || H > 8192 || H % 8 != 0) return false;
    if (M == 0) return true;
    if (!x || !gamma || !beta || !y) return false;
    return aligned(x, 16) && aligned(gamma, 16) && aligned(beta, 16) && aligned(y, 16);
}

float layernorm_eps(float eps) { return (eps > 0.f && std::isfinite(eps)) ? eps : 1e-5f; }

// Workspace of attn_block_fwd: normalised x, packed q|k|v, attention output
// (each bf16, 256-byte aligned), then the FP32 LSE.
struct BlockLayout {
    size_t n_off, qkv_off, a_off, lse_off, total;
};

bool block_layout(int B, int S, int Hq, int Hkv, int D, BlockLayout* L) {
    if (B < 0 || S < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || (D != 64 && D != 128)) return false;
    const long long M = (long long)B * S, hidden = (long long)Hq * D, F = (long long)(Hq + 2 * Hkv) * D;
    if (hidden > 8192 || M > (1LL << 31)) return false;
    auto up = [](size_t x) { return (x + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign; };
    L->n_off = 0;
    L->qkv_off = up(L->n_off + (size_t)M * hidden * 2);
    L->a_off = up(L->qkv_off + (size_t)M * F * 2);
    L->lse_off = up(L->a_off + (size_t)M * hidden * 2);
    L->total = up(L->lse_off + (size_t)B * Hq * S * sizeof(float));
    return true;
}

}  // namespace

extern "C" {

int attn_linear(const void* a, const void* w, const void* bias, const void* residual, void* out, int M, int N, int K,
                attn_stream_t stream) {
    if (!linear_args_ok(a, w, bias, residual, out, M, N, K)) return ATTN_ERR_INVALID_ARG;
    if (M == 0) return ATTN_OK;
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != ATTN_OK) return rc;
    return linear_impl(*dev, a, w, bias, residual, out, M, N, K, reinterpret_cast<cudaStream_t>(stream));
}

int attn_layernorm(const void* x, const void* gamma, const void* beta, void* y, int M, int H, float eps,
                   attn_stream_t stream) {
    if (!layernorm_args_ok(x, gamma, beta, y, M, H)) return ATTN_ERR_INVALID_ARG;
    if (M == 0) return ATTN_OK;
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != ATTN_OK) return rc;
    return attn::launch_layernorm(dev->ln_attr_set, static_cast<const uint16_t*>(x),
                                  static_cast<const uint16_t*>(gamma), static_cast<const uint16_t*>(beta),
                                  static_cast<uint16_t*>(y), M, H, layernorm_eps(eps), dev->num_sms,
                                  reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_qkvpacked(const void* qkv, void* o, float* lse, int B, int S, int Hq, int Hkv, int D, float scale,
                       int mask_kind, const float* mask, attn_stream_t stream) {
    if (Hkv <= 0 || Hq < 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
    const long long F = (long long)(Hq + 2 * Hkv) * D;
    const char* base = static_cast<const char*>(qkv);
    const void* k = base ? base + (size_t)Hq * D * 2 : nullptr;
    const void* v = base ? base + (size_t)(Hq + Hkv) * D * 2 : nullptr;
    return attn_fwd_impl(qkv, k, v, o, lse, B, Hq, Hkv, S, S, D, scale, mask_kind, mask,
                         reinterpret_cast<cudaStream_t>(stream), true, 1, nullptr, 0, nullptr, F, F);
}

size_t attn_block_workspace_bytes(int B, int S, int Hq, int Hkv, int D) {
    BlockLayout L{};
    return block_layout(B, S, Hq, Hkv, D, &L) ? L.total : 0;
}

int attn_block_fwd(const void* x, const void* ln_gamma, const void* ln_beta, const void* w_qkv, const void* b_qkv,
                   const void* w_o, const void* b_o, void* y, int B, int S, int Hq, int Hkv, int D, float eps,
                   int causal, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
    BlockLayout L{};
    if (!block_layout(B, S, Hq, Hkv, D, &L)) {
        if (B < 0 || S < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
        return ATTN_ERR_UNSUPPORTED;                       // head dimension or hidden size
    }
    const int M = B * S, hidden = Hq * D, F = (Hq + 2 * Hkv) * D;
    if (M == 0) return ATTN_OK;
    if (!workspace || !aligned(workspace, kWorkspaceAlign) || workspace_bytes < L.total) return ATTN_ERR_INVALID_ARG;
    if (!layernorm_args_ok(x, ln_gamma, ln_beta, workspace, M, hidden)) return ATTN_ERR_INVALID_ARG;
    if (!linear_args_ok(workspace, w_qkv, b_qkv, nullptr, workspace, M, F, hidden)) return ATTN_ERR_INVALID_ARG;
    if (!linear_args_ok(workspace, w_o, b_o, x, y, M, hidden, hidden)) return ATTN_ERR_INVALID_ARG;
    if (!b_qkv || !b_o) return ATTN_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != ATTN_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    void* n = ws + L.n_off;
    void* qkv = ws + L.qkv_off;
    void* a = ws + L.a_off;
    float* lse = reinterpret_cast<float*>(ws + L.lse_off);
    rc = attn::launch_layernorm(dev->ln_attr_set, static_cast<const uint16_t*>(x),
                                static_cast<const uint16_t*>(ln_gamma), static_cast<const uint16_t*>(ln_beta),
                                static_cast<uint16_t*>(n), M, hidden, layernorm_eps(eps), dev->num_sms, st);
    if (rc != ATTN_OK) return rc;
    rc = linear_impl(*dev, n, w_qkv, b_qkv, nullptr, qkv, M, F, hidden, st);
    if (rc != ATTN_OK) return rc;
    rc = attn_fwd_qkvpacked(qkv, a, lse, B, S, Hq, Hkv, D, 0.f, causal ? ATTN_MASK_CAUSAL : ATTN_MASK_NONE, nullptr,
                            stream);
    if (rc != ATTN_OK) return rc;
    return linear_impl(*dev, a, w_o, b_o, x, y, M, hidden, hidden, st);
}

}  // extern "C"

namespace {

// Scratch for attn_fwd_splitkv_noalloc: one fixed array per device that loads
// this library, held until the process exits, shared by every call.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context. In host code
// the array's name is only a host-side stand-in, so its address must come from
// cudaGetSymbolAddress, once per context, with that context current.
int noalloc_scratch(void** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo* d = nullptr;
    int rc = device_info_locked(&d);
    if (rc != ATTN_OK) return rc;
    if (!d->noalloc_scratch) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
        d->noalloc_scratch = ptr;
    }
    *out = d->noalloc_scratch;
    return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                             int Hkv, int Sq, int Sk, int D, float scale, int mask_kind, const float* mask,
                             int num_splits, attn_stream_t stream) {
    // The same argument checks as attn_fwd_splitkv first; then refuse a problem
    // whose partial results would not fit in the fixed scratch array.
    int rc = check_fwd_args(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mask_kind, mask, num_splits, nullptr);
    if (rc != ATTN_OK) return rc;
    if (attn_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, num_splits) > kNoAllocScratchBytes)
        return ATTN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != ATTN_OK) return rc;
    return attn_fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask,
                         reinterpret_cast<cudaStream_t>(stream), true, num_splits, scratch, kNoAllocScratchBytes);
}

int attn_last_status(attn_stream_t stream) {
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc != ATTN_OK) return rc;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned int word = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_status, sizeof word) != cudaSuccess) return ATTN_ERR_CUDA;
    if (word != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) return ATTN_ERR_CUDA;
    return (word & attn::kStatusTimeout) ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_OK;
}

const char* attn_status_string(int code) {
    switch (code) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
        default: return "ATTN_UNKNOWN_STATUS";
    }
}

int attn_set_wait_timeout_ns(unsigned long long ns) {
    g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs);
    return ATTN_OK;
}

int attn_debug_inject_stall(int on) {
    g_debug_stall.store(on ? 1 : 0);
    return ATTN_OK;
}

int attn_abi_version(void) { return kAbiVersion; }

}  // extern "C"
