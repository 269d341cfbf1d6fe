// Host-buffer entry points attn_fwd_host / attn_fwd_host_f16 (declared in
// include/attn.h): the fused attention with Q, K, V, O, LSE and the mask in
// host memory, pipelined through device staging buffers.
//
// The work is cut into units (b, g): batch entry b and a group g of
// consecutive K/V heads with their query heads. Each unit's Q, K and V are
// copied into one of kSlots staging slots on the library's copy-in stream,
// the fused kernel (through the public attn_fwd / attn_fwd_f16) runs on its
// compute stream, and O and LSE go back on its copy-out stream, so that the
// copies of neighbouring units overlap the computation and each other. A slot
// is refilled only after the unit that used it has been copied out. The three
// streams are joined to the caller's stream at both ends.
//
// This is runtime plumbing around the kernel: every arithmetic step of the
// attention runs in the kernel; only copies are issued here.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/attn.h"
#include "attn_launch.h"

namespace {

constexpr int kSlots = 3;
constexpr int kMaxContexts = 64;
constexpr size_t kAlign = 256;
constexpr int kTargetUnits = 8;       // enough units to overlap copies with compute

// Streams and events of one CUDA context (they belong to the context that was
// current when they were made), keyed by the context's process-unique id.
struct Pipe {
    unsigned long long ctx_id = 0;      // 0: free entry
    bool ready = false;
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t in_done[kSlots] = {}, comp_done[kSlots] = {}, out_done[kSlots] = {};
};

std::mutex g_pipe_mutex;              // one enqueue at a time: the events are shared
Pipe g_pipes[kMaxContexts];

int pipe_for_current_device(Pipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned long long id = 0;
    if (attn::current_context_id(&id) != ATTN_OK) return ATTN_ERR_CUDA;
    Pipe* slot = nullptr;
    for (Pipe& e : g_pipes) {
        if (e.ctx_id == id) { slot = &e; break; }
        if (!slot && e.ctx_id == 0) slot = &e;
    }
    if (slot == nullptr) return ATTN_ERR_UNSUPPORTED;       // more live contexts than the cache holds
    if (slot->ctx_id != id) *slot = Pipe{};
    slot->ctx_id = id;
    Pipe& p = *slot;
    if (!p.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
        bool ok = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.s_comp, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess;
        for (int s = 0; s < kSlots && ok; ++s)
            ok = cudaEventCreateWithFlags(&p.in_done[s], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.comp_done[s], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.out_done[s], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) return ATTN_ERR_CUDA;
        p.ready = true;
    }
    *out = &p;
    return ATTN_OK;
}

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// How the problem is cut: n_groups groups of K/V heads per batch entry (the
// smallest divisor of Hkv giving at least kTargetUnits units in all).
struct Plan {
    int n_groups, hk, hq;                                  // groups; K/V and query heads per unit
    size_t q_bytes, kv_bytes, o_bytes, lse_bytes, slot_bytes, mask_bytes;
};

int make_plan(int B, int Hq, int Hkv, int Sq, int Sk, int D, int mask_kind, Plan* pl) {
    if (B < 0 || Hq < 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_CAUSAL_ADDITIVE) return ATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    int ng = Hkv;
    for (int d = 1; d <= Hkv; ++d)
        if (Hkv % d == 0 && (long long)B * d >= kTargetUnits) { ng = d; break; }
    pl->n_groups = ng;
    pl->hk = Hkv / ng;
    pl->hq = Hq / ng;
    pl->q_bytes = round_up((size_t)Sq * pl->hq * D * 2);
    pl->kv_bytes = round_up((size_t)Sk * pl->hk * D * 2);
    pl->o_bytes = pl->q_bytes;
    pl->lse_bytes = round_up((size_t)pl->hq * Sq * sizeof(float));
    pl->slot_bytes = pl->q_bytes + 2 * pl->kv_bytes + pl->o_bytes + pl->lse_bytes;
    const bool additive = mask_kind == ATTN_MASK_ADDITIVE || mask_kind == ATTN_MASK_CAUSAL_ADDITIVE;
    pl->mask_bytes = additive ? round_up((size_t)B * Sq * Sk * sizeof(float)) : 0;
    return ATTN_OK;
}

int host_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk,
              int D, float scale, int mask_kind, const float* mask, void* workspace, size_t workspace_bytes,
              cudaStream_t stream, bool bf16) {
    Plan pl{};
    const int prc = make_plan(B, Hq, Hkv, Sq, Sk, D, mask_kind, &pl);
    if (prc != ATTN_OK) return prc;
    if (B == 0 || Hq == 0 || Sq == 0) return ATTN_OK;                  // nothing to compute
    const bool additive = pl.mask_bytes > 0;
    const bool kv_empty = Sk == 0;
    if (!q || !o || !lse || (!kv_empty && (!k || !v)) || (additive && !kv_empty && !mask)) return ATTN_ERR_INVALID_ARG;
    const int units = B * pl.n_groups;
    const int slots = std::min(kSlots, units);
    const size_t need = pl.mask_bytes + (size_t)slots * pl.slot_bytes;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0 || workspace_bytes < need)
        return ATTN_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    Pipe* pp = nullptr;
    int rc = pipe_for_current_device(&pp);
    if (rc != ATTN_OK) return rc;
    Pipe& P = *pp;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };

    // Start after everything already queued on the caller's stream.
    if (!ok(cudaEventRecord(P.start, stream)) || !ok(cudaStreamWaitEvent(P.s_in, P.start, 0)) ||
        !ok(cudaStreamWaitEvent(P.s_comp, P.start, 0)) || !ok(cudaStreamWaitEvent(P.s_out, P.start, 0)))
        return ATTN_ERR_CUDA;

    char* ws = static_cast<char*>(workspace);
    char* mask_dev = ws;
    const size_t es = 2;                                          // bytes per 16-bit element
    const size_t q_row = (size_t)Hq * D * es, kv_row = (size_t)Hkv * D * es;
    const size_t q_w = (size_t)pl.hq * D * es, kv_w = (size_t)pl.hk * D * es;
    for (int u = 0; u < units; ++u) {
        const int b = u / pl.n_groups, g = u % pl.n_groups, s = u % slots;
        char* slot = ws + pl.mask_bytes + (size_t)s * pl.slot_bytes;
        char* dq = slot;
        char* dk = dq + pl.q_bytes;
        char* dv = dk + pl.kv_bytes;
        char* dout = dv + pl.kv_bytes;
        float* dl = reinterpret_cast<float*>(dout + pl.o_bytes);
        // ---- copy in (the slot's previous unit has been copied out)
        if (u >= slots && !ok(cudaStreamWaitEvent(P.s_in, P.out_done[s], 0))) return ATTN_ERR_CUDA;
        const char* hq_src = static_cast<const char*>(q) + (size_t)b * Sq * q_row + (size_t)g * q_w;
        if (!ok(cudaMemcpy2DAsync(dq, q_w, hq_src, q_row, q_w, Sq, cudaMemcpyDefault, P.s_in))) return ATTN_ERR_CUDA;
        if (!kv_empty) {
            const size_t off = (size_t)b * Sk * kv_row + (size_t)g * kv_w;
            if (!ok(cudaMemcpy2DAsync(dk, kv_w, static_cast<const char*>(k) + off, kv_row, kv_w, Sk, cudaMemcpyDefault,
                                      P.s_in)) ||
                !ok(cudaMemcpy2DAsync(dv, kv_w, static_cast<const char*>(v) + off, kv_row, kv_w, Sk, cudaMemcpyDefault,
                                      P.s_in)))
                return ATTN_ERR_CUDA;
            if (additive && g == 0) {                              // the mask of entry b, once
                const size_t mb = (size_t)Sq * Sk * sizeof(float);
                if (!ok(cudaMemcpyAsync(mask_dev + (size_t)b * mb, mask + (size_t)b * Sq * Sk, mb, cudaMemcpyDefault,
                                        P.s_in)))
                    return ATTN_ERR_CUDA;
            }
        }
        if (!ok(cudaEventRecord(P.in_done[s], P.s_in))) return ATTN_ERR_CUDA;
        // ---- compute
        if (!ok(cudaStreamWaitEvent(P.s_comp, P.in_done[s], 0))) return ATTN_ERR_CUDA;
        const float* dmask = additive ? reinterpret_cast<const float*>(mask_dev + (size_t)b * Sq * Sk * sizeof(float))
                                      : nullptr;
        rc = bf16 ? attn_fwd(dq, dk, dv, dout, dl, 1, pl.hq, pl.hk, Sq, Sk, D, scale, mask_kind, dmask,
                             reinterpret_cast<attn_stream_t>(P.s_comp))
                  : attn_fwd_f16(dq, dk, dv, dout, dl, 1, pl.hq, pl.hk, Sq, Sk, D, scale, mask_kind, dmask,
                                 reinterpret_cast<attn_stream_t>(P.s_comp));
        if (rc != ATTN_OK) return rc;
        if (!ok(cudaEventRecord(P.comp_done[s], P.s_comp))) return ATTN_ERR_CUDA;
        // ---- copy out
        if (!ok(cudaStreamWaitEvent(P.s_out, P.comp_done[s], 0))) return ATTN_ERR_CUDA;
        char* ho = static_cast<char*>(o) + (size_t)b * Sq * q_row + (size_t)g * q_w;
        float* hl = lse + ((size_t)b * Hq + (size_t)g * pl.hq) * Sq;
        if (!ok(cudaMemcpy2DAsync(ho, q_row, dout, q_w, q_w, Sq, cudaMemcpyDefault, P.s_out)) ||
            !ok(cudaMemcpyAsync(hl, dl, (size_t)pl.hq * Sq * sizeof(float), cudaMemcpyDefault, P.s_out)) ||
            !ok(cudaEventRecord(P.out_done[s], P.s_out)))
            return ATTN_ERR_CUDA;
    }
    // The caller's stream continues once the last copy-out is done (the
    // copy-out stream runs in order, so every earlier unit is done as well).
    if (!ok(cudaStreamWaitEvent(stream, P.out_done[(units - 1) % slots], 0))) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

}  // namespace

extern "C" {

size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int mask_kind) {
    Plan pl{};
    if (make_plan(B, Hq, Hkv, Sq, Sk, D, mask_kind, &pl) != ATTN_OK) return 0;
    const int units = B * pl.n_groups;
    if (units == 0 || Hq == 0 || Sq == 0) return 0;
    return pl.mask_bytes + (size_t)std::min(kSlots, units) * pl.slot_bytes;
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                  int Sk, int D, float scale, int mask_kind, const float* mask, void* workspace,
                  size_t workspace_bytes, attn_stream_t stream) {
    return host_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream), true);
}

int attn_fwd_host_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int Sq, int Sk, int D, float scale, int mask_kind, const float* mask, void* workspace,
                      size_t workspace_bytes, attn_stream_t stream) {
    return host_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream), false);
}

}  // extern "C"
