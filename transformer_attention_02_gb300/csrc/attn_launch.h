// Host-side launchers of the compiled forward-kernel variants.
//
// Each variant (head dimension, causal mask, additive mask, 16-bit type,
// rotary embedding of the queries, GQA head packing) is compiled in one of the fwd_*.cu
// translation units, so that the variants build in parallel; the C ABI in
// attn_api.cu reaches them only through launch_fwd.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

struct FwdParams;

// Launches attn_fwd_kernel<D, CAUSAL, ADDITIVE, BF16, ROPE, PACK> with `grid`
// CTAs on `stream` (tensor maps of Q, K, V and of the output O, which the
// kernel stores through for the upper sub-tiles when it writes 16-bit O). `attr_set` caches, per device, that the
// variant's shared-memory attribute has been set and its register count
// checked (the in-kernel register split needs exactly the launch count).
// Returns ATTN_OK, ATTN_ERR_UNSUPPORTED (register count differs) or
// ATTN_ERR_CUDA.
template <int D, bool CAUSAL, bool ADDITIVE, bool BF16, bool ROPE, bool PACK>
int launch_fwd(bool& attr_set, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& to, const FwdParams& p, int grid, cudaStream_t stream);

// Process-unique id of the current CUDA context (the current device's primary
// context is made current first when no context is). Per-context caches of the
// library are keyed by it. Returns ATTN_OK or ATTN_ERR_CUDA.
int current_context_id(unsigned long long* id);

}  // namespace attn
