/*
 * attn.h — C ABI of the fused attention forward for NVIDIA GB300 (sm_103a).
 *
 * One operation: O = softmax(scale * Q K^T + mask) V, computed in a single
 * kernel launch with the softmax done online, block by block, so that the
 * Sq x Sk score matrix never reaches device memory. The per-row running
 * maximum and sum stay in FP32 on chip; both matrix products accumulate in
 * FP32; the outputs are O in the input's 16-bit type and the FP32 row
 * log-sum-exp.
 *
 * Passages that define the operation (the pages are cited by title):
 *  [GUIDE]  "ATB engineering guide" (hwcomputing.csdn.net/6a59a88310ee7a33f28e5ce9):
 *           §4.1 pattern 2 (MatMul(QK) + Softmax + MatMul(QKV) fused, O(N) memory),
 *           §5.1 (the eager formula: scores * scale -> softmax -> times V),
 *           §2.1 and §8.2 (MhaV3: head_num, kv_head_num for MQA/GQA, scale,
 *           is_causal; the attention mask appended as an optional input),
 *           §7 pitfall 2 (log-sum-exp for numerical stability).
 *  [GRAPH]  "CANN-ATB图优化-昇腾NPU怎么把PyTorch计算图改造成融合算子",
 *           Pattern 2: Q·K^T -> Scale -> Mask -> Softmax -> ·V becomes
 *           FlashAttention(Q, K, V, mask, scale).
 *  [OPS]    "ops-transformer：Transformer算子融合与推理加速实战":
 *           §2.2 (online softmax, block by block), §2.4 (FP32 accumulation,
 *           FP32 max/sum statistics on chip, cast only at write-out),
 *           §3.2 (B and H independent, sequence blocks, local max and sum),
 *           §4.2 ((B, S, H, D) inputs, D of 64 or 128, scale defaults to
 *           1/sqrt(D), optional intermediate output), §6.2 (shape errors are
 *           reported at the interface), §6.4 (empty inputs must work).
 *  [MAP]    "CANN-ops-transformer和ATB-昇腾NPU上算子和加速库怎么配合",
 *           paragraph on how ATB calls ops-transformer: an unsupported head
 *           dimension falls back to standard attention there; here it is an
 *           error code instead, because this library has no second path.
 *
 * Conventions shared by every entry point:
 *  - Pointers marked "device" are CUDA device addresses on the current device;
 *    "host" pointers are ordinary host memory. The caller owns every buffer.
 *  - No call allocates device memory (no cudaMalloc, no cudaFree), keeps
 *    per-call state or synchronises implicitly: work is enqueued on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream). The library's
 *    module does hold two fixed device arrays in every CUDA context that
 *    loads it, for as long as the context lives: a 4-byte run-time status word
 *    and the 32 MiB scratch array used only by attn_fwd_splitkv_noalloc.
 *  - Per-context state (the status word's address, kernel attributes, the
 *    host pipeline's streams) is cached per CUDA context, keyed by the
 *    context's unique id, so the current context may be a device's primary
 *    context or one the caller created; with no context current, the current
 *    device's primary context is made current, as the CUDA runtime does.
 *  - Every argument is checked on the host before anything is launched; a
 *    rejected call launches nothing and writes nothing.
 *  - Return values are attn_status codes (0 = success), as in [GUIDE] §8.1's
 *    "status != 0 means failure" convention.
 */
#ifndef TRANSFORMER_ATTENTION_02_GB300_ATTN_H
#define TRANSFORMER_ATTENTION_02_GB300_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, without requiring the CUDA headers. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_MASK_NONE = 0,             /* every key visible                         */
    ATTN_MASK_CAUSAL = 1,           /* key j visible to query i iff j <= i+Sk-Sq */
    ATTN_MASK_ADDITIVE = 2,         /* FP32 mask (B, Sq, Sk) added to the logits */
    ATTN_MASK_CAUSAL_ADDITIVE = 3   /* both                                      */
} attn_mask_kind;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad mask kind,
                                       Hq not a multiple of Hkv, misalignment    */
    ATTN_ERR_UNSUPPORTED = 2,       /* D not 64/128, device is not sm_103        */
    ATTN_ERR_CUDA = 3,              /* a CUDA runtime/driver call failed          */
    ATTN_ERR_DEVICE_TIMEOUT = 4     /* a kernel gave up on a bounded wait         */
} attn_status;

/*
 * attn_fwd — fused attention forward, bf16 in, bf16 O and FP32 LSE out.
 *
 *   q     device, bf16, (B, Sq, Hq, D)  contiguous, row-major, 16-byte aligned
 *   k, v  device, bf16, (B, Sk, Hkv, D) contiguous, row-major, 16-byte aligned
 *   o     device, bf16, (B, Sq, Hq, D)  written; 16-byte aligned; must not
 *         overlap the inputs
 *   lse   device, FP32, (B, Hq, Sq)     written; natural-log log-sum-exp of
 *         each row of scaled (and masked) logits; 4-byte aligned
 *   B, Hq, Hkv, Sq, Sk, D   sizes; Hq must be a multiple of Hkv (MHA: equal,
 *         GQA: Hq/Hkv query heads share one K/V head, MQA: Hkv = 1); query
 *         head h reads K/V head h / (Hq / Hkv); D must be 64 or 128
 *   scale multiplies Q K^T; a value that is not finite or is <= 0 selects the
 *         default 1/sqrt(D) ([OPS] §4.2; C has no default arguments)
 *   mask_kind  one of attn_mask_kind; causal alignment is bottom-right
 *   mask  device, FP32, (B, Sq, Sk), broadcast over heads, 4-byte aligned;
 *         required for the additive kinds and ignored otherwise; -inf entries
 *         hide a key. Rows are read with 32-byte loads when the mask is
 *         32-byte aligned and Sk % 8 == 0 (16-byte loads when 16-byte aligned
 *         and Sk % 4 == 0), which is faster; any 4-byte aligned mask works.
 *   stream     CUDA stream to enqueue on
 *   A pointer may be null only when its tensor has no elements (for example
 *   k and v when B or Sk is 0).
 *
 * Semantics: o[b,i,h,:] = sum_j softmax_j(s_ij) v[b,j,h/(Hq/Hkv),:] with
 * s_ij = scale <q[b,i,h,:], k[b,j,g,:]> + mask[b,i,j]. A row with no visible
 * key gets o = 0 and lse = -inf (never NaN). B, Hq or Sq of zero is a no-op
 * that returns ATTN_OK; Sk = 0 makes every row such an empty row.
 * Returns ATTN_OK once the work is enqueued (errors found by the kernel at run
 * time are reported by attn_last_status).
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int Hq, int Hkv, int Sq, int Sk, int D,
             float scale, int mask_kind, const float *mask, attn_stream_t stream);

/*
 * attn_fwd_f16 — the same operation with IEEE fp16 Q, K, V and O (FP32
 * accumulation, FP32 running statistics, P rounded to fp16 for the second
 * product, FP32 LSE). The pages run this operator in FP16 ([GUIDE] §5.1
 * benchmark tensors, §8.2 "dtype": FP16). Arguments, layout, alignment,
 * ownership and errors are exactly those of attn_fwd.
 */
int attn_fwd_f16(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int Hq, int Hkv, int Sq, int Sk, int D,
                 float scale, int mask_kind, const float *mask, attn_stream_t stream);

/*
 * GQA head packing (all entry points except attn_fwd_rope): when the query
 * heads per K/V head, G = Hq / Hkv, is a power of two and Sq * G <= 256 (decode
 * and short prefills), the G query heads of a K/V head share each work tile's
 * 128 rows, so each K/V block is streamed once per K/V head rather than once
 * per query head. The results are those of the unpacked computation.
 *
 * Split-key ("split-KV") variants, for few query rows against a long key/value
 * sequence: decode and short prefill over a KV cache ("ATB orchestration blog"
 * (hwcomputing.csdn.net/6a15a709662f9a54cb774da1) §四, FlashAttention with
 * kv_cache; [GUIDE] §6.2, LLaMA/GPT with a KV cache; [MAP], ATB passes the KV
 * cache in and out of FlashAttention). The keys are cut into `num_splits`
 * contiguous ranges of whole 128-key blocks; each (b, h, 256-query-row, range)
 * is one work tile of the fused kernel, which writes the range's FP32 output
 * (normalised within the range) and its LSE ([OPS] §4.2 intermediate output)
 * to the workspace; a second kernel merges the ranges:
 *     lse = log sum_s exp(lse_s),   o = sum_s exp(lse_s - lse) o_s.
 * The result equals attn_fwd's up to rounding.
 *
 *   num_splits  number of key ranges; 0 picks as many as fill one wave of
 *               work tiles on the current device's SMs (1 when the unsplit
 *               tiles already cover them); at most one range per 128-key
 *               block, at most 1024.
 *               When the resolved count is 1 nothing is split and no
 *               workspace is needed.
 *   workspace   device scratch of at least attn_splitkv_workspace_bytes(...)
 *               bytes, 256-byte aligned, owned by the caller; its contents are
 *               overwritten. Two calls in flight at once need two workspaces.
 *   workspace_bytes  its size.
 * Other arguments and errors as for attn_fwd / attn_fwd_f16; a missing,
 * misaligned or too small workspace is ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int Hq, int Hkv, int Sq, int Sk, int D,
                     float scale, int mask_kind, const float *mask, int num_splits,
                     void *workspace, size_t workspace_bytes, attn_stream_t stream);
int attn_fwd_splitkv_f16(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int Hq, int Hkv, int Sq, int Sk, int D,
                         float scale, int mask_kind, const float *mask, int num_splits,
                         void *workspace, size_t workspace_bytes, attn_stream_t stream);

/* attn_splitkv_num_splits — the number of key ranges attn_fwd_splitkv uses
 * for these sizes on the current device (host only; 0 on invalid sizes).
 * For attn_fwd_rope pass Hkv = Hq (its tiles never pack query heads). */
int attn_splitkv_num_splits(int B, int Hq, int Hkv, int Sq, int Sk, int num_splits);

/* attn_splitkv_workspace_bytes — workspace bytes attn_fwd_splitkv needs for
 * these sizes on the current device (host only; 0 when nothing is split or
 * the sizes are invalid). For attn_fwd_rope pass Hkv = Hq. */
size_t attn_splitkv_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int num_splits);

/*
 * attn_fwd_splitkv_noalloc — attn_fwd_splitkv (bf16) for callers that cannot
 * allocate device memory: for example a plug-in running inside a host
 * framework that owns all device memory and forbids allocations after start-up,
 * or a latency-critical path that must not pay for (or synchronise on)
 * cudaMalloc. It takes no workspace: the partial results live in a fixed
 * 32 MiB array in the library's own device memory (a static __device__
 * array, present on every GPU that loads the library until the process exits).
 * The pages have no counterpart; this entry point exists only for such callers.
 *
 *   Arguments, layout, results and errors as for attn_fwd_splitkv.
 *   Limit: attn_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, num_splits) must not
 *   exceed 32 MiB (33554432 bytes); larger problems are refused with
 *   ATTN_ERR_UNSUPPORTED before anything is launched.
 *   The first call in each CUDA context looks up the array's device address
 *   in that context (cudaGetSymbolAddress, which may synchronise); make that
 *   first call before any stream capture.
 *   All calls in a context share the one array and it keeps the last call's
 *   contents. Nothing in it needs to start at zero (every partial result is
 *   written before it is read), but calls whose work overlaps on the GPU (for
 *   example on two streams at once) race on it: serialise them.
 *   The call itself allocates nothing: no cudaMalloc, no cudaFree, no
 *   allocating library routine.
 */
int attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int Hq, int Hkv, int Sq, int Sk, int D,
                             float scale, int mask_kind, const float *mask, int num_splits,
                             attn_stream_t stream);

/*
 * Rotary position embedding (RoPE) fused with the attention: [GUIDE] §4.1
 * fusion pattern 5 (RoPE(Q) + RoPE(K) + attention as one operation, no
 * rotated temporaries) and §8.4 (interleaved pairs, rotary base 10000,
 * fuse_with_attention). The pair (x[2i], x[2i+1]) of a head vector at
 * position pos turns by the angle pos * base^(-2i/D):
 *     (x[2i], x[2i+1]) -> (x[2i] cos - x[2i+1] sin, x[2i+1] cos + x[2i] sin).
 * The rotated vectors are rounded to the input's 16-bit type (the type the
 * tensor cores read), as the reference rotation of §8.4 returns them.
 *
 * attn_rope_table — fills `table` (device, FP32, max_pos x D/2 x 2,
 * 16-byte aligned, caller-owned) with {cos, sin} of pos * base^(-2i/D) for
 * pos < max_pos, i < D/2, evaluated in double and rounded to FP32. D even,
 * base > 1, max_pos * D <= 2^31. Build it once per (max_pos, D, base) and
 * pass it to the calls below.
 */
int attn_rope_table(float *table, int max_pos, int D, double base, attn_stream_t stream);

/*
 * attn_rope_apply / attn_rope_apply_f16 — rotate every head vector of the
 * (B, S, H, D) 16-bit tensor x (device, 16-byte aligned) into y (same shape,
 * may equal x: in place); row s is at position pos0 + s. D a multiple of 8;
 * pos0 >= 0 and pos0 + S <= max_pos. For keys written once into a cache and
 * read by many later calls (the cache then holds rotated keys).
 * Bandwidth-bound: one read and one write of x.
 */
int attn_rope_apply(const void *x, void *y, int B, int S, int H, int D,
                    const float *rope_table, int max_pos, int pos0, attn_stream_t stream);
int attn_rope_apply_f16(const void *x, void *y, int B, int S, int H, int D,
                        const float *rope_table, int max_pos, int pos0, attn_stream_t stream);

/*
 * attn_fwd_rope / attn_fwd_rope_f16 — attention of the rotated queries and
 * keys: O = softmax(scale * rot(Q) rot(K)^T + mask) V, with query row i at
 * position q_pos0 + i and key j at k_pos0 + j.
 *
 * The queries are rotated inside the attention kernel, after each Q tile's
 * load lands in shared memory and before the tensor cores read it; no rotated
 * copy of Q exists. The keys are rotated once per key: rotating a 128-key tile
 * takes about 1,500 warp instructions, every query tile of the head would
 * repeat it (8 to 64 times on typical shapes), and the SM's issue slots in the
 * tensor cores' time for that tile (about 1,000 cycles per product pair at
 * D = 128) are mostly taken by the softmax already. Hence:
 *   k_rot   device buffer of k's shape and layout (16-byte aligned) that
 *           receives rot(K) from a bandwidth-bound pass enqueued before the
 *           attention kernel (k_rot may equal k: the keys are then rotated in
 *           place); or NULL: k already holds rotated keys (a KV cache filled
 *           through attn_rope_apply) and k_pos0 is not used. k_rot is written
 *           only when there is output to compute (B, Hq, Sq, Sk all > 0). It
 *           must not overlap q, v, o, lse or mask.
 *   rope_table, max_pos  the table of attn_rope_table, built for this D;
 *           q_pos0 >= 0 and q_pos0 + Sq <= max_pos; with k_rot, also
 *           k_pos0 >= 0 and k_pos0 + Sk <= max_pos.
 *   num_splits, workspace, workspace_bytes  as for attn_fwd_splitkv
 *           (num_splits = 1 with a NULL workspace: one pass, no split).
 * Other arguments, results and errors as for attn_fwd_splitkv /
 * attn_fwd_splitkv_f16; bad rotary arguments are ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_rope(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int Hq, int Hkv, int Sq, int Sk, int D,
                  float scale, int mask_kind, const float *mask,
                  const float *rope_table, int max_pos, int q_pos0, int k_pos0, void *k_rot,
                  int num_splits, void *workspace, size_t workspace_bytes, attn_stream_t stream);
int attn_fwd_rope_f16(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int Hq, int Hkv, int Sq, int Sk, int D,
                      float scale, int mask_kind, const float *mask,
                      const float *rope_table, int max_pos, int q_pos0, int k_pos0, void *k_rot,
                      int num_splits, void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_fwd_host / attn_fwd_host_f16 — attn_fwd with Q, K, V, O, LSE and the
 * mask in HOST memory (same shapes and layouts), for callers whose tensors
 * live on the host. The pages have no counterpart: this is the copy pipeline
 * around the fused operation, not a step of it.
 * The problem is cut into units of one batch entry and a group of K/V heads
 * (with their query heads); each unit's Q, K, V are copied into one of three
 * device staging slots, the fused kernel runs on it, and its O and LSE are
 * copied back, on three streams of the library, so that the copies of
 * neighbouring units overlap the computation and each other. The additive
 * mask of each batch entry is copied once. The work starts after everything
 * already queued on `stream`, and `stream` continues only once the last copy
 * back has finished: synchronise it before reading o and lse.
 *   q, k, v, o, lse, mask  host pointers (any alignment; page-locked memory
 *               from cudaHostAlloc or cudaHostRegister lets the copies run
 *               asynchronously at full speed, pageable memory works but its
 *               copies are staged by the driver and do not overlap).
 *   workspace   device scratch of at least attn_fwd_host_workspace_bytes(...)
 *               bytes, 256-byte aligned, owned by the caller; two calls in
 *               flight on different streams need two workspaces.
 * The library creates, on first use per device, three streams and a few
 * events that it keeps until the process exits; calls from several host
 * threads are serialised while they enqueue. Other arguments and errors as
 * for attn_fwd / attn_fwd_f16; a missing, misaligned or too small workspace
 * is ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int Hq, int Hkv, int Sq, int Sk, int D,
                  float scale, int mask_kind, const float *mask,
                  void *workspace, size_t workspace_bytes, attn_stream_t stream);
int attn_fwd_host_f16(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int Hq, int Hkv, int Sq, int Sk, int D,
                      float scale, int mask_kind, const float *mask,
                      void *workspace, size_t workspace_bytes, attn_stream_t stream);

/* attn_fwd_host_workspace_bytes — device staging bytes attn_fwd_host needs
 * (host only; 0 for an empty problem or invalid sizes). */
size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int mask_kind);

/*
 * The attention block ("ATB orchestration blog"
 * (hwcomputing.csdn.net/6a15a709662f9a54cb774da1) section 2, the fused
 * attention block of the graph-operator layer and its GraphOp listing):
 *     n   = LayerNorm(x)                (eps, gain gamma, bias beta; over hidden)
 *     qkv = n W_qkv^T + b_qkv           [q | k | v] per token, (Hq + 2 Hkv) D features
 *     a   = attention(q, k, v)          fused kernel above, scale 1/sqrt(D)
 *     y   = a W_o^T + b_o + x           output projection and residual
 * bf16 tensors, FP32 accumulation and statistics; the intermediate tensors n,
 * qkv and a are bf16 in a caller workspace (each GEMM needs whole rows of its
 * input, so they pass through device memory once). Four launches: LayerNorm,
 * the QKV GEMM with its bias fused in the epilogue, the attention reading q,
 * k, v straight from the packed projection output, and the output GEMM with
 * bias and residual fused in the epilogue.
 *
 * attn_layernorm — y = (x - mean) / sqrt(var + eps) * gamma + beta for each of
 * M rows of H values (biased variance; FP32 statistics). x, y (M, H) bf16;
 * gamma, beta (H) bf16; all 16-byte aligned; H a multiple of 8, 8..8192.
 * eps not finite or <= 0 selects 1e-5. y may equal x.
 */
int attn_layernorm(const void *x, const void *gamma, const void *beta, void *y, int M, int H, float eps,
                   attn_stream_t stream);

/*
 * attn_linear — out = a w^T (+ bias) (+ residual) on the tensor cores.
 * a (M, K), w (N, K), residual and out (M, N), bias (N): bf16, row-major,
 * contiguous, 16-byte aligned; bias and residual may be NULL; out may equal
 * residual. N a positive multiple of 32, K a positive multiple of 8.
 */
int attn_linear(const void *a, const void *w, const void *bias, const void *residual, void *out,
                int M, int N, int K, attn_stream_t stream);

/*
 * attn_fwd_qkvpacked — attn_fwd (bf16, self-attention: Sq = Sk = S) with q, k,
 * v taken from one packed tensor qkv (B, S, (Hq + 2 Hkv) D): the features of
 * token (b, s) are [q heads | k heads | v heads], as a fused QKV projection
 * writes them. o (B, S, Hq, D) and lse (B, Hq, S) as for attn_fwd.
 */
int attn_fwd_qkvpacked(const void *qkv, void *o, float *lse, int B, int S, int Hq, int Hkv, int D,
                       float scale, int mask_kind, const float *mask, attn_stream_t stream);

/*
 * attn_block_fwd — the attention block on x (B, S, Hq D) bf16:
 *   ln_gamma, ln_beta (Hq D); w_qkv ((Hq + 2 Hkv) D, Hq D), b_qkv ((Hq + 2 Hkv) D);
 *   w_o (Hq D, Hq D), b_o (Hq D); y (B, S, Hq D) (may equal x). All bf16,
 *   contiguous, 16-byte aligned. causal != 0 applies the causal mask.
 *   eps as for attn_layernorm. D in {64, 128}; Hq D at most 8192.
 *   workspace: device scratch of attn_block_workspace_bytes(...) bytes,
 *   256-byte aligned (it receives n, qkv, the attention output and its LSE).
 */
int attn_block_fwd(const void *x, const void *ln_gamma, const void *ln_beta, const void *w_qkv,
                   const void *b_qkv, const void *w_o, const void *b_o, void *y,
                   int B, int S, int Hq, int Hkv, int D, float eps, int causal,
                   void *workspace, size_t workspace_bytes, attn_stream_t stream);
size_t attn_block_workspace_bytes(int B, int S, int Hq, int Hkv, int D);

/*
 * attn_last_status — synchronises `stream`, then returns and clears the
 * current device's run-time status word: ATTN_OK, or ATTN_ERR_DEVICE_TIMEOUT
 * if any launch since the last call gave up on a bounded wait (the kernel then
 * stops early, leaves its outputs incomplete and releases what it holds), or
 * ATTN_ERR_CUDA if the synchronisation itself failed.
 */
int attn_last_status(attn_stream_t stream);

/* attn_status_string — a static, human-readable name for a status code. */
const char *attn_status_string(int code);

/*
 * attn_set_wait_timeout_ns — limit, in nanoseconds, on every wait inside the
 * kernels (default 2e9 = 2 s; 0 restores the default). Applies to launches
 * made after the call, process-wide. Returns ATTN_OK.
 */
int attn_set_wait_timeout_ns(unsigned long long ns);

/*
 * attn_debug_inject_stall — failure-detection test hook. While `on` is
 * non-zero, every launch makes its MMA warp wait on a barrier that nothing
 * ever signals, so the bounded wait runs out, the kernel records
 * ATTN_ERR_DEVICE_TIMEOUT, drains its own copies in flight, frees its tensor
 * memory and returns. Nothing faults. Returns ATTN_OK.
 */
int attn_debug_inject_stall(int on);

/* attn_abi_version — version of this ABI (incremented on any change). */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TRANSFORMER_ATTENTION_02_GB300_ATTN_H */
