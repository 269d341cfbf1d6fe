"""Python binding of the C ABI declared in ``include/attn.h``.

Argument marshalling only: every step of the attention runs in the CUDA
library ``libattn.so``. There is no fallback of any kind; if the library has
not been built, or the device is not an sm_103 GPU, the calls fail loudly.

``attn_fwd`` and the other functions keep the C names and take raw device
pointers (ints); ``attention`` is the torch convenience wrapper that derives
the sizes from (B, S, H, D) tensors, allocates the outputs with PyTorch and
raises ``AttnError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

MASK_NONE, MASK_CAUSAL, MASK_ADDITIVE, MASK_CAUSAL_ADDITIVE = 0, 1, 2, 3
ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT = 0, 1, 2, 3, 4

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str = "attn_fwd"):
        self.code = code
        super().__init__(f"{what} failed: {attn_status_string(code)} ({code})")


def library_path() -> str:
    return _build.LIBRARY


def lib() -> ctypes.CDLL:
    """Load libattn.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    for f in (L.attn_fwd, L.attn_fwd_f16):
        f.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float, I, P, P]
        f.restype = I
    for f in (L.attn_fwd_splitkv, L.attn_fwd_splitkv_f16):
        f.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float, I, P, I, P, ctypes.c_size_t, P]
        f.restype = I
    for f in (L.attn_fwd_rope, L.attn_fwd_rope_f16):
        f.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float, I, P, P, I, I, I, P, I, P,
                      ctypes.c_size_t, P]
        f.restype = I
    for f in (L.attn_rope_apply, L.attn_rope_apply_f16):
        f.argtypes = [P, P, I, I, I, I, P, I, I, P]
        f.restype = I
    for f in (L.attn_fwd_host, L.attn_fwd_host_f16):
        f.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float, I, P, P, ctypes.c_size_t, P]
        f.restype = I
    L.attn_fwd_host_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    L.attn_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    L.attn_linear.argtypes = [P, P, P, P, P, I, I, I, P]
    L.attn_linear.restype = I
    L.attn_layernorm.argtypes = [P, P, P, P, I, I, ctypes.c_float, P]
    L.attn_layernorm.restype = I
    L.attn_fwd_qkvpacked.argtypes = [P, P, P, I, I, I, I, I, ctypes.c_float, I, P, P]
    L.attn_fwd_qkvpacked.restype = I
    L.attn_block_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, ctypes.c_float, I, P, ctypes.c_size_t, P]
    L.attn_block_fwd.restype = I
    L.attn_block_workspace_bytes.argtypes = [I, I, I, I, I]
    L.attn_block_workspace_bytes.restype = ctypes.c_size_t
    L.attn_rope_table.argtypes = [P, I, I, ctypes.c_double, P]
    L.attn_rope_table.restype = I
    L.attn_fwd_splitkv_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float, I, P, I, P]
    L.attn_fwd_splitkv_noalloc.restype = I
    L.attn_splitkv_num_splits.argtypes = [I, I, I, I, I, I]
    L.attn_splitkv_num_splits.restype = I
    L.attn_splitkv_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    L.attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
    L.attn_last_status.argtypes = [P]
    L.attn_last_status.restype = I
    L.attn_status_string.argtypes = [I]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
    L.attn_set_wait_timeout_ns.restype = I
    L.attn_debug_inject_stall.argtypes = [I]
    L.attn_debug_inject_stall.restype = I
    L.attn_abi_version.argtypes = []
    L.attn_abi_version.restype = I
    _lib = L
    return L


# ---------------------------------------------------------------- raw ABI

def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, stream) -> int:
    return lib().attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, stream)


def attn_fwd_f16(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, stream) -> int:
    return lib().attn_fwd_f16(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, stream)


def attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, num_splits,
                     workspace, workspace_bytes, stream) -> int:
    return lib().attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, num_splits,
                                  workspace, workspace_bytes, stream)


def attn_fwd_splitkv_f16(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, num_splits,
                         workspace, workspace_bytes, stream) -> int:
    return lib().attn_fwd_splitkv_f16(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, num_splits,
                                      workspace, workspace_bytes, stream)


def attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, num_splits,
                             stream) -> int:
    """The allocation-free split-key entry point (bf16): its scratch is the library's fixed 32 MiB array."""
    return lib().attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask,
                                          num_splits, stream)


def attn_fwd_rope(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, rope_table, max_pos, q_pos0,
                  k_pos0, k_rot, num_splits, workspace, workspace_bytes, stream) -> int:
    return lib().attn_fwd_rope(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, rope_table, max_pos,
                               q_pos0, k_pos0, k_rot, num_splits, workspace, workspace_bytes, stream)


def attn_fwd_rope_f16(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, rope_table, max_pos, q_pos0,
                      k_pos0, k_rot, num_splits, workspace, workspace_bytes, stream) -> int:
    return lib().attn_fwd_rope_f16(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, rope_table,
                                   max_pos, q_pos0, k_pos0, k_rot, num_splits, workspace, workspace_bytes, stream)


def attn_rope_table(table, max_pos, D, base, stream) -> int:
    return lib().attn_rope_table(table, max_pos, D, float(base), stream)


def attn_rope_apply(x, y, B, S, H, D, rope_table, max_pos, pos0, stream) -> int:
    return lib().attn_rope_apply(x, y, B, S, H, D, rope_table, max_pos, pos0, stream)


def attn_rope_apply_f16(x, y, B, S, H, D, rope_table, max_pos, pos0, stream) -> int:
    return lib().attn_rope_apply_f16(x, y, B, S, H, D, rope_table, max_pos, pos0, stream)


def attn_fwd_host(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, workspace, workspace_bytes,
                  stream) -> int:
    return lib().attn_fwd_host(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, workspace,
                               workspace_bytes, stream)


def attn_fwd_host_f16(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, workspace, workspace_bytes,
                      stream) -> int:
    return lib().attn_fwd_host_f16(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, mask_kind, mask, workspace,
                                   workspace_bytes, stream)


def attn_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, mask_kind) -> int:
    return int(lib().attn_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, mask_kind))


def attn_linear(a, w, bias, residual, out, M, N, K, stream) -> int:
    return lib().attn_linear(a, w, bias, residual, out, M, N, K, stream)


def attn_layernorm(x, gamma, beta, y, M, H, eps, stream) -> int:
    return lib().attn_layernorm(x, gamma, beta, y, M, H, eps, stream)


def attn_fwd_qkvpacked(qkv, o, lse, B, S, Hq, Hkv, D, scale, mask_kind, mask, stream) -> int:
    return lib().attn_fwd_qkvpacked(qkv, o, lse, B, S, Hq, Hkv, D, scale, mask_kind, mask, stream)


def attn_block_fwd(x, ln_gamma, ln_beta, w_qkv, b_qkv, w_o, b_o, y, B, S, Hq, Hkv, D, eps, causal, workspace,
                   workspace_bytes, stream) -> int:
    return lib().attn_block_fwd(x, ln_gamma, ln_beta, w_qkv, b_qkv, w_o, b_o, y, B, S, Hq, Hkv, D, eps, causal,
                                workspace, workspace_bytes, stream)


def attn_block_workspace_bytes(B, S, Hq, Hkv, D) -> int:
    return int(lib().attn_block_workspace_bytes(B, S, Hq, Hkv, D))


def attn_splitkv_num_splits(B, Hq, Hkv, Sq, Sk, num_splits=0) -> int:
    return lib().attn_splitkv_num_splits(B, Hq, Hkv, Sq, Sk, num_splits)


def attn_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, num_splits=0) -> int:
    return int(lib().attn_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, num_splits))


def attn_last_status(stream) -> int:
    return lib().attn_last_status(stream)


def attn_status_string(code: int) -> str:
    return lib().attn_status_string(int(code)).decode()


def attn_set_wait_timeout_ns(ns: int) -> int:
    return lib().attn_set_wait_timeout_ns(int(ns))


def attn_debug_inject_stall(on: bool) -> int:
    return lib().attn_debug_inject_stall(1 if on else 0)


def attn_abi_version() -> int:
    return lib().attn_abi_version()


# ------------------------------------------------------ torch convenience

def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def attention(q, k, v, *, causal: bool = False, mask=None, scale=None, out=None, lse=None, stream=None):
    """O, LSE = attention(Q, K, V) on (B, S, H, D) bf16 or fp16 CUDA tensors.

    mask: optional FP32 (B, Sq, Sk) additive mask (broadcast over heads).
    scale: None selects 1/sqrt(D). out/lse: optional preallocated outputs.
    bf16 inputs go to attn_fwd, fp16 inputs to attn_fwd_f16.
    """
    import torch
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v must be bf16 or fp16")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (t.is_cuda and t.dtype == q.dtype and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor (B, S, H, D) of q's dtype")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError("q, k, v shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    kind = (MASK_CAUSAL if causal else MASK_NONE) + (MASK_ADDITIVE if mask is not None else 0)
    mptr = None
    if mask is not None:
        if not (mask.is_cuda and mask.dtype == torch.float32 and mask.is_contiguous()
                and tuple(mask.shape) == (B, Sq, Sk)):
            raise ValueError("mask must be a contiguous FP32 CUDA tensor of shape (B, Sq, Sk)")
        mptr = mask.data_ptr()
    sc = float("nan") if scale is None else float(scale)
    fn = attn_fwd if q.dtype == torch.bfloat16 else attn_fwd_f16
    rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            B, Hq, Hkv, Sq, Sk, D, sc, kind, mptr, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc)
    return out, lse


def attention_splitkv(q, k, v, *, causal: bool = False, mask=None, scale=None, num_splits: int = 0,
                      workspace=None, out=None, lse=None, stream=None):
    """attention() with the keys split into ranges that are merged afterwards.

    workspace: optional uint8 CUDA tensor of at least attn_splitkv_workspace_bytes
    bytes (allocated here with PyTorch when omitted).
    """
    import torch
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v must be bf16 or fp16")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (t.is_cuda and t.dtype == q.dtype and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor (B, S, H, D) of q's dtype")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError("q, k, v shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    need = attn_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    kind = (MASK_CAUSAL if causal else MASK_NONE) + (MASK_ADDITIVE if mask is not None else 0)
    mptr = None
    if mask is not None:
        if not (mask.is_cuda and mask.dtype == torch.float32 and mask.is_contiguous()
                and tuple(mask.shape) == (B, Sq, Sk)):
            raise ValueError("mask must be a contiguous FP32 CUDA tensor of shape (B, Sq, Sk)")
        mptr = mask.data_ptr()
    sc = float("nan") if scale is None else float(scale)
    fn = attn_fwd_splitkv if q.dtype == torch.bfloat16 else attn_fwd_splitkv_f16
    rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, Sk, D,
            sc, kind, mptr, int(num_splits), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_splitkv")
    return out, lse


def rope_table(max_pos: int, D: int, base: float = 10000.0, *, device=None, stream=None):
    """FP32 (max_pos, D/2, 2) table of {cos, sin}(pos * base^(-2i/D)), built on the GPU."""
    import torch
    table = torch.empty((max_pos, D // 2, 2), dtype=torch.float32, device=device or "cuda")
    rc = attn_rope_table(table.data_ptr(), max_pos, D, base, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_rope_table")
    return table


def rope_apply(x, table, *, pos0: int = 0, out=None, stream=None):
    """Rotate every head vector of a (B, S, H, D) bf16/fp16 CUDA tensor (row s at
    position pos0 + s) into `out` (new tensor by default; may be x itself)."""
    import torch
    if x.dtype not in (torch.bfloat16, torch.float16) or not (x.is_cuda and x.dim() == 4 and x.is_contiguous()):
        raise ValueError("x must be a contiguous 4-D bf16/fp16 CUDA tensor (B, S, H, D)")
    if out is None:
        out = torch.empty_like(x)
    B, S, H, D = x.shape
    fn = attn_rope_apply if x.dtype == torch.bfloat16 else attn_rope_apply_f16
    rc = fn(x.data_ptr(), out.data_ptr(), B, S, H, D, table.data_ptr(), table.shape[0], int(pos0),
            _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_rope_apply")
    return out


def attention_rope(q, k, v, table, *, q_pos0: int = 0, k_pos0: int = 0, k_rot="new", causal: bool = False,
                   mask=None, scale=None, num_splits: int = 1, workspace=None, out=None, lse=None, stream=None):
    """attention(rot(Q), rot(K), V) with the rotary table of rope_table().

    Q is rotated inside the attention kernel at tile load. k_rot: "new" (a
    tensor allocated here receives the rotated keys), a tensor of k's shape
    (may be k itself: rotated in place), or None (k already holds rotated
    keys). num_splits / workspace as for attention_splitkv (1: no split).
    Returns (out, lse) or, when the keys were rotated here, (out, lse, k_rot).
    """
    import torch
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v must be bf16 or fp16")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (t.is_cuda and t.dtype == q.dtype and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor (B, S, H, D) of q's dtype")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError("q, k, v shapes disagree")
    if not (table.is_cuda and table.dtype == torch.float32 and table.dim() == 3 and table.shape[1:] == (D // 2, 2)
            and table.is_contiguous()):
        raise ValueError("table must be the (max_pos, D/2, 2) FP32 CUDA tensor of rope_table() for this D")
    if isinstance(k_rot, str):
        if k_rot != "new":
            raise ValueError("k_rot must be 'new', a tensor of k's shape, or None")
        k_rot = torch.empty_like(k)
    if k_rot is not None and not (k_rot.is_cuda and k_rot.dtype == k.dtype and k_rot.shape == k.shape
                                  and k_rot.is_contiguous()):
        raise ValueError("k_rot must be a contiguous CUDA tensor of k's shape and dtype")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    need = attn_splitkv_workspace_bytes(B, Hq, Hq, Sq, Sk, D, num_splits)    # rotary tiles never pack heads
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    kind = (MASK_CAUSAL if causal else MASK_NONE) + (MASK_ADDITIVE if mask is not None else 0)
    mptr = None
    if mask is not None:
        if not (mask.is_cuda and mask.dtype == torch.float32 and mask.is_contiguous()
                and tuple(mask.shape) == (B, Sq, Sk)):
            raise ValueError("mask must be a contiguous FP32 CUDA tensor of shape (B, Sq, Sk)")
        mptr = mask.data_ptr()
    sc = float("nan") if scale is None else float(scale)
    fn = attn_fwd_rope if q.dtype == torch.bfloat16 else attn_fwd_rope_f16
    rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, Sk, D,
            sc, kind, mptr, table.data_ptr(), table.shape[0], int(q_pos0), int(k_pos0),
            None if k_rot is None else k_rot.data_ptr(), int(num_splits),
            None if workspace is None else workspace.data_ptr(),
            0 if workspace is None else workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_rope")
    return (out, lse) if k_rot is None else (out, lse, k_rot)


def attention_host(q, k, v, *, causal: bool = False, mask=None, scale=None, out=None, lse=None, workspace=None,
                   device=None, stream=None):
    """attention() for (B, S, H, D) bf16/fp16 tensors in host memory (pin them
    for full speed): copies in, computes and copies back in a pipeline on the
    GPU. Returns (out, lse) in host memory, written once `stream` (default: the
    current stream of `device`) has been synchronised; this function does not
    synchronise. workspace: optional uint8 CUDA tensor of at least
    attn_fwd_host_workspace_bytes bytes (allocated here when omitted).
    """
    import torch
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v must be bf16 or fp16")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not (t.device.type == "cpu" and t.dtype == q.dtype and t.dim() == 4 and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D host tensor (B, S, H, D) of q's dtype")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError("q, k, v shapes disagree")
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, pin_memory=pin)
    kind = (MASK_CAUSAL if causal else MASK_NONE) + (MASK_ADDITIVE if mask is not None else 0)
    mptr = None
    if mask is not None:
        if not (mask.device.type == "cpu" and mask.dtype == torch.float32 and mask.is_contiguous()
                and tuple(mask.shape) == (B, Sq, Sk)):
            raise ValueError("mask must be a contiguous FP32 host tensor of shape (B, Sq, Sk)")
        mptr = mask.data_ptr()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    need = attn_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, kind)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    sc = float("nan") if scale is None else float(scale)
    fn = attn_fwd_host if q.dtype == torch.bfloat16 else attn_fwd_host_f16
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, Sk, D, sc,
                kind, mptr, workspace.data_ptr(), workspace.numel() * workspace.element_size(), s.cuda_stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")
    return out, lse


def _bf16_cuda(name, t, dim=None):
    import torch
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and (dim is None or t.dim() == dim)):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor" + (f" with {dim} dimensions" if dim else ""))


def linear(a, w, bias=None, residual=None, *, out=None, stream=None):
    """out = a w^T (+ bias) (+ residual) for bf16 CUDA tensors a (M, K), w (N, K)."""
    import torch
    _bf16_cuda("a", a, 2)
    _bf16_cuda("w", w, 2)
    M, K = a.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("a and w disagree on K")
    for name, t, shape in (("bias", bias, (N,)), ("residual", residual, (M, N))):
        if t is not None:
            _bf16_cuda(name, t)
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} must have shape {shape}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    rc = attn_linear(a.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(),
                     None if residual is None else residual.data_ptr(), out.data_ptr(), M, N, K, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_linear")
    return out


def layernorm(x, gamma, beta, eps: float = 1e-5, *, out=None, stream=None):
    """Row-wise LayerNorm over the last dimension of a bf16 CUDA tensor."""
    import torch
    for name, t in (("x", x), ("gamma", gamma), ("beta", beta)):
        _bf16_cuda(name, t)
    H = x.shape[-1]
    M = x.numel() // H if H else 0
    if out is None:
        out = torch.empty_like(x)
    rc = attn_layernorm(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), out.data_ptr(), M, H, float(eps),
                        _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_layernorm")
    return out


def attention_qkvpacked(qkv, Hq: int, Hkv: int, D: int, *, causal: bool = False, scale=None, out=None, lse=None,
                        stream=None):
    """Self-attention on a packed (B, S, (Hq + 2 Hkv) D) bf16 tensor [q | k | v]."""
    import torch
    _bf16_cuda("qkv", qkv, 3)
    B, S, F = qkv.shape
    if F != (Hq + 2 * Hkv) * D:
        raise ValueError("qkv's last dimension must be (Hq + 2 Hkv) D")
    if out is None:
        out = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=qkv.device)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=qkv.device)
    sc = float("nan") if scale is None else float(scale)
    rc = attn_fwd_qkvpacked(qkv.data_ptr(), out.data_ptr(), lse.data_ptr(), B, S, Hq, Hkv, D, sc,
                            MASK_CAUSAL if causal else MASK_NONE, None, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_qkvpacked")
    return out, lse


def attention_block(x, ln_gamma, ln_beta, w_qkv, b_qkv, w_o, b_o, *, Hq: int, Hkv: int, D: int,
                    causal: bool = True, eps: float = 1e-5, out=None, workspace=None, stream=None):
    """The attention block (LayerNorm, QKV projection, attention, output
    projection, residual) on x (B, S, Hq*D) bf16 CUDA; returns y."""
    import torch
    for name, t in (("x", x), ("ln_gamma", ln_gamma), ("ln_beta", ln_beta), ("w_qkv", w_qkv), ("b_qkv", b_qkv),
                    ("w_o", w_o), ("b_o", b_o)):
        _bf16_cuda(name, t)
    B, S, H = x.shape
    F = (Hq + 2 * Hkv) * D
    if H != Hq * D or tuple(w_qkv.shape) != (F, H) or tuple(b_qkv.shape) != (F,) or tuple(w_o.shape) != (H, H) \
            or tuple(b_o.shape) != (H,) or tuple(ln_gamma.shape) != (H,) or tuple(ln_beta.shape) != (H,):
        raise ValueError("attention block shapes disagree")
    if out is None:
        out = torch.empty_like(x)
    need = attn_block_workspace_bytes(B, S, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    rc = attn_block_fwd(x.data_ptr(), ln_gamma.data_ptr(), ln_beta.data_ptr(), w_qkv.data_ptr(), b_qkv.data_ptr(),
                        w_o.data_ptr(), b_o.data_ptr(), out.data_ptr(), B, S, Hq, Hkv, D, float(eps),
                        1 if causal else 0, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_block_fwd")
    return out
