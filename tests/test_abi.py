"""The C-ABI library builds, loads and exports every symbol include/attn.h
declares; argument checks that happen on the host before any CUDA call are
exercised without a GPU (fake, never-dereferenced pointer values)."""
import os
import re
import subprocess

import pytest

from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

P = 0x10000          # a 16-byte aligned stand-in address: validation fails before any use


@pytest.fixture(scope="module")
def lib():
    B.build()
    return A.lib()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = declared_functions()
    assert {"attn_fwd", "attn_last_status", "attn_status_string"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", A.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, f"{name} is declared in attn.h but not exported"
        getattr(lib, name)


def test_abi_version(lib):
    assert A.attn_abi_version() >= 1


def test_status_strings(lib):
    assert A.attn_status_string(0) == "ATTN_OK"
    assert A.attn_status_string(1) == "ATTN_ERR_INVALID_ARG"
    assert A.attn_status_string(2) == "ATTN_ERR_UNSUPPORTED"
    assert A.attn_status_string(3) == "ATTN_ERR_CUDA"
    assert A.attn_status_string(4) == "ATTN_ERR_DEVICE_TIMEOUT"
    assert A.attn_status_string(99) == "ATTN_UNKNOWN_STATUS"


def _call(q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=2, Sq=16, Sk=16, D=64, scale=0.0, kind=0, mask=None):
    return A.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, kind, mask, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), A.ATTN_ERR_INVALID_ARG),
    (dict(k=None), A.ATTN_ERR_INVALID_ARG),
    (dict(v=None), A.ATTN_ERR_INVALID_ARG),
    (dict(o=None), A.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), A.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), A.ATTN_ERR_INVALID_ARG),
    (dict(Sq=-3), A.ATTN_ERR_INVALID_ARG),
    (dict(Sk=-3), A.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), A.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=4), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=-1), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=2, mask=None), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=3, mask=None), A.ATTN_ERR_INVALID_ARG),
    (dict(q=P + 8), A.ATTN_ERR_INVALID_ARG),            # not 16-byte aligned
    (dict(o=P + 2), A.ATTN_ERR_INVALID_ARG),
    (dict(lse=P + 2), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=2, mask=P + 1), A.ATTN_ERR_INVALID_ARG),
    (dict(D=96), A.ATTN_ERR_UNSUPPORTED),                # head dim must be 64 or 128
    (dict(D=32), A.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), A.ATTN_ERR_UNSUPPORTED),
    (dict(Sq=(1 << 30) + 1), A.ATTN_ERR_INVALID_ARG),
])
def test_invalid_arguments_are_rejected_before_launch(lib, kw, code):
    assert _call(**kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(Hq=0), dict(Sq=0)])
def test_empty_problem_is_a_no_op(lib, kw):
    # nothing to compute: success without touching the device (no GPU here)
    assert _call(**kw) == A.ATTN_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(A, "_lib", None)
    monkeypatch.setattr(A, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        A.lib()


# ------------------------------------------------------------ split keys (host only)

def test_splitkv_range_count_and_workspace_size(lib):
    # automatic choice without a GPU (148 SMs assumed): fill one wave of tiles
    assert A.attn_splitkv_num_splits(1, 16, 16, 1, 8192, 0) == 8      # 16 tiles: 9 wanted, 64 blocks -> 8 x 8
    assert A.attn_splitkv_num_splits(4, 32, 32, 1, 4096, 0) == 1      # 128 tiles already: no split
    # GQA decode packs the 4 query heads of each K/V head into one tile: 4 x 8 = 32
    # tiles, so 4 ranges fill the SMs (148 // 32 = 4) instead of none
    assert A.attn_splitkv_num_splits(4, 32, 8, 1, 4096, 0) == 4
    # no packing for a group that is not a power of two, or too many query rows
    assert A.attn_splitkv_num_splits(1, 32, 8, 1, 4096, 0) == 16     # 8 packed tiles: 18 wanted -> 16 x 2 blocks
    assert A.attn_splitkv_num_splits(1, 32, 32, 1, 4096, 0) == 4     # MHA: 32 tiles -> 4 ranges
    assert A.attn_splitkv_num_splits(4, 24, 8, 1, 4096, 0) == 1      # group of 3: 96 unpacked tiles
    assert A.attn_splitkv_num_splits(1, 32, 8, 100, 4096, 0) == 4    # 100 x 4 rows > 256: unpacked, 32 tiles
    # explicit counts are capped by the number of 128-key blocks and made even-sized
    assert A.attn_splitkv_num_splits(1, 8, 8, 1, 1000, 3) == 3       # 8 blocks -> 3+3+2
    assert A.attn_splitkv_num_splits(1, 8, 8, 1, 1000, 100) == 8
    assert A.attn_splitkv_num_splits(1, 8, 8, 1, 1000, 5) == 4       # 2 blocks per range
    assert A.attn_splitkv_num_splits(1, 8, 8, 1, 0, 4) == 1          # no keys, no split
    # a prefill with plenty of tiles is not split and needs no workspace
    assert A.attn_splitkv_num_splits(4, 32, 32, 2048, 2048, 0) == 1
    assert A.attn_splitkv_workspace_bytes(4, 32, 32, 2048, 2048, 128, 0) == 0
    # workspace = FP32 O of every range, then (256-byte aligned) FP32 LSE of every range
    rows = 4 * 32 * 1
    o_bytes = 2 * rows * 128 * 4
    assert A.attn_splitkv_workspace_bytes(4, 32, 32, 1, 4096, 128, 2) == ((o_bytes + 255) // 256) * 256 + 2 * rows * 4
    assert A.attn_splitkv_workspace_bytes(4, 32, 32, 1, 4096, 96, 2) == 0   # unsupported head dim
    assert A.attn_splitkv_num_splits(-1, 32, 32, 1, 4096, 0) == 0
    assert A.attn_splitkv_num_splits(1, 32, 0, 1, 4096, 0) == 0


def _call_split(num_splits=4, ws=P, ws_bytes=1 << 30, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=2, Sq=16, Sk=4096, D=64, scale=0.0, kind=0, mask=None)
    a.update(kw)
    return A.attn_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Sq"],
                              a["Sk"], a["D"], a["scale"], a["kind"], a["mask"], num_splits, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(num_splits=-1), A.ATTN_ERR_INVALID_ARG),
    (dict(ws=None), A.ATTN_ERR_INVALID_ARG),                 # a split needs a workspace
    (dict(ws=P + 128), A.ATTN_ERR_INVALID_ARG),              # not 256-byte aligned
    (dict(ws_bytes=64), A.ATTN_ERR_INVALID_ARG),             # too small
    (dict(D=80), A.ATTN_ERR_UNSUPPORTED),
    (dict(B=0), A.ATTN_OK),                                  # empty: nothing to do, no workspace needed
])
def test_splitkv_arguments_are_checked_before_launch(lib, kw, code):
    assert _call_split(**kw) == code


# ------------------------------------------------------- rotary embedding (host only)

def _call_rope(table=P, max_pos=4096, q_pos0=0, k_pos0=0, k_rot=P, num_splits=1, ws=None, ws_bytes=0, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=2, Sq=16, Sk=64, D=128, scale=0.0, kind=1, mask=None)
    a.update(kw)
    return A.attn_fwd_rope(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"],
                           a["D"], a["scale"], a["kind"], a["mask"], table, max_pos, q_pos0, k_pos0, k_rot,
                           num_splits, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(table=None), A.ATTN_ERR_INVALID_ARG),
    (dict(table=P + 8), A.ATTN_ERR_INVALID_ARG),             # table must be 16-byte aligned
    (dict(max_pos=0), A.ATTN_ERR_INVALID_ARG),
    (dict(q_pos0=-1), A.ATTN_ERR_INVALID_ARG),
    (dict(max_pos=20, q_pos0=5), A.ATTN_ERR_INVALID_ARG),    # query rows 5..20 past the table
    (dict(max_pos=64, k_pos0=1), A.ATTN_ERR_INVALID_ARG),    # keys 1..64 past the table
    (dict(k_pos0=-2), A.ATTN_ERR_INVALID_ARG),
    (dict(k_rot=P + 4), A.ATTN_ERR_INVALID_ARG),
    (dict(num_splits=4, Sk=4096), A.ATTN_ERR_INVALID_ARG),   # a split needs a workspace
    (dict(D=96), A.ATTN_ERR_UNSUPPORTED),
    (dict(B=0), A.ATTN_OK),                                  # empty: nothing to do
])
def test_rope_arguments_are_checked_before_launch(lib, kw, code):
    assert _call_rope(**kw) == code


def test_rope_without_key_rotation_ignores_the_key_positions(lib):
    # k_rot NULL: the keys are taken as already rotated and k_pos0 is not
    # checked, so validation passes and the call gets as far as the device
    # query (ATTN_ERR_CUDA without a GPU, not ATTN_ERR_INVALID_ARG)
    assert _call_rope(k_rot=None, k_pos0=-5, max_pos=64) != A.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("args,code", [
    ((P, 4096, 127, 10000.0), A.ATTN_ERR_INVALID_ARG),       # odd D
    ((P, 4096, 128, 1.0), A.ATTN_ERR_INVALID_ARG),           # base must exceed 1
    ((P, 4096, 128, float("inf")), A.ATTN_ERR_INVALID_ARG),
    ((P, -1, 128, 10000.0), A.ATTN_ERR_INVALID_ARG),
    ((P + 4, 4096, 128, 10000.0), A.ATTN_ERR_INVALID_ARG),   # misaligned
    ((None, 4096, 128, 10000.0), A.ATTN_ERR_INVALID_ARG),
    ((P, 1 << 24, 256, 10000.0), A.ATTN_ERR_INVALID_ARG),    # more than 2^31 entries
    ((None, 0, 128, 10000.0), A.ATTN_OK),                     # empty table: nothing to do
])
def test_rope_table_arguments(lib, args, code):
    assert A.attn_rope_table(*args, None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(D=100), A.ATTN_ERR_INVALID_ARG),                   # D must be a multiple of 8
    (dict(pos0=-1), A.ATTN_ERR_INVALID_ARG),
    (dict(S=100, max_pos=99), A.ATTN_ERR_INVALID_ARG),
    (dict(x=P + 2), A.ATTN_ERR_INVALID_ARG),
    (dict(y=None), A.ATTN_ERR_INVALID_ARG),
    (dict(table=P + 8), A.ATTN_ERR_INVALID_ARG),
    (dict(B=0), A.ATTN_OK),
    (dict(S=0, pos0=4096), A.ATTN_OK),
])
def test_rope_apply_arguments(lib, kw, code):
    a = dict(x=P, y=P, B=2, S=64, H=4, D=128, table=P, max_pos=4096, pos0=0)
    a.update(kw)
    for fn in (A.attn_rope_apply, A.attn_rope_apply_f16):
        assert fn(a["x"], a["y"], a["B"], a["S"], a["H"], a["D"], a["table"], a["max_pos"], a["pos0"], None) == code


# ------------------------------------------------------ host-buffer pipeline (host only)

def test_host_pipeline_workspace_size(lib):
    # Llama-2-7B shape: 4 entries x 2 groups of 16 heads = 8 units, three slots of
    # Q + K + V + O (8 MiB each) + LSE (16 x 2048 FP32)
    per_slot = 4 * (2048 * 16 * 128 * 2) + 16 * 2048 * 4
    assert A.attn_fwd_host_workspace_bytes(4, 32, 32, 2048, 2048, 128, 1) == 3 * per_slot
    # an additive mask adds B x Sq x Sk FP32, staged once
    assert A.attn_fwd_host_workspace_bytes(4, 32, 32, 2048, 2048, 128, 3) == 3 * per_slot + 4 * 2048 * 2048 * 4
    assert A.attn_fwd_host_workspace_bytes(0, 32, 32, 2048, 2048, 128, 1) == 0
    assert A.attn_fwd_host_workspace_bytes(4, 32, 32, 2048, 2048, 96, 1) == 0


def _call_host(ws=P, ws_bytes=1 << 34, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=2, Hq=4, Hkv=2, Sq=64, Sk=64, D=128, scale=0.0, kind=1, mask=None)
    a.update(kw)
    return A.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"],
                           a["D"], a["scale"], a["kind"], a["mask"], ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ws=None), A.ATTN_ERR_INVALID_ARG),
    (dict(ws=P + 64), A.ATTN_ERR_INVALID_ARG),                # not 256-byte aligned
    (dict(ws_bytes=1024), A.ATTN_ERR_INVALID_ARG),
    (dict(q=None), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=2, mask=None), A.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=5), A.ATTN_ERR_INVALID_ARG),
    (dict(D=96), A.ATTN_ERR_UNSUPPORTED),
    (dict(B=0), A.ATTN_OK),
    (dict(Sq=0), A.ATTN_OK),
])
def test_host_pipeline_arguments_are_checked_before_launch(lib, kw, code):
    assert _call_host(**kw) == code


# ------------------------------------------------------------ attention block (host only)

@pytest.mark.parametrize("kw,code", [
    (dict(N=48), A.ATTN_ERR_INVALID_ARG),                    # N must be a multiple of 32
    (dict(K=12), A.ATTN_ERR_INVALID_ARG),                    # K a multiple of 8
    (dict(N=0), A.ATTN_ERR_INVALID_ARG),
    (dict(M=-1), A.ATTN_ERR_INVALID_ARG),
    (dict(a=None), A.ATTN_ERR_INVALID_ARG),
    (dict(w=P + 8), A.ATTN_ERR_INVALID_ARG),
    (dict(bias=P + 2), A.ATTN_ERR_INVALID_ARG),
    (dict(M=0), A.ATTN_OK),
])
def test_linear_arguments(lib, kw, code):
    a = dict(a=P, w=P, bias=None, residual=None, out=P, M=64, N=64, K=64)
    a.update(kw)
    assert A.attn_linear(a["a"], a["w"], a["bias"], a["residual"], a["out"], a["M"], a["N"], a["K"], None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(H=12), A.ATTN_ERR_INVALID_ARG),
    (dict(H=8200), A.ATTN_ERR_INVALID_ARG),
    (dict(gamma=None), A.ATTN_ERR_INVALID_ARG),
    (dict(y=P + 4), A.ATTN_ERR_INVALID_ARG),
    (dict(M=0), A.ATTN_OK),
])
def test_layernorm_arguments(lib, kw, code):
    a = dict(x=P, gamma=P, beta=P, y=P, M=8, H=256)
    a.update(kw)
    assert A.attn_layernorm(a["x"], a["gamma"], a["beta"], a["y"], a["M"], a["H"], 1e-5, None) == code


def test_block_workspace_layout(lib):
    # n (M x H), packed qkv (M x 3H), attention output (M x H) in bf16, then FP32 LSE
    B, S, Hq, D = 4, 2048, 32, 128
    M, H = B * S, Hq * D
    assert A.attn_block_workspace_bytes(B, S, Hq, Hq, D) == (M * H + M * 3 * H + M * H) * 2 + B * Hq * S * 4
    assert A.attn_block_workspace_bytes(B, S, Hq, 8, D) == (M * H + M * (Hq + 16) * D + M * H) * 2 + B * Hq * S * 4
    assert A.attn_block_workspace_bytes(1, 16, 4, 4, 96) == 0          # head dimension
    assert A.attn_block_workspace_bytes(1, 16, 128, 128, 128) == 0     # hidden above 8192


@pytest.mark.parametrize("kw,code", [
    (dict(ws=None), A.ATTN_ERR_INVALID_ARG),
    (dict(ws_bytes=100), A.ATTN_ERR_INVALID_ARG),
    (dict(D=96), A.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=3, Hkv=2), A.ATTN_ERR_INVALID_ARG),
    (dict(b_qkv=None), A.ATTN_ERR_INVALID_ARG),
    (dict(x=P + 8), A.ATTN_ERR_INVALID_ARG),
    (dict(B=0), A.ATTN_OK),
])
def test_block_arguments(lib, kw, code):
    a = dict(x=P, g=P, b=P, w_qkv=P, b_qkv=P, w_o=P, b_o=P, y=P, B=1, S=64, Hq=4, Hkv=4, D=64, ws=P, ws_bytes=1 << 30)
    a.update(kw)
    assert A.attn_block_fwd(a["x"], a["g"], a["b"], a["w_qkv"], a["b_qkv"], a["w_o"], a["b_o"], a["y"], a["B"], a["S"],
                            a["Hq"], a["Hkv"], a["D"], 1e-5, 1, a["ws"], a["ws_bytes"], None) == code


def _noalloc(q=P, k=P, v=P, o=P, lse=P, B=4, Hq=32, Hkv=32, Sq=2048, Sk=2048, D=128, kind=1, mask=None,
             splits=4):
    return A.attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, 0.0, kind, mask, splits, None)


@pytest.mark.parametrize("kw,code", [
    # Invalid arguments on a problem too large for the scratch array are still
    # reported as invalid (the same checks as attn_fwd_splitkv run first).
    (dict(Hq=33, Hkv=2), A.ATTN_ERR_INVALID_ARG),
    (dict(q=None), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=5), A.ATTN_ERR_INVALID_ARG),
    (dict(kind=2, mask=None), A.ATTN_ERR_INVALID_ARG),
    (dict(o=P + 4), A.ATTN_ERR_INVALID_ARG),
    (dict(splits=-1), A.ATTN_ERR_INVALID_ARG),
    (dict(D=80), A.ATTN_ERR_UNSUPPORTED),
    # Valid arguments whose partial results exceed the 32 MiB array.
    (dict(), A.ATTN_ERR_UNSUPPORTED),
])
def test_noalloc_checks_arguments_before_the_scratch_limit(lib, kw, code):
    assert _noalloc(**kw) == code
