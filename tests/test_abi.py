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
    assert A.attn_splitkv_num_splits(1, 16, 1, 8192, 0) == 8      # 16 tiles: 9 wanted, 64 blocks -> 8 x 8
    assert A.attn_splitkv_num_splits(4, 32, 1, 4096, 0) == 1      # 128 tiles already: no split
    # explicit counts are capped by the number of 128-key blocks and made even-sized
    assert A.attn_splitkv_num_splits(1, 8, 1, 1000, 3) == 3       # 8 blocks -> 3+3+2
    assert A.attn_splitkv_num_splits(1, 8, 1, 1000, 100) == 8
    assert A.attn_splitkv_num_splits(1, 8, 1, 1000, 5) == 4       # 2 blocks per range
    assert A.attn_splitkv_num_splits(1, 8, 1, 0, 4) == 1          # no keys, no split
    # a prefill with plenty of tiles is not split and needs no workspace
    assert A.attn_splitkv_num_splits(4, 32, 2048, 2048, 0) == 1
    assert A.attn_splitkv_workspace_bytes(4, 32, 2048, 2048, 128, 0) == 0
    # workspace = FP32 O of every range, then (256-byte aligned) FP32 LSE of every range
    rows = 4 * 32 * 1
    o_bytes = 2 * rows * 128 * 4
    assert A.attn_splitkv_workspace_bytes(4, 32, 1, 4096, 128, 2) == ((o_bytes + 255) // 256) * 256 + 2 * rows * 4
    assert A.attn_splitkv_workspace_bytes(4, 32, 1, 4096, 96, 2) == 0   # unsupported head dim
    assert A.attn_splitkv_num_splits(-1, 32, 1, 4096, 0) == 0


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
