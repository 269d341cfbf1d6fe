"""Failure detection without a GPU fault: every wait inside the kernel is
bounded. The test hook makes the MMA warp wait on a barrier nothing signals;
with a 50 ms limit the kernel must give up, report ATTN_ERR_DEVICE_TIMEOUT
through attn_last_status, release what it holds, and leave the context usable
for the next (correct) call. Nothing traps, faults or hangs."""
import pytest
import torch

from gpu_helpers import check
from transformer_attention_02_gb300 import attn as A
from transformer_attention_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    cfg = I.AttnConfig("t", 2, 4, 2, 512, 512, 128, causal=True, seed=7)
    q, k, v, _ = I.make_inputs(cfg)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert A.attn_last_status(stream) == A.ATTN_OK            # start clean
    A.attn_set_wait_timeout_ns(50_000_000)
    A.attn_debug_inject_stall(True)
    try:
        A.attention(qd, kd, vd, causal=True)                  # enqueued fine
        assert A.attn_last_status(stream) == A.ATTN_ERR_DEVICE_TIMEOUT
    finally:
        A.attn_debug_inject_stall(False)
        A.attn_set_wait_timeout_ns(0)
    assert A.attn_last_status(stream) == A.ATTN_OK            # the status word was cleared
    o, lse = A.attention(qd, kd, vd, causal=True)
    assert A.attn_last_status(stream) == A.ATTN_OK
    check(o, lse, q, k, v, None, cfg.mask_kind, label="after timeout")
