"""Failure detection on the GPU without a GPU fault: a bounded device-side
wait that nothing completes gives up, the status word reports a timeout,
and the context keeps working (the attention kernels use the same wait)."""
import numpy as np
import pytest
import torch

from ulysses_sequence_attention_usp_gb300 import binding as B

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    B.usp_device_status()                       # start from a clear status word
    B.usp_selftest_bounded_wait(20000)          # 20 ms limit
    with pytest.raises(B.UspError) as e:
        B.usp_device_status()
    assert e.value.status == 5                  # USP_ERR_TIMEOUT
    B.usp_device_status()                       # reported once, then cleared
    # the context is still usable: a small forward runs and its status is OK
    S, P, Hq, Hkv, D = 300, 2, 4, 2, 64
    d = B.make_dims(S, P, Hq, Hkv, D)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    q = torch.randn(P, S, Hq // P, D, **bf)
    k = torch.randn(P, S, Hkv // P, D, **bf)
    v = torch.randn(P, S, Hkv // P, D, **bf)
    pos = torch.empty(S, dtype=torch.int32, device="cuda")
    doc = torch.empty_like(pos)
    B.usp_pad_shard(d, None, 0, None, pos, doc)
    o = torch.empty_like(q)
    lse = torch.empty(P, Hq // P, S, dtype=torch.float32, device="cuda")
    B.usp_attn_fwd(d, q, k, v, doc, o, lse)
    B.usp_device_status()
    assert torch.isfinite(o.float()).all()
