"""usp_attn_bwd_noalloc: the backward for callers that cannot allocate
device memory when they call it (their allocator reserved it up front, or
their policy forbids allocation after start-up).  Its scratch is a fixed
device array inside the library instead of a caller-provided workspace.  It
runs the same deterministic kernels on the same inputs as usp_attn_bwd, so
its gradients must be bitwise equal to usp_attn_bwd's -- on every call, since
the array keeps the previous call's contents.  This file is collected last
so that a failure here does not hide the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from ulysses_sequence_attention_usp_gb300 import binding as B

FAKE = 1 << 20   # aligned address; the rejected call never dereferences it
LIMIT = 32 << 20


def test_rejects_problem_larger_than_fixed_scratch():
    # 8 ranks x 8 heads x 131072 rows x 2 arrays x 4 B = 64 MiB > 32 MiB
    d = B.make_dims(131072, 8, 64, 8, 128)
    st = B.raw_call("usp_attn_bwd_noalloc", ctypes.byref(d), *([FAKE] * 11))
    assert st == 3                     # USP_ERR_UNSUPPORTED, nothing launched
    d = B.make_dims(131072, 8, 64, 7, 128)
    assert B.raw_call("usp_attn_bwd_noalloc", ctypes.byref(d), *([FAKE] * 11)) == 2


def test_limit_is_exact():
    # 1024 query heads x 4096 rows x 2 arrays x 4 B is exactly the 32 MiB
    # array; one more 128-row tile of workspace rows is refused on the host
    d = B.make_dims(4096, 8, 1024, 8, 64)
    assert B.usp_attn_bwd_workspace(d) == LIMIT
    d = B.make_dims(4096 + 128, 8, 1024, 8, 64)
    assert B.usp_attn_bwd_workspace(d) == LIMIT + 1024 * 128 * 2 * 4
    assert B.raw_call("usp_attn_bwd_noalloc", ctypes.byref(d), *([FAKE] * 11)) == 3


def _problem(S, P, Hq, Hkv, D, cu_host=None, seed=0):
    torch.manual_seed(seed)
    cu = None if cu_host is None else torch.from_numpy(cu_host).cuda()
    d = B.make_dims(S, P, Hq, Hkv, D, cu, cu_host)
    hq, hkv = Hq // P, Hkv // P
    bf = dict(dtype=torch.bfloat16, device="cuda")
    q = torch.randn(P, S, hq, D, **bf)
    k = torch.randn(P, S, hkv, D, **bf)
    v = torch.randn(P, S, hkv, D, **bf)
    do = torch.randn(P, S, hq, D, **bf)
    pos = torch.empty(S, dtype=torch.int32, device="cuda")
    doc = torch.empty_like(pos)
    B.usp_pad_shard(d, None, 0, None, pos, doc)
    o = torch.empty_like(q)
    lse = torch.empty(P, hq, S, dtype=torch.float32, device="cuda")
    B.usp_attn_fwd(d, q, k, v, doc, o, lse)
    n = B.usp_attn_bwd_workspace(d)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    B.usp_attn_bwd(d, q, k, v, o, lse, do, doc, *ref, ws, n)
    B.usp_device_status()
    return d, (q, k, v, o, lse, do, doc), ref


def _check_bitwise(d, args, ref):
    for _ in range(2):                 # two calls in a row share the scratch
        got = [torch.full_like(t, 7.0) for t in ref]
        B.usp_attn_bwd_noalloc(d, *args, *got)
        B.usp_device_status()
        for a, b in zip(got, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward():
    S, P, Hq, Hkv, D = 3000, 2, 8, 2, 128
    cu_host = np.array([0, 700, 701, 2100, 3000], np.int32)
    d, args, ref = _problem(S, P, Hq, Hkv, D, cu_host)
    _check_bitwise(d, args, ref)


@pytest.mark.gpu
def test_noalloc_backward_at_the_scratch_limit():
    # the workspace of this problem fills the whole fixed array, so the
    # second vector (LSE*log2(e)) ends exactly at the array's last byte
    d, args, ref = _problem(4096, 8, 1024, 8, 64, seed=1)
    assert B.usp_attn_bwd_workspace(d) == LIMIT
    _check_bitwise(d, args, ref)
