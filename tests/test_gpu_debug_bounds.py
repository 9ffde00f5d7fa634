"""The library built with index guards (build(debug=True)): every global
index a kernel computes is checked against the extent usp_dims implies for
its buffer, and an out-of-range one sets a status bit (USP_ERR_OUT_OF_BOUNDS)
instead of being read or written.  With compute-sanitizer closed on this
pool, this build is the bounds check of the small parity cases.

The guarded library is loaded in a child process (USP_DEBUG_BOUNDS=1), which
runs the small-case GPU parity tests; each of them reads the device status
word after its launches, so a pass means that no guard fired."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SMALL_CASES = [
    "tests/test_gpu_attention.py::test_attention_kernels_vs_fp64",
    "tests/test_gpu_attention.py::test_pipeline_vs_full_sequence",
    "tests/test_gpu_repack.py::test_pad_shard_positions_docs",
    "tests/test_gpu_repack.py::test_seq_to_head_tiny",
    "tests/test_gpu_repack.py::test_seq_to_head_small_ragged",
    "tests/test_gpu_repack.py::test_seq_to_head_reads_unpadded_source",
    "tests/test_gpu_repack.py::test_head_to_seq_bit_exact",
    "tests/test_gpu_bidirectional.py",
    "tests/test_gpu_ring.py",
    "tests/test_gpu_zigzag.py",
    "tests/test_gpu_allgather.py::test_allgather_step_vs_oracle",
    "tests/test_gpu_debug_bounds.py::test_guard_reports_out_of_range_document_id",
]


# larger grids under the guards: the 8K pipeline (forward, both backward
# passes, every permutation) and the 120K permutations on sampled rows,
# including rows past the grid-stride threshold
LARGE_CASES = [
    "tests/test_gpu_attention.py::test_full_workload_sampled[qwen8k]",
    "tests/test_gpu_repack.py::test_seq_to_head_120k_yarn_sampled_rows",
    "tests/test_gpu_repack.py::test_head_to_seq_120k_sampled_rows",
]


def _child(args, timeout=1200):
    env = dict(os.environ, USP_DEBUG_BOUNDS="1")
    return subprocess.run([sys.executable] + args, cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=timeout)


def test_small_parity_cases_run_clean_under_index_guards():
    from ulysses_sequence_attention_usp_gb300 import build
    build.build(debug=True)
    r = _child(["-c", "from ulysses_sequence_attention_usp_gb300 import binding as B; "
                      "assert B.usp_debug_build(); print(B.LIB_PATH)"])
    assert r.returncode == 0 and "_build_debug" in r.stdout, r.stdout + r.stderr
    r = _child(["-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                "-k", "not full_size and not full_workload and not 120k", *SMALL_CASES])
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1]


def test_guard_reports_out_of_range_document_id():
    """A document id past the end of cu_seqlens in the device `doc` array
    (which the host cannot see) makes the attention kernels index cu_seqlens
    out of range; the guarded build reports it instead of reading there.
    Runs only against the guarded library: the release build has no guard
    for this, so the input is never given to it."""
    import numpy as np
    import torch
    from ulysses_sequence_attention_usp_gb300 import binding as B
    if not B.usp_debug_build():
        pytest.skip("needs the library built with index guards (USP_DEBUG_BOUNDS=1)")
    S, P, Hq, Hkv, D = 256, 2, 4, 2, 64
    cu_host = np.array([0, 100, 256], np.int32)
    d = B.make_dims(S, P, Hq, Hkv, D, torch.from_numpy(cu_host).cuda(), cu_host)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    q = torch.randn(P, S, Hq // P, D, **bf)
    k = torch.randn(P, S, Hkv // P, D, **bf)
    v = torch.randn(P, S, Hkv // P, D, **bf)
    doc = torch.zeros(S, dtype=torch.int32, device="cuda")
    doc[100:] = 1
    doc[200] = 7                       # cu_seqlens has 3 entries
    o = torch.empty_like(q)
    lse = torch.empty(P, Hq // P, S, dtype=torch.float32, device="cuda")
    B.usp_attn_fwd(d, q, k, v, doc, o, lse)
    with pytest.raises(B.UspError) as e:
        B.usp_device_status()
    assert e.value.status == 6        # USP_ERR_OUT_OF_BOUNDS
    B.usp_device_status()             # reported once, then cleared


def test_large_cases_run_clean_under_index_guards():
    from ulysses_sequence_attention_usp_gb300 import build
    build.build(debug=True)
    r = _child(["-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider", *LARGE_CASES])
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1]
