"""CPU checks of the seeded workload generator and of the bench's pair
counting: the packed 64K workload has the documented 13 documents, inputs are
reproducible per (seed, tensor), and the FLOP accounting's attended-pair
count equals a brute-force count of visible (query, key) pairs under the
oracle's mask."""
import numpy as np
import pytest

import bench
from oracle import usp_oracle as O
from ulysses_sequence_attention_usp_gb300.inputs import (WORKLOADS, cu_seqlens, doc_lengths,
                                                         make_inputs, normal_bf16)


def test_packed_workload_documents():
    lens = doc_lengths(65536)
    assert lens == [4656, 1304, 590, 542, 8578, 12109, 4191, 6416, 3369, 13083, 8655, 517, 1526]
    assert sum(lens) == 65536
    assert all(512 <= n <= 16384 for n in lens[:-1]) and 1 <= lens[-1] <= 16384
    cu = cu_seqlens(lens)
    assert cu[0] == 0 and cu[-1] == 65536 and np.all(np.diff(cu) > 0)


def test_inputs_are_reproducible_per_seed_and_tensor():
    a = normal_bf16((64, 4, 8), 0, "q")
    assert np.array_equal(a, normal_bf16((64, 4, 8), 0, "q"))
    assert not np.array_equal(a, normal_bf16((64, 4, 8), 0, "k"))
    assert not np.array_equal(a, normal_bf16((64, 4, 8), 1, "q"))
    x = O.bf16_to_f64(normal_bf16((20000,), 3, "v"))
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1.0) < 0.05      # N(0, 1) in bf16
    inp = make_inputs(WORKLOADS["tiny"], 0)
    assert inp.q.shape == (256, 4, 64) and inp.k.shape == (256, 2, 64)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S,lens", [(37, None), (40, [10, 1, 0, 20, 9]), (1, None)])
def test_attended_pairs_match_the_mask(S, lens, causal):
    cu = None if lens is None else cu_seqlens(lens)
    _, doc = O.positions_docs(S, 1, cu)
    vis = O._visible(np.arange(S), doc, causal)
    assert bench.attended_pairs(S, cu, causal) == int(vis.sum())


def test_l2_note_says_whether_steps_are_l2_warm():
    l2 = 129 << 20
    big = bench.l2_note(2 * (983_040_000 + 245_760_000), l2)   # the 120K workload
    small = bench.l2_note(2 * (256 * 4 * 64 * 2 + 256 * 2 * 64 * 2), l2)
    assert "larger than L2" in big and "no flush" in big
    assert "smaller than L2" in small and "not flushed" in small
    assert "258 MB memset" in big and "258 MB memset" in small


def test_both_arms_print_the_same_config_keys():
    import types
    wl = WORKLOADS["sp8_120k"]
    for cp, zz, ring in (("ulysses", False, 1), ("ulysses", True, 1), ("ulysses", False, 4),
                         ("allgather", False, 1)):
        a = types.SimpleNamespace(cp=cp, bidirectional=False, zigzag=zz, ring=ring)
        c = bench.workload_config(a, wl, 1)
        assert c["workload"] == "sp8_120k" and c["S"] == 120000 and c["ring"] == ring
        assert ("all-gather" in c["shards"]) == (cp == "allgather")
        assert ("zigzag" in c["shards"]) == zz


def test_both_arms_lines_share_the_config():
    # both arms build their JSON line from bench.base_line, so `config` is the
    # same dict for the same flags (the GPU arm's L2 note is a separate key)
    import types
    wl = WORKLOADS["sp8_120k"]
    a = types.SimpleNamespace(cp="ulysses", bidirectional=False, zigzag=False, ring=1,
                              steps=5, warmup=3)
    gpu = bench.base_line(a, wl, 1, 3.5e5, 339.0, "bf16")
    ref = dict(impl="reference", **bench.base_line(a, wl, 1, 10.0, 1.2e7, "f64"))
    assert gpu["config"] == ref["config"] and "l2" not in gpu["config"]
    for k in ("metric", "unit", "higher_is_better", "scaling", "n_gpus", "steps", "warmup"):
        assert gpu[k] == ref[k]
    src = open(bench.__file__).read()
    assert src.count("base_line(args, wl,") == 3      # the definition and one call per arm


def test_clock_summary_parses_nvidia_smi_lines():
    lines = ["1935, 2070, 1380.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "1965, 2070, 1390.1, 0x0000000000000000, Not Active, Not Active, Not Active, "
             "Not Active",
             "garbled"]
    d = bench.ClockSampler._summary(lines)
    assert d == {"sm_mhz": 1950.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 2}
    assert bench.ClockSampler._summary([]) is None


def test_parity_sample_reports_maxima():
    import types
    import torch
    Sp, D = 5, 4
    rng = np.random.default_rng(0)
    ref = {"o": rng.standard_normal((Sp, 1, D)), "dq": rng.standard_normal((Sp, 1, D)),
           "lse": rng.standard_normal((1, Sp))}
    o = np.zeros((8, 2, D))
    o[:Sp, 0] = ref["o"][:, 0] + 0.01
    dq = np.zeros((8, 2, D))
    dq[:Sp, 0] = ref["dq"][:, 0] * 1.02
    lse = np.zeros((1, 2, 8))
    lse[0, 0, :Sp] = ref["lse"][0] - 3e-4
    ua = types.SimpleNamespace(o=torch.tensor(o), dq=torch.tensor(dq), lse=torch.tensor(lse))
    r = bench.parity_sample(ua, types.SimpleNamespace(Hq=2), ref, Sp)
    assert abs(r["o_max_abs"] - 0.01) < 1e-6 and abs(r["o_mean_abs"] - 0.01) < 1e-6
    assert abs(r["dq_max_rel"] - 0.02) < 1e-6
    assert abs(r["lse_max_abs"] - 3e-4) < 1e-6
    assert r["within_criteria"] is False          # mean |dO| 1e-2 > 2e-3
