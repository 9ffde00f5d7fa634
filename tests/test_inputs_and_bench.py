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
