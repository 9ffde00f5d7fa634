"""The K/V all-gather context-parallel path with real collectives: P gloo
ranks on the CPU each hold one contiguous shard, gather every rank's K/V
with all_gather, attend their own rows, and reduce-scatter dK/dV (an
all_reduce of the partials followed by each rank keeping its rows).  The
assembled result must equal the oracle's one-process simulation of the same
path and the full-sequence computation (basetenlabs/Megatron-LM PR #7 "GLM-5.2
131k context parallelism", Purpose: KV all-gather forward, dKV
reduce-scatter backward)."""
import math
import os
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

S, HQ, HKV, D = 21, 4, 1, 8
CU = [0, 9, 10, 21]
SCALE = 1.0 / math.sqrt(D)


def _inputs():
    rng = np.random.default_rng(42)
    return (rng.standard_normal((S, HQ, D)), rng.standard_normal((S, HKV, D)),
            rng.standard_normal((S, HKV, D)), rng.standard_normal((S, HQ, D)))


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from oracle import usp_oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=world)
    qa, ka, va, doa = _inputs()
    cu = np.array(CU)
    cos, sin = O.rope_cos_sin(64, D, 1.0e4)
    pos, doc = O.positions_docs(S, world, cu)
    S_pad = pos.shape[0]
    S_loc = S_pad // world
    rows = np.arange(rank * S_loc, (rank + 1) * S_loc)
    # this rank's shard of the padded tensors, rotated at global positions
    q_r = O.rope_rotate(O.shard_pad(qa, world)[rows], pos[rows], cos, sin)
    k_r = O.rope_rotate(O.shard_pad(ka, world)[rows], pos[rows], cos, sin)
    v_r = O.shard_pad(va, world)[rows]
    do_r = O.shard_pad(doa, world)[rows]
    # all-gather of K and V in rank order
    ks = [torch.zeros(S_loc, HKV, D, dtype=torch.float64) for _ in range(world)]
    vs = [torch.zeros(S_loc, HKV, D, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(ks, torch.from_numpy(np.ascontiguousarray(k_r)))
    dist.all_gather(vs, torch.from_numpy(np.ascontiguousarray(v_r)))
    k_all = torch.cat(ks).numpy()
    v_all = torch.cat(vs).numpy()
    G = HQ // HKV
    q_glob = np.zeros((S_pad, HQ, D))
    do_glob = np.zeros((S_pad, HQ, D))
    q_glob[rows], do_glob[rows] = q_r, do_r
    o = np.zeros((S_loc, HQ, D))
    dq = np.zeros((S_loc, HQ, D))
    dk_part = np.zeros((S_pad, HKV, D))
    dv_part = np.zeros((S_pad, HKV, D))
    for h in range(HQ):
        o[:, h], _ = O.attention_rows(q_glob[:, h], k_all[:, h // G], v_all[:, h // G], doc, rows,
                                      SCALE)
        a, b, c = O.attention_bwd_head(q_glob[:, h], k_all[:, h // G], v_all[:, h // G],
                                       do_glob[:, h], doc, SCALE, rows=rows)
        dq[:, h] = a
        dk_part[:, h // G] += b
        dv_part[:, h // G] += c
    # reduce-scatter: sum every rank's partials, keep this rank's rows
    tk, tv = torch.from_numpy(dk_part), torch.from_numpy(dv_part)
    dist.all_reduce(tk)
    dist.all_reduce(tv)
    dk = O.rope_rotate(tk.numpy()[rows], pos[rows], cos, sin, inverse=True)
    dv = tv.numpy()[rows]
    dq = O.rope_rotate(dq, pos[rows], cos, sin, inverse=True)
    q.put((rank, o, dq, dk, dv))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,port", [(2, 29631), (3, 29637)])
def test_gloo_ranks_equal_simulation_and_full_sequence(world, port):
    from oracle import usp_oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got = {n: np.concatenate([r[i] for r in res])[:S] for i, n in
           enumerate(("o", "dq", "dk", "dv"), start=1)}
    qa, ka, va, doa = _inputs()
    cos, sin = O.rope_cos_sin(64, D, 1.0e4)
    cu = np.array(CU)
    sim = O.allgather_cp(qa, ka, va, doa, cu, cos, sin, SCALE, world)
    ref = O.full_sequence(qa, ka, va, doa, cu, cos, sin, SCALE)
    for n in got:
        assert np.allclose(got[n], sim[n], atol=1e-12, rtol=0), n
        assert np.allclose(got[n], ref[n], atol=1e-12, rtol=0), n
