"""The oracle's key-gradient function evaluated over row chunks in spawned
worker processes (numpy only; no torch, no CUDA), so that dK/dV of the
first keys of a 120 000-row document -- which every later query row sees --
can be checked against fp64 in about a minute.

The parent writes the bf16 bits of one KV head's inputs to .npy files; each
worker maps them read-only, rotates rows exactly (fp64 RoPE), and returns
the partial dK/dV of the chosen keys summed over its chunk of query rows.
Each query row's contribution depends on that row alone, so the partial sums
add up to the full gradient (pinned in tests/test_oracle_attention.py)."""
from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

from oracle import usp_oracle as O

_W = {}


def _init(path, D, scale, causal):
    ld = lambda n: np.load(os.path.join(path, n + ".npy"), mmap_mode="r")  # noqa: E731
    _W.update(q=ld("q"), do=ld("do"), k=ld("k"), v=ld("v"), pos=ld("pos"), doc=ld("doc"),
              cos=ld("cos"), sin=ld("sin"), D=D, scale=scale, causal=causal, kr=None)


def _rot(bits, rows):
    x = O.bf16_to_f64(np.asarray(bits))
    pos = np.asarray(_W["pos"][rows])
    return O.rope_rotate(x[:, None, :], pos, _W["cos"], _W["sin"])[:, 0]


def _chunk(task):
    """task = (head index i, first row a, end row b, keys): partial dK, dV of
    the keys (rotated frame) over query rows [a, b) of head i."""
    i, a, b, keys = task
    hi = b if _W["causal"] else _W["k"].shape[0]
    if _W["kr"] is None or _W["kr"].shape[0] < hi:
        n = _W["k"].shape[0]
        _W["kr"] = _rot(_W["k"][:n], np.arange(n))
        _W["vf"] = O.bf16_to_f64(np.asarray(_W["v"][:n]))
    rows = np.arange(a, b)
    q = np.zeros((hi, _W["D"]))
    do = np.zeros((hi, _W["D"]))
    q[rows] = _rot(_W["q"][a:b, i], rows)
    do[rows] = O.bf16_to_f64(np.asarray(_W["do"][a:b, i]))
    return O.attention_bwd_keys(q, _W["kr"][:hi], _W["vf"][:hi], do, np.asarray(_W["doc"][:hi]),
                                _W["scale"], keys, rows=rows, causal=_W["causal"])


def dkdv_keys(q_bits, k_bits, v_bits, do_bits, pos, doc, cos, sin, scale, keys, rows,
              causal=True, chunk=256, workers=None):
    """Pre-RoPE dK, dV of one KV head at ``keys``, summed over the query heads
    of its group and the query rows ``rows`` (a contiguous range).

    q_bits/do_bits: bf16 bits [T][G][D] of the group's query heads; k_bits,
    v_bits: [T][D]; pos/doc: [T]; cos/sin: exact fp64 RoPE tables."""
    T, G, D = q_bits.shape
    keys = np.asarray(keys, np.int64)
    a0, b0 = int(rows[0]), int(rows[-1]) + 1
    tasks = [(i, a, min(b0, a + chunk), keys) for i in range(G) for a in range(a0, b0, chunk)]
    if workers is None:
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 4
        try:   # keep several GB of headroom: a worker holds ~1 GB at 120K rows
            mem_gb = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE") / 2 ** 30
        except (ValueError, OSError):
            mem_gb = 16.0
        workers = max(1, min(cores, int(mem_gb // 3)))
    dk = np.zeros((keys.shape[0], D))
    dv = np.zeros_like(dk)
    with tempfile.TemporaryDirectory() as path:
        for n, arr in (("q", q_bits), ("do", do_bits), ("k", k_bits), ("v", v_bits),
                       ("pos", pos), ("doc", doc), ("cos", cos), ("sin", sin)):
            np.save(os.path.join(path, n + ".npy"), np.ascontiguousarray(arr))
        # workers do their own BLAS on one thread each; spawn, never fork, so
        # that no CUDA state of the parent is inherited
        old = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS")}
        os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")
        try:
            ctx = mp.get_context("spawn")
            with ctx.Pool(workers, initializer=_init, initargs=(path, D, scale, causal)) as pool:
                for a, b in pool.imap_unordered(_chunk, tasks):
                    dk += a
                    dv += b
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
    dk = O.rope_rotate(dk[:, None, :], np.asarray(pos)[keys], cos, sin, inverse=True)[:, 0]
    return dk, dv
