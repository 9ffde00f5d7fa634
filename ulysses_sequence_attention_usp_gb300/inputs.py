"""Seeded synthetic inputs for the USP attention hot path.

This module only draws random numbers and names workload shapes.  It holds
none of the method's arithmetic (no padding, permutation, RoPE or attention),
so both the CUDA path and the CPU oracle may consume what it produces.

Workloads (shapes of the pages' Qwen3-8B / GLM-5.2 long-context runs):

* ``tiny``      S=256,    P=2, Hq/Hkv/D = 4/2/64,   RoPE base 1e4
* ``qwen8k``    S=8192,   P=8, 32/8/128,            RoPE base 1e6
* ``long32k``   S=32768,  P=8, 32/8/128,            RoPE base 1e6
* ``long32k_pad`` S=32766 (padded to 32768), P=8, 32/8/128
* ``sp8_120k``  S=120000, P=8, 32/8/128, YaRN-scaled RoPE to 131072
* ``thd64k``    65536 packed tokens, documents log-uniform[512,16384]
                (last truncated), P=8, 64/8/128, RoPE base 1e6

Values are N(0,1) drawn in fp32 by ``numpy.random.default_rng(seed)`` and
rounded to bf16 (round to nearest even).  Separate generator streams are used
for the document lengths, Q, K, V and dO so that changing one tensor's shape
leaves the others unchanged.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    S: int                    # valid tokens
    P: int                    # Ulysses degree (virtual shards)
    Hq: int
    Hkv: int
    D: int
    rope_base: float
    yarn_factor: float = 1.0  # 1.0 => plain RoPE
    yarn_orig_ctx: int = 0    # native context of the YaRN-scaled model
    rope_len: int = 0         # table length; 0 => S_pad
    thd: bool = False         # packed documents (cu_seqlens) if True

    @property
    def S_pad(self) -> int:
        return -(-self.S // self.P) * self.P

    @property
    def S_loc(self) -> int:
        return self.S_pad // self.P

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def table_len(self) -> int:
        return self.rope_len if self.rope_len else self.S_pad


WORKLOADS = {
    "tiny": Workload("tiny", 256, 2, 4, 2, 64, 1.0e4),
    "qwen8k": Workload("qwen8k", 8192, 8, 32, 8, 128, 1.0e6),
    "long32k": Workload("long32k", 32768, 8, 32, 8, 128, 1.0e6),
    "long32k_pad": Workload("long32k_pad", 32766, 8, 32, 8, 128, 1.0e6),
    "sp8_120k": Workload("sp8_120k", 120000, 8, 32, 8, 128, 1.0e6,
                         yarn_factor=4.0, yarn_orig_ctx=32768, rope_len=131072),
    "thd64k": Workload("thd64k", 65536, 8, 64, 8, 128, 1.0e6, thd=True),
}

# Stream ids: one independent generator per tensor, all from the same seed.
_STREAM = {"doclens": 0, "q": 1, "k": 2, "v": 3, "do": 4}


def _rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.default_rng([seed, _STREAM[stream]]) if stream != "doclens" \
        else np.random.default_rng(seed)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def normal_bf16(shape, seed: int, stream: str, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) fp32 draws rounded to bf16, as uint16 bits of the given shape."""
    rng = _rng(seed, stream)
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = f32_to_bf16_bits(rng.standard_normal(hi - lo, dtype=np.float32))
    return out.reshape(shape)


def doc_lengths(total: int, seed: int = 0, lo: int = 512, hi: int = 16384) -> list:
    """Document lengths L = round(exp(U(ln lo, ln hi))), drawn until they reach
    ``total``; the last one is truncated so that they sum to ``total``."""
    rng = _rng(seed, "doclens")
    lens, s = [], 0
    while s < total:
        n = int(round(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
        lens.append(n)
        s += n
    lens[-1] -= s - total
    return lens


def cu_seqlens(lens) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: np.ndarray            # uint16 bf16 bits [S][Hq][D] (pre-RoPE, unpadded)
    k: np.ndarray            # [S][Hkv][D]
    v: np.ndarray            # [S][Hkv][D]
    do: np.ndarray           # [S][Hq][D] upstream gradient of O
    cu: Optional[np.ndarray]  # int32 [n_docs+1] or None (one sequence)


def make_inputs(wl: Workload, seed: int = 0, with_do: bool = True,
                lens=None) -> Inputs:
    """Draw Q, K, V (and dO) for ``wl``.  For packed workloads the document
    lengths are ``lens`` if given, else drawn by :func:`doc_lengths`."""
    S, D = wl.S, wl.D
    q = normal_bf16((S, wl.Hq, D), seed, "q")
    k = normal_bf16((S, wl.Hkv, D), seed, "k")
    v = normal_bf16((S, wl.Hkv, D), seed, "v")
    do = normal_bf16((S, wl.Hq, D), seed, "do") if with_do else None
    cu = None
    if wl.thd:
        cu = cu_seqlens(lens if lens is not None else doc_lengths(S, seed))
        assert int(cu[-1]) == S
    return Inputs(wl, q, k, v, do, cu)


def custom_workload(S, P, Hq, Hkv, D, base=1.0e4, thd_lens=None, name="custom",
                    yarn_factor=1.0, yarn_orig_ctx=0, rope_len=0) -> Workload:
    return Workload(name, S, P, Hq, Hkv, D, base, yarn_factor, yarn_orig_ctx,
                    rope_len, thd=thd_lens is not None)
