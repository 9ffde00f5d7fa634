"""The USP attention forward + backward as one object over the C ABI.

:class:`UlyssesAttention` owns the device buffers of one problem size and
runs the hot path by calling the library's entry points in order
(SpecForge PR #728 "feat(dspark): add Ulysses sequence parallel training",
Modifications):

forward:   positions/documents (+ shard copies for the zigzag layout)
           ->  seq->head all-to-all (+RoPE on Q,K), padding rows as zeros
           ->  local causal GQA attention per head group  ->  head->seq (O)
backward:  seq->head (dO)  ->  attention backward
           ->  head->seq (dQ, dK with the inverse rotation; dV)

In the contiguous shard layout the all-to-all reads the caller's unpadded
tensors directly: padding rows are zero by definition, so the library
writes them without reading anything and no padded copy is made.  The
zigzag layout reorders rows, so there the inputs are first copied into
padded zigzag shards.

PyTorch provides device memory and the stream only; every step runs in the
library's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def _check_input(name, t, rows, heads, D, device):
    """The C ABI cannot see buffer sizes, so a tensor of the wrong shape would
    be read out of bounds on the device: check it here."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.device.type != device.type or (device.index is not None and
                                        t.device.index != device.index):
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != (rows, heads, D):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {(rows, heads, D)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class _GraphStep:
    """CUDA-graph capture of one step (forward + backward), shared by the
    attention pipelines."""

    def capture_step(self, q, k, v, do):
        """Record one forward + backward of these input tensors into a CUDA
        graph and return it (a torch.cuda.CUDAGraph): each replay() runs the
        step's kernels again on the tensors' current contents, into the same
        output buffers, without a host-side launch per kernel (small
        problems are launch-bound).  One eager step runs first, so that the
        library's modules are loaded and its kernel attributes set before
        capture."""
        dev = self.device
        self.step(q, k, v, do)
        torch.cuda.current_stream(dev).synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            graph.capture_begin(capture_error_mode="thread_local")
            try:
                self.step(q, k, v, do)
            finally:
                graph.capture_end()
        torch.cuda.current_stream(dev).wait_stream(side)
        return graph


class UlyssesAttention(_GraphStep):
    def __init__(self, S, P, Hq, Hkv, D, cu_seqlens=None, rope_base=1.0e4, yarn_factor=1.0,
                 yarn_orig_ctx=0, rope_len=0, scale=0.0, device="cuda", rope_table=None,
                 causal=True, zigzag=False, ring=1):
        self.S, self.P, self.Hq, self.Hkv, self.D = int(S), int(P), int(Hq), int(Hkv), int(D)
        unit = 2 * self.P if zigzag else self.P      # zigzag: 2P equal chunks
        self.S_pad = -(-self.S // unit) * unit
        self.zigzag = bool(zigzag)
        self.ring = int(ring)
        if self.ring < 1:
            raise ValueError("ring must be >= 1")
        self.device = torch.device(device)
        dev = self.device
        self.cu_host = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, np.int32)
        self.cu_dev = None if self.cu_host is None else torch.from_numpy(self.cu_host).to(dev)
        self.causal = bool(causal)
        self.dims = B.make_dims(S, P, Hq, Hkv, D, self.cu_dev, self.cu_host, scale, causal,
                                zigzag)
        self.rope_len = int(rope_len) if rope_len else self.S_pad
        if rope_table is None:
            rope_table = B.usp_rope_table(self.rope_len, D, rope_base, yarn_factor, yarn_orig_ctx)
        self.rope_host = rope_table
        self.rope = torch.from_numpy(np.ascontiguousarray(rope_table)).to(dev)
        Sp, hq, hkv = self.S_pad, Hq // P, Hkv // P
        bf = torch.bfloat16
        e = lambda *s, dt=bf: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.pos = e(Sp, dt=torch.int32)
        self.doc = e(Sp, dt=torch.int32)
        if self.zigzag:   # padded zigzag shards of the inputs
            self.q_seq, self.k_seq, self.v_seq = e(Sp, Hq, D), e(Sp, Hkv, D), e(Sp, Hkv, D)
            self.do_seq = e(Sp, Hq, D)
        self.q_h, self.k_h, self.v_h = e(P, Sp, hq, D), e(P, Sp, hkv, D), e(P, Sp, hkv, D)
        self.do_h, self.o_h = e(P, Sp, hq, D), e(P, Sp, hq, D)
        self.lse = e(P, hq, Sp, dt=torch.float32)
        self.dq_h, self.dk_h, self.dv_h = e(P, Sp, hq, D), e(P, Sp, hkv, D), e(P, Sp, hkv, D)
        self.o, self.dq = e(Sp, Hq, D), e(Sp, Hq, D)
        self.dk, self.dv = e(Sp, Hkv, D), e(Sp, Hkv, D)
        self.ws_bytes = B.usp_attn_bwd_workspace(self.dims)
        self.ws = e(max(1, self.ws_bytes), dt=torch.uint8)
        if self.ring > 1:   # partial results of one ring step and the fp32 accumulator
            self.o_part = e(P, Sp, hq, D)
            self.lse_part = e(P, hq, Sp, dt=torch.float32)
            self.o_acc = e(P, Sp, hq, D, dt=torch.float32)
        self._forward_done = False

    # -- steps -------------------------------------------------------------
    def forward(self, q, k, v, stream=None):
        """q [S][Hq][D], k/v [S][Hkv][D] bf16 device tensors (pre-RoPE).
        Returns O [S_pad][Hq][D] in the sequence-sharded layout (global row
        order, or zigzag shard order when zigzag=True); padding rows are 0."""
        for n, t, h in (("q", q, self.Hq), ("k", k, self.Hkv), ("v", v, self.Hkv)):
            _check_input(n, t, self.S, h, self.D, self.device)
        d, st = self.dims, stream
        if self.zigzag:
            B.usp_pad_shard(d, q, self.Hq, self.q_seq, self.pos, self.doc, st)
            B.usp_pad_shard(d, k, self.Hkv, self.k_seq, None, None, st)
            B.usp_pad_shard(d, v, self.Hkv, self.v_seq, None, None, st)
            q, k, v = self.q_seq, self.k_seq, self.v_seq
        else:
            B.usp_pad_shard(d, None, 0, None, self.pos, self.doc, st)
        B.usp_seq_to_head_rope(d, q, self.Hq, self.pos, self.rope, self.rope_len, 1, self.q_h, st)
        B.usp_seq_to_head_rope(d, k, self.Hkv, self.pos, self.rope, self.rope_len, 1, self.k_h, st)
        B.usp_seq_to_head_rope(d, v, self.Hkv, None, None, 0, 0, self.v_h, st)
        self.attention_forward(st)
        B.usp_head_to_seq(d, self.o_h, self.Hq, None, None, 0, 0, self.o, st)
        self._forward_done = True
        return self.o

    def attention_forward(self, stream=None):
        """The attention of the head-layout Q, K, V into o_h and lse: one call,
        or with ring > 1 the ring steps -- step c attends to key rows
        [c*L, (c+1)*L), the partial results are merged (log-sum-exp) into an
        fp32 accumulator, and the last merge writes O and its LSE.  The
        backward then runs on the merged O and LSE: with every key chunk
        resident, the ring backward's per-block sums equal the key- and
        query-stationary passes over the whole range."""
        d, st = self.dims, stream
        if self.ring == 1:
            B.usp_attn_fwd(d, self.q_h, self.k_h, self.v_h, self.doc, self.o_h, self.lse, st)
            return
        L = -(-self.S_pad // self.ring)
        for c in range(self.ring):
            lo, hi = min(self.S_pad, c * L), min(self.S_pad, (c + 1) * L)
            B.usp_attn_fwd_window(d, self.q_h, self.k_h, self.v_h, self.doc, lo, hi,
                                  self.o_part, self.lse_part, st)
            B.usp_lse_merge(d, self.o_acc, self.lse, self.o_part, self.lse_part, c == 0,
                            self.o_h if c == self.ring - 1 else None, st)

    def backward(self, do, stream=None):
        """do [S][Hq][D] bf16 (dL/dO).  Returns dQ, dK, dV [S_pad][H][D]: the
        gradients of the pre-RoPE sequence-sharded inputs, in the same shard
        layout as O."""
        if not self._forward_done:
            raise RuntimeError("backward before forward")
        _check_input("do", do, self.S, self.Hq, self.D, self.device)
        d, st = self.dims, stream
        if self.zigzag:
            B.usp_pad_shard(d, do, self.Hq, self.do_seq, None, None, st)
            do = self.do_seq
        B.usp_seq_to_head_rope(d, do, self.Hq, None, None, 0, 0, self.do_h, st)
        B.usp_attn_bwd(d, self.q_h, self.k_h, self.v_h, self.o_h, self.lse, self.do_h, self.doc,
                       self.dq_h, self.dk_h, self.dv_h, self.ws, self.ws_bytes, st)
        B.usp_head_to_seq(d, self.dq_h, self.Hq, self.pos, self.rope, self.rope_len, -1,
                          self.dq, st)
        B.usp_head_to_seq(d, self.dk_h, self.Hkv, self.pos, self.rope, self.rope_len, -1,
                          self.dk, st)
        B.usp_head_to_seq(d, self.dv_h, self.Hkv, None, None, 0, 0, self.dv, st)
        return self.dq, self.dk, self.dv

    def step(self, q, k, v, do, stream=None):
        self.forward(q, k, v, stream)
        return self.backward(do, stream)

    def check(self, stream=None):
        B.usp_device_status(stream)


class AllGatherCPAttention(_GraphStep):
    """Context parallelism with a K/V all-gather over P virtual ranks
    (basetenlabs/Megatron-LM PR #7 "GLM-5.2 131k context parallelism",
    Purpose: the CP forward all-gathers the KV of every rank, the backward
    reduce-scatters dKV; contiguous partition; positions from the global
    cu_seqlens).

    Rank r holds the contiguous rows [r*S_loc, (r+1)*S_loc) of Q, K, V with
    all heads, so no head count has to be divisible by P: this is the
    layout for fewer KV heads than ranks, which the all-to-all cannot shard.
    On one GPU the shards are row ranges of one sequence-layout buffer, so
    the all-gather of K/V is that buffer itself and the reduce-scatter of
    dK/dV is the key-stationary backward pass's sum over the query rows of
    every rank.  A step is therefore

      positions/documents -> RoPE of Q and K at global positions
      -> attention of every rank's rows over all keys (one launch)
      -> backward (delta, dK/dV, dQ) -> inverse RoPE of dQ and dK

    with the library's entry points called on a one-shard geometry; V, O,
    dO and dV are used in place, never copied.  Rows are not padded: equal
    shards on P devices would add only masked rows (document -1), which
    change no valid output.
    """

    def __init__(self, S, P, Hq, Hkv, D, cu_seqlens=None, rope_base=1.0e4, yarn_factor=1.0,
                 yarn_orig_ctx=0, rope_len=0, scale=0.0, device="cuda", rope_table=None,
                 causal=True):
        self.S, self.P, self.Hq, self.Hkv, self.D = int(S), int(P), int(Hq), int(Hkv), int(D)
        if self.P < 1:
            raise ValueError("P must be >= 1")
        self.S_loc = -(-self.S // self.P)
        self.device = torch.device(device)
        dev = self.device
        self.cu_host = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, np.int32)
        self.cu_dev = None if self.cu_host is None else torch.from_numpy(self.cu_host).to(dev)
        self.causal = bool(causal)
        # one shard holding every row: the gathered view all ranks share
        self.dims = B.make_dims(S, 1, Hq, Hkv, D, self.cu_dev, self.cu_host, scale, causal)
        self.rope_len = int(rope_len) if rope_len else self.S
        if rope_table is None:
            rope_table = B.usp_rope_table(self.rope_len, D, rope_base, yarn_factor, yarn_orig_ctx)
        self.rope_host = rope_table
        self.rope = torch.from_numpy(np.ascontiguousarray(rope_table)).to(dev)
        S_ = self.S
        bf = torch.bfloat16
        e = lambda *s, dt=bf: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.pos = e(S_, dt=torch.int32)
        self.doc = e(S_, dt=torch.int32)
        self.q_r, self.k_r = e(S_, Hq, D), e(S_, Hkv, D)        # rotated Q, K
        self.o = e(S_, Hq, D)
        self.lse = e(Hq, S_, dt=torch.float32)
        self.dq_r, self.dk_r = e(S_, Hq, D), e(S_, Hkv, D)      # gradients, rotated frame
        self.dq, self.dk, self.dv = e(S_, Hq, D), e(S_, Hkv, D), e(S_, Hkv, D)
        self.ws_bytes = B.usp_attn_bwd_workspace(self.dims)
        self.ws = e(max(1, self.ws_bytes), dt=torch.uint8)
        self._v = None

    def shard(self, x, r):
        """Rank r's rows of a sequence-layout tensor (a view)."""
        return x[r * self.S_loc:min(self.S, (r + 1) * self.S_loc)]

    def forward(self, q, k, v, stream=None):
        """q [S][Hq][D], k/v [S][Hkv][D] bf16 contiguous device tensors
        (pre-RoPE, every rank's rows in rank order).  Returns O [S][Hq][D]."""
        for n, t, h in (("q", q, self.Hq), ("k", k, self.Hkv), ("v", v, self.Hkv)):
            _check_input(n, t, self.S, h, self.D, self.device)
        d, st = self.dims, stream
        B.usp_pad_shard(d, None, 0, None, self.pos, self.doc, st)
        B.usp_seq_to_head_rope(d, q, self.Hq, self.pos, self.rope, self.rope_len, 1, self.q_r,
                               st)
        B.usp_seq_to_head_rope(d, k, self.Hkv, self.pos, self.rope, self.rope_len, 1, self.k_r,
                               st)
        self._v = v
        B.usp_attn_fwd(d, self.q_r, self.k_r, v, self.doc, self.o, self.lse, st)
        return self.o

    def backward(self, do, stream=None):
        """do [S][Hq][D] bf16 contiguous.  Returns dQ, dK, dV [S][H][D], the
        gradients of the pre-RoPE inputs (rank r's rows are its shard)."""
        if self._v is None:
            raise RuntimeError("backward before forward")
        _check_input("do", do, self.S, self.Hq, self.D, self.device)
        d, st = self.dims, stream
        B.usp_attn_bwd(d, self.q_r, self.k_r, self._v, self.o, self.lse, do, self.doc,
                       self.dq_r, self.dk_r, self.dv, self.ws, self.ws_bytes, st)
        B.usp_head_to_seq(d, self.dq_r, self.Hq, self.pos, self.rope, self.rope_len, -1,
                          self.dq, st)
        B.usp_head_to_seq(d, self.dk_r, self.Hkv, self.pos, self.rope, self.rope_len, -1,
                          self.dk, st)
        return self.dq, self.dk, self.dv

    def step(self, q, k, v, do, stream=None):
        self.forward(q, k, v, stream)
        return self.backward(do, stream)

    def check(self, stream=None):
        B.usp_device_status(stream)
