"""Helpers shared by the GPU parity tests: host<->device transfer of bf16
bit patterns, and oracle evaluations restricted to sampled rows so that the
full-size workloads can be checked in seconds."""
import math

import numpy as np
import torch

from oracle import usp_oracle as O

# Tolerances (the same everywhere):
O_MAX, O_MEAN = 2e-2, 2e-3          # attention output vs fp64
GRAD_REL = 5e-2                     # dQ/dK/dV max|diff| / max|ref| per tensor
GRAD_ABS_FLOOR = 1e-4               # when the exact gradient is identically 0
LSE_ABS = 1e-3


def to_dev(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.cuda().view(torch.bfloat16)


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_o(got, ref, what="O"):
    d = np.abs(got - ref)
    assert d.max() <= O_MAX and d.mean() <= O_MEAN, (what, d.max(), d.mean())


def check_grad(got, ref, what):
    """max|got - ref| <= GRAD_REL * max|ref|.  When the exact gradient is
    identically zero (e.g. one token per document: softmax over a single key
    has zero gradient w.r.t. its score) the relative criterion is empty; the
    GPU then keeps the residue of delta = dO.O computed with bf16 O, and
    GRAD_ABS_FLOOR bounds it."""
    err = np.abs(got - ref).max()
    bound = max(GRAD_REL * np.abs(ref).max(), GRAD_ABS_FLOOR)
    assert err <= bound, (what, err, bound)
    return err


def check_lse(got, ref, tol=LSE_ABS):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.all(got[~fin] == ref[~fin])
    if fin.any():
        err = np.abs(got[fin] - ref[fin]).max()
        assert err <= tol, (err, tol)


def lse_tol_end_to_end(q_rot_norm_max, k_rot_norm_max, scale):
    """LSE tolerance when the GPU rounds the rotated Q and K to bf16 but the
    reference rotates exactly: each score moves by at most
    scale*(|dq||k| + |q||dk| + |dq||dk|) with |dq| <= 2^-8 |q| (bf16 unit
    roundoff), and the LSE of a row moves by at most its largest score
    change; 1e-3 is added for fp32 accumulation."""
    u = 2.0 ** -8
    return LSE_ABS + scale * (2 * u + u * u) * q_rot_norm_max * k_rot_norm_max


class SampledOracle:
    """Oracle values at chosen rows of one full-size problem.

    Inputs are the pre-RoPE bf16 bits of the unpadded sequence; RoPE is the
    exact fp64 rotation of the oracle (this is the end-to-end reference).
    """

    def __init__(self, q, k, v, do, cu, wl, causal=True):
        self.wl = wl
        self.causal = causal
        S, D = wl.S, wl.D
        self.S = S
        self.G = wl.Hq // wl.Hkv
        self.scale = 1.0 / math.sqrt(D)
        self.pos, self.doc = O.positions_docs(S, 1, cu)
        self.cos, self.sin = O.rope_cos_sin(max(wl.table_len, S), D, wl.rope_base,
                                            wl.yarn_factor, wl.yarn_orig_ctx)
        self.q, self.k, self.v, self.do = q, k, v, do
        self._kr = {}
        self._kb = {}
        self._table = None

    def table(self):
        """The fp32 (cos, sin) table the GPU run is given (built by the oracle)."""
        if self._table is None:
            wl = self.wl
            self._table = O.rope_table_f32(max(wl.table_len, self.S), wl.D, wl.rope_base,
                                           wl.yarn_factor, wl.yarn_orig_ctx)
        return self._table

    def lse_rows_recipe(self, h, rows):
        """LSE of head h at the given rows when the attention is fed the bf16
        rotated Q and K of the fp32 recipe (the GPU's actual inputs): exact
        fp64 attention of those bf16 values, so only the kernel's own
        arithmetic separates the two."""
        kh = h // self.G
        if kh not in self._kb:
            kr = O.rope_recipe_bf16(self.k[:, kh:kh + 1], self.pos[:self.S], self.table())
            self._kb[kh] = O.bf16_to_f64(kr[:, 0])
        rows = np.asarray(rows)
        qr = np.zeros((self.S, self.wl.D))
        qr[rows] = O.bf16_to_f64(O.rope_recipe_bf16(self.q[rows, h:h + 1], self.pos[rows],
                                                    self.table())[:, 0])
        _, lse = O.attention_rows(qr, self._kb[kh], O.bf16_to_f64(self.v[:, kh]), self.doc,
                                  rows, self.scale, self.causal)
        return lse

    def dkv_keys(self, kh, keys, rows, workers=None):
        """Pre-RoPE dK and dV of KV head kh at ``keys`` from every query row in
        ``rows`` (all the rows that see them), evaluated over row chunks in
        spawned worker processes (tests/oracle_pool.py)."""
        from oracle_pool import dkdv_keys
        G = self.G
        return dkdv_keys(self.q[:, kh * G:(kh + 1) * G], self.k[:, kh], self.v[:, kh],
                         self.do[:, kh * G:(kh + 1) * G], self.pos, self.doc, self.cos,
                         self.sin, self.scale, keys, rows, causal=self.causal, workers=workers)

    def _rot(self, bits_rows, rows):
        x = O.bf16_to_f64(bits_rows)
        return O.rope_rotate(x[:, None, :], self.pos[rows], self.cos, self.sin)[:, 0]

    def k_rot(self, kh):
        if kh not in self._kr:
            self._kr[kh] = self._rot(self.k[:, kh], np.arange(self.S))
        return self._kr[kh]

    def fwd_rows(self, h, rows):
        kh = h // self.G
        qr = np.zeros((self.S, self.wl.D))
        qr[rows] = self._rot(self.q[rows, h], rows)
        return O.attention_rows(qr, self.k_rot(kh), O.bf16_to_f64(self.v[:, kh]), self.doc,
                                np.asarray(rows), self.scale, self.causal)

    def dq_rows(self, h, rows):
        """Pre-RoPE dQ of head h at the given rows."""
        kh = h // self.G
        qr = np.zeros((self.S, self.wl.D))
        qr[rows] = self._rot(self.q[rows, h], rows)
        dq, _, _ = O.attention_bwd_head(qr, self.k_rot(kh), O.bf16_to_f64(self.v[:, kh]),
                                        O.bf16_to_f64(self.do[:, h]), self.doc, self.scale,
                                        rows=np.asarray(rows), causal=self.causal)
        return O.rope_rotate(dq[:, None, :], self.pos[rows], self.cos, self.sin,
                             inverse=True)[:, 0]

    def dkv_tail(self, kh, u_lo, u_hi, q_lo=None):
        """Pre-RoPE dK and dV of KV head kh at keys [u_lo, u_hi), which must lie
        in one document that ends at u_hi.  The queries that see them are
        [u_lo, u_hi) when causal; bidirectional, pass q_lo = the document's
        first row so that all of its queries contribute."""
        rows = np.arange(u_lo if q_lo is None else q_lo, u_hi)
        dk = np.zeros((u_hi - u_lo, self.wl.D))
        dv = np.zeros_like(dk)
        for i in range(self.G):
            h = kh * self.G + i
            qr = np.zeros((self.S, self.wl.D))
            qr[rows] = self._rot(self.q[rows, h], rows)
            _, a, b = O.attention_bwd_head(qr, self.k_rot(kh), O.bf16_to_f64(self.v[:, kh]),
                                           O.bf16_to_f64(self.do[:, h]), self.doc, self.scale,
                                           rows=rows, causal=self.causal)
            dk += a[u_lo:u_hi]
            dv += b[u_lo:u_hi]
        keys = np.arange(u_lo, u_hi)
        dk = O.rope_rotate(dk[:, None, :], self.pos[keys], self.cos, self.sin, inverse=True)[:, 0]
        return dk, dv


def check_sampled_full_size(wl, inp, orc, o, lse, dq, dk, dv, seed, buf_of=None,
                            tail_keys=True):
    """Oracle checks of one full-size step on sampled rows: O, dQ and LSE
    (1e-3 against the recipe-rotated bf16 Q, K) for three query heads, and
    dK/dV of the last 48 keys of the sequence (or of the last document) for
    the first and last KV heads.  o, dq, dk, dv are the sequence-layout
    outputs ([rows][H][D] device tensors), lse the head-layout LSE
    ([Hq][S_pad] after reshaping); buf_of maps a global row to its row in
    the sequence-layout buffers (identity when None)."""
    S = wl.S
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, S // 2, S - 1], rng.integers(0, S, 8)]))
    bo = (lambda r: r) if buf_of is None else (lambda r: buf_of[r])
    heads = sorted({0, wl.Hq - 1, int(rng.integers(0, wl.Hq))})
    got_o, ref_o, got_l, ref_l, got_dq, ref_dq = [], [], [], [], [], []
    for h in heads:
        r_o, _ = orc.fwd_rows(h, rows)
        got_o.append(to_f64(o[bo(rows), h]))
        ref_o.append(r_o)
        got_l.append(lse[h, rows].cpu().numpy().astype(np.float64))
        ref_l.append(orc.lse_rows_recipe(h, rows))
        got_dq.append(to_f64(dq[bo(rows), h]))
        ref_dq.append(orc.dq_rows(h, rows))
    check_o(np.concatenate(got_o), np.concatenate(ref_o))
    check_grad(np.concatenate(got_dq), np.concatenate(ref_dq), "dq")
    check_lse(np.concatenate(got_l), np.concatenate(ref_l))
    if tail_keys:
        end = S if inp.cu is None else int(inp.cu[-1])
        lo = end - 48
        for kh in sorted({0, wl.Hkv - 1}):
            r_dk, r_dv = orc.dkv_tail(kh, lo, end)
            idx = bo(np.arange(lo, end))
            check_grad(to_f64(dk[idx, kh]), r_dk, "dk")
            check_grad(to_f64(dv[idx, kh]), r_dv, "dv")
