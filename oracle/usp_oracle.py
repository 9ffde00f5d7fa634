"""CPU fp64 oracle for Ulysses sequence-parallel (USP) attention.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the GPU path computes.  It is imported by ``tests/``, by
``__graft_entry__.smoke()`` (one small check) and by ``bench.py``'s CPU
baseline leg, and by nothing else: the library under
``ulysses_sequence_attention_usp_gb300`` never calls it, and it shares no code
with that library.

Sources (the pages this follows; none of them writes Ulysses out as equations):

* SpecForge PR #728 "feat(dspark): add Ulysses sequence parallel training",
  section Modifications: inputs and their *absolute* positions are sharded and
  padded across the SP group; Q, K and V go through separate all-to-alls before
  *local* attention; head counts must be divisible by the Ulysses degree.
  Section Accuracy Test: loss and gradient parity against full-sequence
  attention is the correctness criterion.
* basetenlabs/Megatron-LM PR #7 "GLM-5.2 131k context parallelism", section
  Purpose: contiguous partition of packed (THD) sequences; RoPE positions come
  from the *global* cu_seqlens; the RoPE table must cover the padded length.
* zhtmike/verl PR #45 "[trainer] feat: support sequence parallel": sequence
  lengths are padded for SP alignment; SP and non-SP fwd / fwd+bwd must agree.
* SpecForge PR #728, section Accuracy Test (Qwen3-8B run): "YaRN context
  131,072" -- the YaRN table follows Peng et al., "YaRN: Efficient Context
  Window Extension of Large Language Models" (2023), sections 3.2-3.4.

Readings where the pages are silent (each one is listed in the design notes):
contiguous head groups per rank; rotate-half RoPE pairing (d, d + D/2);
padding at the global tail with positions that keep counting; pad rows are
never keys, their O rows are 0 and their LSE is -inf; scale 1/sqrt(D);
natural-log LSE; the fp32 rounding recipe of :func:`rope_recipe_bf16`.

Parity pins: every function here is pinned by ``tests/test_oracle*.py``
against facts other than itself (closed forms, invariants, library routines
such as torch's scaled_dot_product_attention, brute force loops, finite
differences).  The YaRN ramp constants (beta_fast=32, beta_slow=1, original
context 32768, factor 4) are a reading, not fixed by the pages: parity
unpinned for those constants beyond the factor=1 special case and the
limiting regimes of the ramp.

Arrays: bf16 values travel as ``uint16`` bit patterns; all arithmetic is fp64
unless a function states otherwise.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# bf16 <-> float conversion (IEEE bit manipulation, round to nearest even)
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bits, nearest with ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# Shard + pad, positions and document ids
# (SpecForge #728 Modifications; verl #45 "pads seq-lens for SP alignment";
#  Megatron-LM #7 Purpose: contiguous partition, global cu_seqlens)
# ---------------------------------------------------------------------------


def padded_len(S: int, P: int) -> int:
    """S rounded up to a multiple of the Ulysses degree P."""
    return -(-S // P) * P


def shard_pad(x: np.ndarray, P: int) -> np.ndarray:
    """[S][H][D] -> [S_pad][H][D]; rows S..S_pad-1 are zero.  Shard r is the
    contiguous row range [r*S_loc, (r+1)*S_loc)."""
    S = x.shape[0]
    out = np.zeros((padded_len(S, P),) + x.shape[1:], dtype=x.dtype)
    out[:S] = x
    return out


# ---------------------------------------------------------------------------
# Zigzag partition (Megatron-LM PR #7 "GLM-5.2 131k context parallelism",
# closing comment: upstream replaced the contiguous partition by a zigzag
# one).  Reading: the padded sequence is cut into 2P equal chunks and rank r
# holds chunks r and 2P-1-r, in that order, so every rank gets the same
# share of causal work.  Rows stay global everywhere else: positions,
# documents and the head layout after the all-to-all are in global order.
# ---------------------------------------------------------------------------


def zigzag_padded_len(S: int, P: int) -> int:
    """S rounded up to a multiple of 2P (2P equal chunks)."""
    return -(-S // (2 * P)) * (2 * P)


def zigzag_order(S_pad: int, P: int) -> np.ndarray:
    """order[i] = global row held at row i of the sharded buffer, i = r*2C + s
    for rank r and local row s (C = S_pad / 2P)."""
    C = S_pad // (2 * P)
    order = np.zeros(S_pad, dtype=np.int64)
    for r in range(P):
        for s in range(2 * C):
            chunk = r if s < C else 2 * P - 1 - r
            order[r * 2 * C + s] = chunk * C + (s % C)
    return order


def shard_pad_zigzag(x: np.ndarray, P: int) -> np.ndarray:
    """[S][H][D] -> [S_pad][H][D] in zigzag shard order; rows of the padding
    (global rows >= S) are zero."""
    S = x.shape[0]
    S_pad = zigzag_padded_len(S, P)
    out = np.zeros((S_pad,) + x.shape[1:], dtype=x.dtype)
    for i, t in enumerate(zigzag_order(S_pad, P)):
        if t < S:
            out[i] = x[t]
    return out


def seq_to_head_zigzag(x_seq: np.ndarray, P: int) -> np.ndarray:
    """All-to-all from zigzag shards to head groups in global row order:
    X_head[g][order[i]][j] = X_seq[i][g*H/P + j]."""
    S_pad, H, D = x_seq.shape
    hp = H // P
    out = np.zeros((P, S_pad, hp, D), dtype=x_seq.dtype)
    order = zigzag_order(S_pad, P)
    for i in range(S_pad):
        for g in range(P):
            out[g, order[i]] = x_seq[i, g * hp:(g + 1) * hp]
    return out


def head_to_seq_zigzag(x_head: np.ndarray) -> np.ndarray:
    """Inverse of :func:`seq_to_head_zigzag`."""
    P, S_pad, hp, D = x_head.shape
    out = np.zeros((S_pad, P * hp, D), dtype=x_head.dtype)
    order = zigzag_order(S_pad, P)
    for i in range(S_pad):
        for g in range(P):
            out[i, g * hp:(g + 1) * hp] = x_head[g, order[i]]
    return out


def positions_docs(S: int, P: int, cu=None, S_pad=None):
    """Absolute positions and document ids of the S_pad padded rows.

    Row t < S belongs to document d with cu[d] <= t < cu[d+1] and has position
    t - cu[d] (positions restart at documents, never at shard boundaries).
    Pad rows t >= S get doc -1 and keep counting inside the last document, so
    the RoPE table has to cover S_pad positions.  ``cu=None`` means one
    document [0, S).  ``S_pad`` overrides the padded length (the zigzag
    partition pads to a multiple of 2P).
    """
    S_pad = padded_len(S, P) if S_pad is None else S_pad
    cu = np.array([0, S], dtype=np.int64) if cu is None else np.asarray(cu, np.int64)
    assert cu[0] == 0 and cu[-1] == S and np.all(np.diff(cu) >= 0)
    pos = np.zeros(S_pad, dtype=np.int64)
    doc = np.full(S_pad, -1, dtype=np.int64)
    for d in range(len(cu) - 1):
        a, b = int(cu[d]), int(cu[d + 1])
        pos[a:b] = np.arange(b - a)
        doc[a:b] = d
    last_start = int(cu[-2]) if len(cu) >= 2 else 0
    pos[S:] = np.arange(S, S_pad) - last_start
    return pos, doc


# ---------------------------------------------------------------------------
# Ulysses all-to-all as a permutation (SpecForge #728 Modifications)
#   rank r holds X_seq[r] = rows [r*S_loc, (r+1)*S_loc) with all H heads;
#   after the all-to-all, rank g holds all S_pad rows of heads
#   [g*H/P, (g+1)*H/P):  X_head[g][r*S_loc + s][j] = X_seq[r][s][g*H/P + j]
# ---------------------------------------------------------------------------


def seq_to_head_loops(x_seq: np.ndarray, P: int) -> np.ndarray:
    """The all-to-all written as an explicit index loop (small inputs only)."""
    S_pad, H, D = x_seq.shape
    S_loc, hp = S_pad // P, H // P
    out = np.zeros((P, S_pad, hp, D), dtype=x_seq.dtype)
    for g in range(P):
        for r in range(P):
            for s in range(S_loc):
                for j in range(hp):
                    out[g, r * S_loc + s, j, :] = x_seq[r * S_loc + s, g * hp + j, :]
    return out


def seq_to_head(x_seq: np.ndarray, P: int) -> np.ndarray:
    """[S_pad][H][D] -> [P][S_pad][H/P][D], the same permutation as the loop."""
    S_pad, H, D = x_seq.shape
    assert S_pad % P == 0 and H % P == 0
    return np.ascontiguousarray(
        x_seq.reshape(S_pad, P, H // P, D).transpose(1, 0, 2, 3))


def head_to_seq(x_head: np.ndarray) -> np.ndarray:
    """Inverse all-to-all: [P][S_pad][H/P][D] -> [S_pad][H][D]."""
    P, S_pad, hp, D = x_head.shape
    return np.ascontiguousarray(x_head.transpose(1, 0, 2, 3).reshape(S_pad, P * hp, D))


def check_heads(P: int, Hq: int, Hkv: int) -> None:
    """SpecForge #728 Modifications: Q and KV head counts must be divisible by
    the Ulysses degree (and GQA needs Hkv | Hq)."""
    if P < 1 or Hq % P or Hkv % P or Hq % Hkv:
        raise ValueError(f"head counts Hq={Hq}, Hkv={Hkv} not divisible by P={P}")


# ---------------------------------------------------------------------------
# RoPE tables: rotate-half pairs (i, i + D/2), inv_freq_i = base^(-2i/D);
# YaRN (Peng et al. 2023, sec. 3.2 "NTK-by-parts" ramp, sec. 3.4 mscale)
# ---------------------------------------------------------------------------


def rope_inv_freq(D: int, base: float, factor: float = 1.0, orig_ctx: int = 0,
                  beta_fast: float = 32.0, beta_slow: float = 1.0) -> np.ndarray:
    """Per-pair angular frequencies (fp64), YaRN-blended when factor != 1.

    Pair i rotates at inv_freq_i = base^(-2i/D).  With YaRN, pairs whose
    wavelength fits many times into the original context (high frequency)
    keep their frequency, pairs whose wavelength exceeds it are slowed down by
    ``factor``, and a linear ramp over the pair index blends the two between
    the correction dimensions of beta_fast and beta_slow rotations.
    """
    i = np.arange(D // 2, dtype=np.float64)
    extrap = np.array([base ** (-2.0 * k / D) for k in i], dtype=np.float64)
    if factor == 1.0:
        return extrap
    interp = extrap / factor

    def corr_dim(n_rot):  # pair index whose wavelength gives n_rot turns
        return D * math.log(orig_ctx / (n_rot * 2 * math.pi)) / (2 * math.log(base))

    lo = max(math.floor(corr_dim(beta_fast)), 0)
    hi = min(math.ceil(corr_dim(beta_slow)), D - 1)
    if hi == lo:
        hi = lo + 0.001
    ramp = np.clip((i - lo) / (hi - lo), 0.0, 1.0)      # 0: keep, 1: interpolate
    return extrap - ramp * (extrap - interp)


def rope_mscale(factor: float) -> float:
    """YaRN attention temperature factor applied to cos and sin."""
    return 1.0 if factor <= 1.0 else 0.1 * math.log(factor) + 1.0


def rope_cos_sin(n_pos: int, D: int, base: float, factor: float = 1.0,
                 orig_ctx: int = 0):
    """fp64 cos/sin tables [n_pos][D/2] of theta = pos * inv_freq (scaled)."""
    inv = rope_inv_freq(D, base, factor, orig_ctx)
    theta = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    m = rope_mscale(factor)
    return np.cos(theta) * m, np.sin(theta) * m


def rope_table_f32(n_pos: int, D: int, base: float, factor: float = 1.0,
                   orig_ctx: int = 0) -> np.ndarray:
    """The table both paths consume: float32 [n_pos][D/2][2] = (cos, sin),
    each the fp64 value rounded to fp32."""
    c, s = rope_cos_sin(n_pos, D, base, factor, orig_ctx)
    return np.ascontiguousarray(np.stack([c, s], axis=-1).astype(np.float32))


def rope_rotate(x: np.ndarray, pos: np.ndarray, cos: np.ndarray, sin: np.ndarray,
                inverse: bool = False) -> np.ndarray:
    """Exact fp64 rotation of x[..., T, H, D] at positions pos[T].

    y[i] = x[i] cos - x[i+D/2] sin,  y[i+D/2] = x[i+D/2] cos + x[i] sin;
    ``inverse`` rotates by -theta (the transpose, used to carry gradients
    back to pre-RoPE Q and K)."""
    D = x.shape[-1]
    h = D // 2
    c = cos[pos][:, None, :]
    s = sin[pos][:, None, :] * (-1.0 if inverse else 1.0)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_recipe_bf16(x_bits: np.ndarray, pos: np.ndarray, table: np.ndarray,
                     inverse: bool = False) -> np.ndarray:
    """Rotation of bf16 x[T, H, D] with the fp32 table, rounded to bf16.

    The pages fix no rounding, so both paths use this one, operation by
    operation in IEEE fp32 (no fused multiply-add):
        a = x1*c, b = x2*s, y1 = bf16(a - b)
        e = x2*c, f = x1*s, y2 = bf16(e + f)
    with s negated for the inverse rotation.
    """
    D = x_bits.shape[-1]
    h = D // 2
    x = (np.asarray(x_bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    c = table[pos, :, 0][:, None, :].astype(np.float32)
    s = table[pos, :, 1][:, None, :].astype(np.float32)
    if inverse:
        s = -s
    x1, x2 = x[..., :h], x[..., h:]
    y1 = np.float32(x1 * c) - np.float32(x2 * s)
    y2 = np.float32(x2 * c) + np.float32(x1 * s)
    return f32_to_bf16(np.concatenate([y1, y2], axis=-1))


# ---------------------------------------------------------------------------
# Attention (SpecForge #728 Modifications: local attention per head group;
# Accuracy Test: parity with full-sequence attention).  Causal GQA with a
# per-document mask: key u is visible to query t iff doc(u) == doc(t) >= 0
# and u <= t.  Q head h reads KV head h // (Hq/Hkv).
#
# causal=False is the bidirectional variant (zhtmike/verl PR #45 "[trainer]
# feat: support sequence parallel", What does this PR do: Ulysses SP for the
# Diffusers SDPA attention, whose attention mask masks the padding added for
# SP alignment): key u is visible to query t iff doc(u) == doc(t) >= 0, so
# pad rows (doc -1) are never keys and every row of a document sees the
# whole document.
# ---------------------------------------------------------------------------

_ROW_CHUNK = 2048  # rows are evaluated in independent chunks to bound memory


def _visible(rows: np.ndarray, doc: np.ndarray, causal: bool = True) -> np.ndarray:
    u = np.arange(doc.shape[0])
    dr = doc[rows][:, None]
    vis = (dr >= 0) & (doc[None, :] == dr)
    return vis & (u[None, :] <= rows[:, None]) if causal else vis


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, doc: np.ndarray,
                   rows: np.ndarray, scale: float, causal: bool = True):
    """Softmax attention of single-head fp64 q[T,D], k, v for the query rows
    ``rows``.  Returns O[len(rows), D] and LSE[len(rows)] (natural log; -inf
    and O=0 for a row with no visible key)."""
    rows = np.asarray(rows, dtype=np.int64)
    s = (q[rows] @ k.T) * scale
    vis = _visible(rows, doc, causal)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    o = np.zeros((rows.shape[0], q.shape[1]))
    o[has] = (e[has] @ v) / l[has, None]
    lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    return o, lse


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, doc: np.ndarray,
                  scale: float, causal: bool = True):
    """q[T][Hq][D], k/v[T][Hkv][D] (fp64) -> O[T][Hq][D], LSE[Hq][T]."""
    T, Hq, D = q.shape
    G = Hq // k.shape[1]
    o = np.zeros((T, Hq, D))
    lse = np.zeros((Hq, T))
    for h in range(Hq):
        for a in range(0, T, _ROW_CHUNK):
            rows = np.arange(a, min(T, a + _ROW_CHUNK))
            o[rows, h], lse[h, rows] = attention_rows(q[:, h], k[:, h // G],
                                                      v[:, h // G], doc, rows, scale, causal)
    return o, lse


# ---------------------------------------------------------------------------
# Ring attention over R virtual ring ranks (SpecForge #728 configures a
# Ulysses x Ring mesh, "Ulysses=8 / Ring=1" in its run; verl #45 builds a
# (dp, ring, ulysses) mesh).  Reading: the key/value rows are cut into R
# contiguous chunks; each ring step attends to one chunk and yields a
# partial (O, LSE) normalised within that chunk; partials are merged with
# the log-sum-exp combine  LSE = ln sum_i exp(LSE_i),
# O = sum_i exp(LSE_i - LSE) O_i, which gives the attention over all chunks.
# ---------------------------------------------------------------------------


def attention_window(q, k, v, doc, scale, k_lo, k_hi, causal=True):
    """Attention of every query row over the keys in rows [k_lo, k_hi) only
    (mask as usual): q[T][Hq][D], k/v[T][Hkv][D] -> O[T][Hq][D], LSE[Hq][T]
    (LSE -inf and O = 0 for a row with no visible key in the window)."""
    T = q.shape[0]
    inside = (np.arange(T) >= k_lo) & (np.arange(T) < k_hi)
    doc_w = np.where(inside, doc, -2)          # keys outside the window match no row
    o = np.zeros(q.shape)
    lse = np.zeros((q.shape[1], T))
    G = q.shape[1] // k.shape[1]
    for h in range(q.shape[1]):
        for a in range(0, T, _ROW_CHUNK):
            rows = np.arange(a, min(T, a + _ROW_CHUNK))
            sc = (q[rows, h] @ k[:, h // G].T) * scale
            vis = _visible(rows, doc, causal) & (doc_w[None, :] == doc[rows][:, None])
            sc = np.where(vis, sc, -np.inf)
            m = sc.max(axis=1)
            has = np.isfinite(m)
            m_safe = np.where(has, m, 0.0)
            e = np.exp(sc - m_safe[:, None])
            l = e.sum(axis=1)
            o[rows[has], h] = (e[has] @ v[:, h // G]) / l[has, None]
            lse[h, rows] = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    return o, lse


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Log-sum-exp combine of two partial results (O[T][H][D], LSE[H][T])."""
    lse = np.logaddexp(lse_a, lse_b)
    fin = np.isfinite(lse)
    w_a = np.where(fin, np.exp(np.where(fin, lse_a - np.where(fin, lse, 0.0), -np.inf)), 0.0)
    w_b = np.where(fin, np.exp(np.where(fin, lse_b - np.where(fin, lse, 0.0), -np.inf)), 0.0)
    o = o_a * w_a.T[:, :, None] + o_b * w_b.T[:, :, None]
    return o, lse


def ring_fwd(q, k, v, doc, scale, R, causal=True):
    """Attention as R ring steps over contiguous key chunks, merged."""
    T = q.shape[0]
    L = -(-T // R)
    o = np.zeros(q.shape)
    lse = np.full((q.shape[1], T), -np.inf)
    for c in range(R):
        o_c, lse_c = attention_window(q, k, v, doc, scale, c * L, min(T, (c + 1) * L), causal)
        o, lse = lse_merge(o, lse, o_c, lse_c)
    return o, lse


def attention_bwd_head(q, k, v, do, doc, scale, rows=None, causal=True):
    """Gradients of L = sum(O * dO) for one head (fp64, q/k/v/do [T][D]).

    With P = softmax rows:  dV = P^T dO;  dP = dO V^T;
    dS = P * (dP - rowsum(P * dP))  (softmax Jacobian);
    dQ = scale dS K;  dK = scale dS^T Q.
    ``rows`` restricts the query rows that contribute (default all); dK/dV are
    then partial sums over those rows and dQ is returned for them only."""
    T, D = q.shape
    rows_all = np.arange(T) if rows is None else np.asarray(rows, np.int64)
    dq = np.zeros((rows_all.shape[0], D))
    dk = np.zeros((T, D))
    dv = np.zeros((T, D))
    for a in range(0, rows_all.shape[0], _ROW_CHUNK):
        rows = rows_all[a:a + _ROW_CHUNK]
        s = (q[rows] @ k.T) * scale
        vis = _visible(rows, doc, causal)
        s = np.where(vis, s, -np.inf)
        m = s.max(axis=1)
        has = np.isfinite(m)
        m_safe = np.where(has, m, 0.0)
        e = np.where(vis, np.exp(s - m_safe[:, None]), 0.0)
        l = e.sum(axis=1)
        p = e / np.where(has, l, 1.0)[:, None]
        dp = do[rows] @ v.T
        dsm = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        dq[a:a + rows.shape[0]] = scale * (dsm @ k)
        dk += scale * (dsm.T @ q[rows])
        dv += p.T @ do[rows]
    return dq, dk, dv


def attention_bwd_keys(q, k, v, do, doc, scale, keys, rows=None, causal=True):
    """dK and dV of one head (fp64, q/k/v/do [T][D]) at the key rows ``keys``
    only, summed over the query rows ``rows`` (default: all rows).

    The same gradient as :func:`attention_bwd_head`, evaluated without the
    full T x T matrices: each query row t first gets its own softmax
    denominator LSE_t and output O_t from :func:`attention_rows` (over every
    key it sees), and delta_t = dO_t . O_t, which equals sum_u P_tu dP_tu
    because O_t = sum_u P_tu v_u.  Then, for the chosen keys only,
    P_tu = exp(scale q_t.k_u - LSE_t), dP_tu = dO_t.v_u,
    dS_tu = P_tu (dP_tu - delta_t), dK_u = scale sum_t dS_tu q_t and
    dV_u = sum_t P_tu dO_t.  Row sets may be split into chunks and the
    partial sums added (each row's terms depend on that row alone), which is
    how long sequences are evaluated in parallel."""
    T, D = q.shape
    keys = np.asarray(keys, np.int64)
    rows_all = np.arange(T) if rows is None else np.asarray(rows, np.int64)
    dk = np.zeros((keys.shape[0], D))
    dv = np.zeros((keys.shape[0], D))
    for a in range(0, rows_all.shape[0], _ROW_CHUNK):
        rows = rows_all[a:a + _ROW_CHUNK]
        # causal: no key after the chunk's last row is visible to it
        hi = int(rows.max()) + 1 if causal else T
        o, lse = attention_rows(q[:hi], k[:hi], v[:hi], doc[:hi], rows, scale, causal)
        delta = (do[rows] * o).sum(axis=1)
        vis = _visible(rows, doc, causal)[:, keys]
        has = np.isfinite(lse)
        s = (q[rows] @ k[keys].T) * scale
        p = np.where(vis & has[:, None],
                     np.exp(s - np.where(has, lse, 0.0)[:, None]), 0.0)
        dp = do[rows] @ v[keys].T
        ds = p * (dp - delta[:, None])
        dk += scale * (ds.T @ q[rows])
        dv += p.T @ do[rows]
    return dk, dv


def attention_bwd(q, k, v, do, doc, scale, causal=True):
    """All heads: q/do[T][Hq][D], k/v[T][Hkv][D] -> dq, dk, dv (fp64).  dK and
    dV of a KV head are summed over the Hq/Hkv query heads that read it."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros((T, Hkv, D))
    dv = np.zeros((T, Hkv, D))
    for h in range(Hq):
        a, b, c = attention_bwd_head(q[:, h], k[:, h // G], v[:, h // G], do[:, h],
                                     doc, scale, causal=causal)
        dq[:, h] = a
        dk[:, h // G] += b
        dv[:, h // G] += c
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Whole forward + backward, two ways.  Both return, for the S valid rows:
# O[S][Hq][D], LSE[Hq][S], loss = sum(O * dO), and the gradients of the loss
# with respect to the pre-RoPE, sequence-sharded Q, K, V.
# ---------------------------------------------------------------------------


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


def full_sequence(q, k, v, do, cu, cos, sin, scale, causal=True):
    """Reference computation on the unsharded sequence (fp64 inputs [S][H][D])."""
    S = q.shape[0]
    pos, doc = positions_docs(S, 1, cu)
    qr = rope_rotate(q, pos, cos, sin)
    kr = rope_rotate(k, pos, cos, sin)
    o, lse = attention_fwd(qr, kr, v, doc, scale, causal)
    dqr, dkr, dv = attention_bwd(qr, kr, v, do, doc, scale, causal)
    dq = rope_rotate(dqr, pos, cos, sin, inverse=True)
    dk = rope_rotate(dkr, pos, cos, sin, inverse=True)
    return dict(o=o, lse=lse, loss=float((o * do).sum()), dq=dq, dk=dk, dv=dv)


def ulysses(q, k, v, do, cu, cos, sin, scale, P, causal=True, zigzag=False):
    """The Ulysses path: pad and shard, all-to-all to head groups, RoPE at
    absolute positions, attention per head group, all-to-all back.  With
    ``zigzag`` the shards are the zigzag partition (the head layout is the
    same global-order layout either way)."""
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    check_heads(P, Hq, Hkv)
    if zigzag:
        pos, doc = positions_docs(S, P, cu, S_pad=zigzag_padded_len(S, P))
        to_head = lambda x: seq_to_head_zigzag(shard_pad_zigzag(x, P), P)  # noqa: E731
        to_seq = lambda x: head_to_seq_zigzag(x)[np.argsort(zigzag_order(x.shape[1], P))]  # noqa: E731,E501
    else:
        pos, doc = positions_docs(S, P, cu)
        to_head = lambda x: seq_to_head(shard_pad(x, P), P)  # noqa: E731
        to_seq = head_to_seq
    heads = {n: to_head(x) for n, x in (("q", q), ("k", k), ("v", v), ("do", do))}
    S_pad = pos.shape[0]
    hq, hkv = Hq // P, Hkv // P
    o_h = np.zeros((P, S_pad, hq, D))
    lse_h = np.zeros((P, hq, S_pad))
    dq_h = np.zeros((P, S_pad, hq, D))
    dk_h = np.zeros((P, S_pad, hkv, D))
    dv_h = np.zeros((P, S_pad, hkv, D))
    for g in range(P):   # each virtual rank works on its own head group
        qg = rope_rotate(heads["q"][g], pos, cos, sin)
        kg = rope_rotate(heads["k"][g], pos, cos, sin)
        vg = heads["v"][g]
        o_h[g], lse_h[g] = attention_fwd(qg, kg, vg, doc, scale, causal)
        a, b, c = attention_bwd(qg, kg, vg, heads["do"][g], doc, scale, causal)
        dq_h[g] = rope_rotate(a, pos, cos, sin, inverse=True)
        dk_h[g] = rope_rotate(b, pos, cos, sin, inverse=True)
        dv_h[g] = c
    # back to sequence layout, then to global row order for the comparison
    o = to_seq(o_h)[:S]
    lse = lse_h.reshape(Hq, S_pad)[:, :S]
    return dict(o=o, lse=lse, loss=float((o * do).sum()),
                dq=to_seq(dq_h)[:S], dk=to_seq(dk_h)[:S], dv=to_seq(dv_h)[:S])


# ---------------------------------------------------------------------------
# Context parallelism with a K/V all-gather (basetenlabs/Megatron-LM PR #7,
# "GLM-5.2 131k context parallelism", Purpose: the CP forward all-gathers the
# KV of every rank and its backward reduce-scatters dKV; contiguous
# partition; positions from the global cu_seqlens).  Reading: P ranks hold
# contiguous shards of S_loc padded rows of Q, K, V and dO with all heads, so
# no head count has to be divisible by P.  Each rank rotates its own rows at
# their global positions, gathers the K/V shards of all ranks in rank order
# (which is the global row order), attends its query rows to every key with
# the global causal / document mask, and in the backward computes dQ for its
# rows and partial dK, dV over all key rows from its query rows alone.  The
# partials of all ranks are summed and each rank keeps its own shard's rows
# (the reduce-scatter), which it rotates back.
# ---------------------------------------------------------------------------


def allgather_cp(q, k, v, do, cu, cos, sin, scale, P, causal=True, return_partials=False):
    """The K/V all-gather CP path over P virtual ranks (fp64 inputs [S][H][D]).
    Returns the same dict as :func:`full_sequence`; with ``return_partials``
    also each rank's pre-reduction dK/dV partials, [P][S_pad][Hkv][D] in the
    rotated frame."""
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    if Hkv < 1 or Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    pos, doc = positions_docs(S, P, cu)
    S_pad = pos.shape[0]
    S_loc = S_pad // P
    rows = [np.arange(r * S_loc, (r + 1) * S_loc) for r in range(P)]
    padded = {n: shard_pad(x, P) for n, x in (("q", q), ("k", k), ("v", v), ("do", do))}
    shard = {n: [x[rows[r]] for r in range(P)] for n, x in padded.items()}
    # every rank rotates its own Q and K rows at their global positions
    q_rot = [rope_rotate(shard["q"][r], pos[rows[r]], cos, sin) for r in range(P)]
    k_rot = [rope_rotate(shard["k"][r], pos[rows[r]], cos, sin) for r in range(P)]
    # all-gather: the K/V shards of all ranks, concatenated in rank order
    k_all = np.concatenate(k_rot)
    v_all = np.concatenate(shard["v"])
    o_sh, lse_sh, dq_sh = [], [], []
    dk_part = np.zeros((P, S_pad, Hkv, D))
    dv_part = np.zeros((P, S_pad, Hkv, D))
    for r in range(P):
        # rank r's query rows sit at their global rows, so that the mask and
        # the causal order use global indices
        q_glob = np.zeros((S_pad, Hq, D))
        do_glob = np.zeros((S_pad, Hq, D))
        q_glob[rows[r]] = q_rot[r]
        do_glob[rows[r]] = shard["do"][r]
        o_r = np.zeros((S_loc, Hq, D))
        lse_r = np.zeros((Hq, S_loc))
        dq_r = np.zeros((S_loc, Hq, D))
        for h in range(Hq):
            kh, vh = k_all[:, h // G], v_all[:, h // G]
            o_r[:, h], lse_r[h] = attention_rows(q_glob[:, h], kh, vh, doc, rows[r], scale,
                                                 causal)
            a, b, c = attention_bwd_head(q_glob[:, h], kh, vh, do_glob[:, h], doc, scale,
                                         rows=rows[r], causal=causal)
            dq_r[:, h] = a
            dk_part[r, :, h // G] += b
            dv_part[r, :, h // G] += c
        o_sh.append(o_r)
        lse_sh.append(lse_r)
        dq_sh.append(rope_rotate(dq_r, pos[rows[r]], cos, sin, inverse=True))
    # reduce-scatter: sum the partials of all ranks, rank r keeps its rows
    dk_sum = dk_part.sum(axis=0)
    dv_sum = dv_part.sum(axis=0)
    dk_sh = [rope_rotate(dk_sum[rows[r]], pos[rows[r]], cos, sin, inverse=True)
             for r in range(P)]
    dv_sh = [dv_sum[rows[r]] for r in range(P)]
    o = np.concatenate(o_sh)[:S]
    out = dict(o=o, lse=np.concatenate(lse_sh, axis=1)[:, :S], loss=float((o * do).sum()),
               dq=np.concatenate(dq_sh)[:S], dk=np.concatenate(dk_sh)[:S],
               dv=np.concatenate(dv_sh)[:S])
    if return_partials:
        out["dk_part"], out["dv_part"] = dk_part, dv_part
    return out
