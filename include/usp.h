/*
 * usp.h -- C ABI of the GB300-native Ulysses sequence-parallel (USP)
 * attention hot path.
 *
 * What the calls compute (sources: SpecForge PR #728 "feat(dspark): add
 * Ulysses sequence parallel training", sections Modifications and Accuracy
 * Test; basetenlabs/Megatron-LM PR #7 "GLM-5.2 131k context parallelism",
 * section Purpose; zhtmike/verl PR #45 "[trainer] feat: support sequence
 * parallel"):
 *
 *   A sequence of S tokens (one document, or packed documents described by
 *   cu_seqlens) is padded to S_pad = ceil(S/P)*P rows and split into P
 *   contiguous shards of S_loc = S_pad/P rows, one per Ulysses rank.  The P
 *   ranks are P virtual shards in this GPU's memory.  The all-to-all that
 *   gives every rank the full sequence of its own head group becomes an
 *   on-device permutation; RoPE is applied at absolute positions on the way.
 *   Each head group then runs causal GQA attention (forward and backward);
 *   the inverse permutation returns outputs and gradients to sequence
 *   shards.  The result equals full-sequence attention.
 *
 * Layouts (all bf16 tensors row-major, element type __nv_bfloat16):
 *   "seq"  : x_seq[t][h][d],            t in [0,S_pad), h in [0,H), d in [0,D)
 *            shard r is rows [r*S_loc, (r+1)*S_loc)
 *   "head" : x_head[g][t][j][d],        g in [0,P), j in [0,H/P)
 *            x_head[g][t][j] holds global head h = g*(H/P) + j of row t;
 *            it is the concatenation of the P all-to-all messages rank g
 *            receives.
 *   lse    : float  [P][Hq/P][S_pad]    natural-log softmax denominators
 *   pos,doc: int32  [S_pad]             absolute position / document id
 *                                       (doc = -1 on pad rows)
 *   rope_cs: float  [rope_len][D/2][2]  (cos, sin) of pair i at position p;
 *                                       pair i rotates elements (i, i+D/2)
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless the name ends in _host.  The
 *     caller owns every buffer; no call allocates or frees device memory.
 *     Buffer sizes are not passed and cannot be checked: each buffer must
 *     hold the layout its argument documents for the given usp_dims (the
 *     Python pipeline objects check tensor shapes before calling).
 *   - Tensor buffers must be 16-byte aligned; D must be 64 or 128.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and return after enqueueing.  Arguments are validated
 *     on the host before anything is launched; a call that returns an error
 *     has launched nothing.
 *   - Byte offsets are 64-bit throughout, so S_pad*H*D may exceed 2^31.
 *   - Device-side waits are bounded.  A kernel that gives up records it in
 *     a device status word and exits; usp_device_status() reports it.
 *   - Calls keep no state between invocations and may be issued from any
 *     host thread (the library's per-process lookups -- device addresses of
 *     its status word and scratch, the SM count -- are made race-free).
 */
#ifndef USP_H_
#define USP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define USP_ABI_VERSION 1

typedef enum {
  USP_OK = 0,
  USP_ERR_INVALID_ARG = 1,          /* NULL/misaligned pointer, bad size, bad table */
  USP_ERR_HEADS_NOT_DIVISIBLE = 2,  /* P does not divide Hq or Hkv, or Hkv does not divide Hq */
  USP_ERR_UNSUPPORTED = 3,          /* e.g. D not in {64,128} */
  USP_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
  USP_ERR_TIMEOUT = 5,              /* a device-side wait gave up (see usp_device_status) */
  USP_ERR_OUT_OF_BOUNDS = 6         /* a debug build's index guard stopped an access
                                       outside a buffer's extent (see usp_debug_build) */
} usp_status;

/* Problem description shared by all calls. */
typedef struct {
  int64_t S;                        /* valid tokens (sum of document lengths), >= 0 */
  int32_t P;                        /* Ulysses degree = number of virtual shards, >= 1.
                                       P = 1 is one shard holding every row: its
                                       head layout is the sequence layout, so
                                       the calls then rotate in place of the
                                       all-to-all and attend over [S][H][D]
                                       buffers directly -- the data path of
                                       context parallelism with a K/V
                                       all-gather (Megatron-LM #7, Purpose),
                                       which takes any Hkv dividing Hq */
  int32_t Hq, Hkv, D;               /* query heads, key/value heads, head dim (64|128) */
  const int32_t* cu_seqlens;        /* device int32 [n_docs+1], global document
                                       boundaries; NULL => one document [0,S) */
  const int32_t* cu_seqlens_host;   /* optional host copy of cu_seqlens; when given
                                       it is checked (cu[0]=0, non-decreasing,
                                       cu[n_docs]=S) before launch */
  int32_t n_docs;                   /* documents in cu_seqlens (ignored if NULL) */
  int32_t causal;                   /* 1: causal within each document; 0:
                                       bidirectional within each document
                                       (verl PR #45, Diffusers SDPA under
                                       Ulysses); anything else is
                                       USP_ERR_INVALID_ARG */
  float scale;                      /* softmax scale; 0 => 1/sqrt(D) */
  int32_t zigzag;                   /* shard layout of the sequence-sharded
                                       buffers: 0 contiguous (rank r holds
                                       rows [r*S_pad/P, (r+1)*S_pad/P)); 1
                                       zigzag (Megatron-LM #7, closing
                                       comment): S_pad is a multiple of 2P,
                                       the sequence is cut into 2P equal
                                       chunks and rank r holds chunks r and
                                       2P-1-r, in that order.  Anything else
                                       is USP_ERR_INVALID_ARG.  Head-layout
                                       buffers, pos and doc are in global row
                                       order either way. */
} usp_dims;

/*
 * usp_pad_shard -- shard + pad one activation tensor and (optionally) emit
 * the absolute positions and document ids of the padded rows.
 * (SpecForge #728, Modifications: inputs and absolute positions are sharded
 * and padded across the SP group; verl #45: sequence lengths padded for SP
 * alignment; Megatron-LM #7, Purpose: positions from the GLOBAL cu_seqlens.)
 *
 *   x     [S][H][D] bf16 (input, unpadded)
 *   x_seq [S_pad][H][D] bf16 (output): rows < S copied, rows >= S zero;
 *         with zigzag, row r*(S_pad/P) + s holds global row
 *         (s < C ? r : 2P-1-r)*C + s % C, C = S_pad/(2P).
 *         x_seq == x is allowed for the contiguous layout (in place; the
 *         buffer must hold S_pad rows), not for zigzag.
 *   pos   [S_pad] int32 or NULL: t - cu[doc(t)]; pad rows keep counting in
 *         the last document.
 *   doc   [S_pad] int32 or NULL: document index of row t, -1 for pad rows.
 * x may be NULL with H = 0 to emit only pos/doc.
 */
usp_status usp_pad_shard(const usp_dims* dims, const void* x, int32_t H,
                         void* x_seq, int32_t* pos, int32_t* doc, void* stream);

/*
 * usp_seq_to_head_rope -- the seq->head all-to-all (SpecForge #728,
 * Modifications: separate Q/K/V all-to-alls before local attention), fused
 * with RoPE at absolute positions.
 *
 *   x_seq  [S_pad][H][D] bf16 (shard layout of dims->zigzag) -> x_head
 *          [P][S_pad][H/P][D] bf16 in global row order.  Padding rows
 *          (global rows t >= S) are zero by definition: their head-layout
 *          rows are written as zeros and x_seq is never read there.  In the
 *          contiguous layout x_seq may therefore be the caller's unpadded
 *          [S][H][D] tensor itself (no usp_pad_shard copy is needed; that
 *          call then only emits pos/doc).
 *   rope_mode 0: plain permutation (V, dO); pos/rope_cs may be NULL.
 *   rope_mode 1: rotate every (d, d+D/2) pair of row t by the table entry
 *                at pos[t]; -1 rotates by the negated angle.
 *   Rounding (identical in every kernel): with x1 = x[d], x2 = x[d+D/2],
 *   (c, s) = rope_cs[pos][d] and s negated for mode -1, in IEEE fp32 with
 *   no fused multiply-add:  y[d] = bf16_rne(x1*c - x2*s),
 *                           y[d+D/2] = bf16_rne(x2*c + x1*s).
 *   rope_len must be >= S_pad (or > the largest position when
 *   cu_seqlens_host is given): USP_ERR_INVALID_ARG otherwise
 *   (Megatron-LM #7, Purpose: the table must cover the padded length).
 */
usp_status usp_seq_to_head_rope(const usp_dims* dims, const void* x_seq, int32_t H,
                                const int32_t* pos, const float* rope_cs,
                                int64_t rope_len, int32_t rope_mode,
                                void* x_head, void* stream);

/*
 * usp_attn_fwd -- local causal GQA attention of every head group
 * (SpecForge #728, Modifications: local attention after the all-to-all;
 * Accuracy Test: equal to full-sequence attention).
 *
 * For group g, local query head j (global h = g*Hq/P + j, reading KV head
 * h / (Hq/Hkv)) and row t with doc(t) >= 0:
 *   O[t]   = sum_{u in M(t)} softmax_u(scale * q_t . k_u) v_u
 *   LSE[t] = ln sum_{u in M(t)} exp(scale * q_t . k_u)
 *   M(t)   = { u : doc(u) == doc(t), u <= t }         (causal = 1)
 *   M(t)   = { u : doc(u) == doc(t) }                 (causal = 0)
 * Rows with doc(t) = -1 (padding) get O = 0 and LSE = -inf, and are never
 * keys (in the bidirectional case this is the padding mask).
 *   q_h [P][S_pad][Hq/P][D], k_h/v_h [P][S_pad][Hkv/P][D] (bf16, head layout)
 *   doc [S_pad] int32 (from usp_pad_shard)
 *   o_h [P][S_pad][Hq/P][D] bf16 (output), lse [P][Hq/P][S_pad] fp32 (output)
 * fp32 accumulation; no atomics, so the result is deterministic.
 */
usp_status usp_attn_fwd(const usp_dims* dims, const void* q_h, const void* k_h,
                        const void* v_h, const int32_t* doc, void* o_h, float* lse,
                        void* stream);

/*
 * usp_attn_fwd_window -- usp_attn_fwd over the keys in rows [k_lo, k_hi)
 * only: one ring step of ring attention (SpecForge #728 runs a Ulysses x
 * Ring mesh, "Ulysses=8 / Ring=1"; verl #45 builds a (dp, ring, ulysses)
 * mesh).  M(t) of usp_attn_fwd is cut to k_lo <= u < k_hi; O is normalised
 * within the window and LSE is the log-sum-exp over it (O = 0, LSE = -inf
 * for a row that sees no key in the window).  Same arguments and errors as
 * usp_attn_fwd, plus 0 <= k_lo <= k_hi <= S_pad (else USP_ERR_INVALID_ARG).
 * Partial results of disjoint windows combine with usp_lse_merge into the
 * attention over their union.
 */
usp_status usp_attn_fwd_window(const usp_dims* dims, const void* q_h, const void* k_h,
                               const void* v_h, const int32_t* doc, int64_t k_lo,
                               int64_t k_hi, void* o_h, float* lse, void* stream);

/*
 * usp_lse_merge -- merge one partial attention result into an accumulator
 * (the log-sum-exp combine of ring attention):
 *   LSE = ln(exp(LSE_acc) + exp(LSE_part)),
 *   O   = exp(LSE_acc - LSE) O_acc + exp(LSE_part - LSE) O_part,
 * a -inf term weighing 0 (both -inf: O = 0, LSE = -inf).
 *   o_acc   [P][S_pad][Hq/P][D] fp32, in/out (ignored as input if first)
 *   lse_acc [P][Hq/P][S_pad] fp32, in/out (ignored as input if first)
 *   o_part  [P][S_pad][Hq/P][D] bf16, lse_part [P][Hq/P][S_pad] fp32: the
 *           outputs of usp_attn_fwd_window
 *   first   1: the accumulator is set to the partial result; 0: merged
 *   o_out   NULL, or [P][S_pad][Hq/P][D] bf16 that receives the merged O
 *           (the last step writes the forward's O this way; lse_acc is
 *           then its LSE)
 * All pointers 16-byte aligned.  fp32 arithmetic; deterministic.
 */
usp_status usp_lse_merge(const usp_dims* dims, float* o_acc, float* lse_acc,
                         const void* o_part, const float* lse_part, int32_t first,
                         void* o_out, void* stream);

/*
 * usp_attn_bwd -- gradients of loss L with dL/dO = dO through usp_attn_fwd
 * (SpecForge #728, Accuracy Test: gradient parity with full-sequence
 * attention; verl #45: SP and non-SP fwd+bwd agree).
 *   P_tu = exp(scale q_t.k_u - LSE_t),   delta_t = sum_d dO_t[d] O_t[d]
 *   dV_u = sum_t P_tu dO_t,   dS_tu = P_tu (dO_t.v_u - delta_t)
 *   dQ_t = scale sum_u dS_tu k_u,   dK_u = scale sum_t dS_tu q_t
 * dK/dV of a KV head are summed over the Hq/Hkv query heads reading it.
 * Gradients of pad rows are 0.
 *   inputs as usp_attn_fwd plus o_h, lse (its outputs) and do_h
 *   (upstream gradient, head layout); outputs dq_h, dk_h, dv_h (bf16,
 *   head layout, same shapes as q_h, k_h, v_h).
 *   workspace: device scratch of at least usp_attn_bwd_workspace(dims)
 *   bytes, 256-byte aligned, not used concurrently by another call.
 * dQ is produced by a query-stationary pass and dK/dV by a key-stationary
 * pass, so no atomics are used and the result is deterministic.
 */
usp_status usp_attn_bwd(const usp_dims* dims, const void* q_h, const void* k_h,
                        const void* v_h, const void* o_h, const float* lse,
                        const void* do_h, const int32_t* doc, void* dq_h, void* dk_h,
                        void* dv_h, void* workspace, size_t ws_bytes, void* stream);

/*
 * usp_attn_bwd_noalloc -- usp_attn_bwd for callers that cannot allocate
 * device memory when they call it: for example a serving process whose
 * caching allocator reserved the device memory up front, or a runtime whose
 * policy forbids cudaMalloc after start-up (it synchronises the device and
 * can fail once memory is exhausted or fragmented).  The pages have no
 * counterpart; this is a convenience of this library.
 *
 * Same arguments, results and errors as usp_attn_bwd, minus the workspace:
 * the scratch lives in one fixed 32 MiB device array inside the library
 * (held by every GPU that loads the library until the process exits).  The
 * call allocates nothing and calls no allocating routine.  The results are
 * bitwise those of usp_attn_bwd.
 *   - Limit: usp_attn_bwd_workspace(dims) must be <= 32 MiB, i.e.
 *     P * (Hq/P) * ceil(S_pad/128)*128 <= 4194304; larger problems return
 *     USP_ERR_UNSUPPORTED before anything touches the device.
 *   - The first call on a device looks up the array's device address with
 *     that device current.  With CUDA's default lazy module loading that
 *     first lookup is also what loads the library's backward module and
 *     gives the array its 32 MiB of device memory, so make the first call
 *     on each device before reserving the rest of the device's memory (or
 *     run with CUDA_MODULE_LOADING=EAGER), and before any stream capture.
 *   - All calls on one device share that device's array, which keeps the
 *     previous call's contents (every entry a call reads, it first
 *     rewrites).  Calls on the same device that overlap on the GPU --
 *     whether issued on different streams or from different host threads --
 *     race on the array and give wrong gradients: order them on one stream.
 *     Calls on other devices use their own copy of the array.
 */
usp_status usp_attn_bwd_noalloc(const usp_dims* dims, const void* q_h, const void* k_h,
                                const void* v_h, const void* o_h, const float* lse,
                                const void* do_h, const int32_t* doc, void* dq_h, void* dk_h,
                                void* dv_h, void* stream);

/* Bytes of workspace usp_attn_bwd needs for dims: two fp32 arrays of
 * P*(Hq/P) rows of ceil(S_pad/128)*128 entries (delta_t and LSE_t*log2(e)),
 * each rounded up to 256 bytes.  Returns 0 for invalid dims and SIZE_MAX
 * when the size does not fit in size_t. */
size_t usp_attn_bwd_workspace(const usp_dims* dims);

/*
 * usp_head_to_seq -- the inverse all-to-all (head -> seq) that returns the
 * attention output to sequence shards after local attention (SpecForge #728,
 * Modifications), and carries the gradients back the same way; rope_mode -1
 * applies the inverse rotation so that dQ and dK become gradients of the
 * pre-RoPE inputs, which is what the gradient-parity criterion compares
 * (SpecForge #728, Accuracy Test).  Same rounding and table rules as
 * usp_seq_to_head_rope.
 *   x_head [P][S_pad][H/P][D] bf16 -> x_seq [S_pad][H][D] bf16 (shard
 *          layout of dims->zigzag), x_seq[t][g*H/P + j] = x_head[g][t][j]
 */
usp_status usp_head_to_seq(const usp_dims* dims, const void* x_head, int32_t H,
                           const int32_t* pos, const float* rope_cs, int64_t rope_len,
                           int32_t rope_mode, void* x_seq, void* stream);

/*
 * usp_rope_table -- fill a HOST buffer out_host[n_pos][D/2][2] with
 * fp32(cos(theta)*m), fp32(sin(theta)*m) where theta = p * inv_freq_i is
 * evaluated in double, inv_freq_i = base^(-2i/D), and for yarn_factor > 1
 * the YaRN blend (Peng et al. 2023): pairs turning more than 32 times over
 * yarn_orig_ctx keep inv_freq_i, pairs turning less than once use
 * inv_freq_i / yarn_factor, a linear ramp over i in between, and
 * m = 0.1 ln(yarn_factor) + 1 (m = 1 without YaRN).
 * (SpecForge #728, Accuracy Test: Qwen3-8B with "YaRN context 131,072".)
 */
usp_status usp_rope_table(int64_t n_pos, int32_t D, double base, double yarn_factor,
                          int32_t yarn_orig_ctx, float* out_host);

/*
 * usp_device_status -- synchronise `stream`, then report and clear the
 * device status word: USP_ERR_TIMEOUT if a kernel's bounded wait gave up,
 * USP_ERR_OUT_OF_BOUNDS if a debug build's index guard fired,
 * USP_ERR_INVALID_ARG if a kernel met a position outside the RoPE table,
 * USP_ERR_CUDA if the stream reported an error, else USP_OK.
 */
usp_status usp_device_status(void* stream);

/*
 * usp_debug_build -- 1 if this library was built with index guards: every
 * global-memory index a kernel computes is checked against the extent that
 * usp_dims implies for its buffer, and an out-of-range index sets a status
 * bit (reported as USP_ERR_OUT_OF_BOUNDS) and skips the access instead of
 * reading or writing out of bounds; 0 for the release build.  (The kind of
 * fault this catches -- an out-of-range RoPE table gather that fired a
 * device-side assert -- is the one basetenlabs/Megatron-LM PR #7, Purpose,
 * describes.)
 */
int usp_debug_build(void);

/*
 * usp_selftest_bounded_wait -- diagnostic for the failure-detection path:
 * launches one CTA whose thread waits, exactly as the attention kernels
 * wait, on an mbarrier that nothing completes, giving up after limit_us
 * microseconds (1..1000000; USP_ERR_INVALID_ARG otherwise).  The CTA then
 * records a timeout in the device status word and exits, so the next
 * usp_device_status() returns USP_ERR_TIMEOUT (and clears it) while the
 * CUDA context stays usable.  Nothing traps, faults or hangs.
 */
usp_status usp_selftest_bounded_wait(int32_t limit_us, void* stream);

const char* usp_status_string(usp_status s);
int usp_abi_version(void);

/* Number of kernels this library has launched in this process so far
 * (all devices, all streams); a diagnostic for benchmarks. */
uint64_t usp_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* USP_H_ */
