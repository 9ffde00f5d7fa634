// Shard/pad and the Ulysses all-to-all as on-device permutations.
//
// SpecForge PR #728 "feat(dspark): add Ulysses sequence parallel training",
// Modifications: sequences and their absolute positions are padded and
// sharded across the SP group, and Q, K, V each go through an all-to-all
// before local attention.  On one GPU the P ranks are P slices of the same
// buffer, so the all-to-all is the permutation
//     x_head[g][t][j][:] = x_seq[t][g*H/P + j][:]
// in which every (t, g) pair moves one contiguous chunk of H/P*D elements.
// RoPE at the absolute position pos[t] (Megatron-LM PR #7 "GLM-5.2 131k
// context parallelism", Purpose: positions from the global cu_seqlens) is
// fused into the permutation, so each element is read once and written once.
//
// Both kernels are HBM-bound: 16-byte loads and stores, streaming cache
// hints, one warp per token row and several heads in flight per thread.
// The sequence-sharded side may use the zigzag shard layout; it only
// changes which buffer row holds global row t.
#include "usp_common.cuh"

namespace {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// Zigzag shard layout (Megatron-LM PR #7, closing comment): 2P chunks of C
// rows; rank r holds chunks r and 2P-1-r, so global row t sits at row
// zz_row(t) of the sharded buffer and buffer row i holds global row
// zz_global(i).  C = 0 means the contiguous layout (row t at row t).
__device__ __forceinline__ int64_t zz_row(int64_t t, int64_t C, int P) {
  if (C == 0) return t;
  const int64_t c = t / C, s = t - c * C;
  return c < P ? c * 2 * C + s : (2 * P - 1 - c) * 2 * C + C + s;
}
__device__ __forceinline__ int64_t zz_global(int64_t i, int64_t C, int P) {
  if (C == 0) return i;
  const int64_t r = i / (2 * C), s = i - r * 2 * C;
  return s < C ? r * C + s : (2 * P - 1 - r) * C + (s - C);
}

// ---------------------------------------------------------------- pad/shard
// Largest d in [0, n_docs) with cu[d] <= t (documents are contiguous).
__device__ __forceinline__ int doc_of(const int32_t* cu, int n_docs, int64_t t) {
  int lo = 0, hi = n_docs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// x holds n_valid_vec 16-byte vectors (S rows), y n_total_vec (S_pad rows).
__global__ void __launch_bounds__(256) pad_shard_kernel(
    const uint4* __restrict__ x, uint4* __restrict__ y, int64_t n_valid_vec,
    int64_t n_total_vec, int inplace, int32_t* __restrict__ pos, int32_t* __restrict__ doc,
    const int32_t* __restrict__ cu, int n_docs, int64_t S, int64_t S_pad, int64_t row_vec,
    int64_t zz_chunk, int P, unsigned* status) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  if (zz_chunk == 0) {
    for (int64_t i = i0; i < n_total_vec; i += stride) {
      if (!usp::in_bounds(i, 1, n_total_vec, status)) continue;
      if (i < n_valid_vec) {
        if (!inplace && usp::in_bounds(i, 1, n_valid_vec, status))
          st_stream(y + i, ld_stream(x + i));
      } else {
        st_stream(y + i, zero);
      }
    }
  } else {   // buffer row r holds global row zz_global(r): a row permutation
    for (int64_t i = i0; i < n_total_vec; i += stride) {
      const int64_t r = i / row_vec, c = i - r * row_vec;
      const int64_t t = zz_global(r, zz_chunk, P);
      const int64_t xi = t * row_vec + c;
      if (!usp::in_bounds(i, 1, n_total_vec, status)) continue;
      st_stream(y + i, t < S && usp::in_bounds(xi, 1, n_valid_vec, status) ? ld_stream(x + xi)
                                                                           : zero);
    }
  }
  if (pos == nullptr && doc == nullptr) return;
  for (int64_t t = i0; t < S_pad; t += stride) {
    int d = 0;
    int64_t start = 0;
    if (cu != nullptr) {
      d = doc_of(cu, n_docs, t);
      if (usp::in_bounds(d, 1, n_docs + 1, status)) start = __ldg(cu + d);
    }
    if (!usp::in_bounds(t, 1, S_pad, status)) continue;
    if (pos) pos[t] = (int32_t)(t - start);
    if (doc) doc[t] = t < S ? d : -1;
  }
}

// ------------------------------------------------------------------ repack
// One warp per R consecutive token rows.  A head's D elements are covered
// by D/16 threads; thread `sub` owns pairs [8*sub, 8*sub+8): elements
// d = 8*sub..+7 and their rotation partners d + D/2.  32/(D/16) heads are
// processed per step and kUnroll steps (spread over the R rows) are loaded
// before any is stored.  R = 2 for tensors with few heads, so that a warp
// still has kUnroll loads in flight behind each row's dependent position
// and table reads.
// Seq -> head: padding rows (global t >= S) are zero by definition, so the
// kernel takes zeros for them instead of reading the source (which
// therefore only needs its valid rows: the caller's unpadded tensor serves
// directly in the contiguous layout, and no padding copy is made).  The
// zeros still go through the rotation, so a padding row's output is
// bitwise what rotating a zero-filled row gives (signed zeros included).
template <int D, int MODE, bool TO_HEAD, int R>
__global__ void __launch_bounds__(256) repack_kernel(
    const bf16* __restrict__ src, bf16* __restrict__ dst, const int32_t* __restrict__ pos,
    const float* __restrict__ cs, int64_t rope_len, int64_t S, int64_t S_pad, int H, int hp,
    unsigned* status, int64_t zz_chunk, int P) {
  constexpr int TPH = D / 16;
  constexpr int HPI = 32 / TPH;
  constexpr int kUnroll = 4;
  constexpr int UPR = kUnroll / R;               // load steps per row
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPH;
  const int slot = lane / TPH;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // element extents usp_dims implies (index guards of debug builds): the
  // sequence side holds S rows, or all S_pad rows of zigzag shards
  const int64_t n_seq = (TO_HEAD && zz_chunk == 0 ? S : S_pad) * H * (int64_t)D;
  const int64_t n_head = S_pad * H * (int64_t)D;
  const int64_t n_src = TO_HEAD ? n_seq : n_head, n_dst = TO_HEAD ? n_head : S_pad * H * (int64_t)D;

  for (int64_t tb = warp * R; tb < S_pad; tb += nwarps * R) {
    int64_t srow[R];
    bool pad_row[R], zero_row[R];
    float c[R][8], s[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t t = tb + r;
      srow[r] = zz_row(t, zz_chunk, P);            // row of t in the sharded buffer
      pad_row[r] = TO_HEAD && t >= S;              // zeros, nothing read
      zero_row[r] = false;
      if (MODE != 0 && t < S_pad) {
        const int p = usp::in_bounds(t, 1, S_pad, status) ? __ldg(pos + t) : -1;
        if (p < 0 || (int64_t)p >= rope_len) {
          if (lane == 0) usp::set_status(status, usp::kErrRopeRange);
          zero_row[r] = true;
#pragma unroll
          for (int i = 0; i < 8; ++i) { c[r][i] = 0.f; s[r][i] = 0.f; }
        } else {
          const int64_t toff = ((int64_t)p * (D / 2) + 8 * sub) * 2;
          const bool tab_ok = usp::in_bounds(toff, 16, rope_len * D, status);
          const float4* tp = reinterpret_cast<const float4*>(cs + (tab_ok ? toff : 0));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 v = __ldg(tp + i);
            c[r][2 * i] = v.x; s[r][2 * i] = v.y; c[r][2 * i + 1] = v.z; s[r][2 * i + 1] = v.w;
          }
          if (MODE < 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) s[r][i] = -s[r][i];
          }
        }
      }
    }
    for (int h0 = slot; h0 < H; h0 += UPR * HPI) {
      uint4 lo[kUnroll], hi[kUnroll];
      int64_t doff[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int r = u / UPR;
        const int h = h0 + (u % UPR) * HPI;
        const int64_t t = tb + r;
        doff[u] = -1;
        if (h < H && t < S_pad) {
          const int g = h / hp, j = h - g * hp;
          const int64_t seq_off = (srow[r] * H + h) * (int64_t)D;
          const int64_t head_off = (((int64_t)g * S_pad + t) * hp + j) * (int64_t)D;
          const bf16* sp = src + (TO_HEAD ? seq_off : head_off);
          doff[u] = TO_HEAD ? head_off : seq_off;
          const int64_t so = (TO_HEAD ? seq_off : head_off) + 8 * sub;
          if (pad_row[r] || !usp::in_bounds(so, 8, n_src, status) ||
              !usp::in_bounds(so + D / 2, 8, n_src, status)) {
            lo[u] = make_uint4(0, 0, 0, 0);
            hi[u] = lo[u];
          } else {
            lo[u] = ld_stream(sp + 8 * sub);
            hi[u] = ld_stream(sp + D / 2 + 8 * sub);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (doff[u] < 0) continue;
        const int r = u / UPR;
        uint4 a = lo[u], b = hi[u];
        if (MODE != 0) {
          const bf16* xa = reinterpret_cast<const bf16*>(&lo[u]);
          const bf16* xb = reinterpret_cast<const bf16*>(&hi[u]);
          bf16* ya = reinterpret_cast<bf16*>(&a);
          bf16* yb = reinterpret_cast<bf16*>(&b);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float x1 = __bfloat162float(xa[i]);
            const float x2 = __bfloat162float(xb[i]);
            // IEEE fp32, each product rounded separately (no FMA contraction)
            const float y1 = __fsub_rn(__fmul_rn(x1, c[r][i]), __fmul_rn(x2, s[r][i]));
            const float y2 = __fadd_rn(__fmul_rn(x2, c[r][i]), __fmul_rn(x1, s[r][i]));
            ya[i] = __float2bfloat16_rn(y1);
            yb[i] = __float2bfloat16_rn(y2);
          }
          if (zero_row[r]) { a = make_uint4(0, 0, 0, 0); b = a; }
        }
        bf16* dp = dst + doff[u];
        if (usp::in_bounds(doff[u] + 8 * sub, 8, n_dst, status) &&
            usp::in_bounds(doff[u] + D / 2 + 8 * sub, 8, n_dst, status)) {
          st_stream(dp + 8 * sub, a);
          st_stream(dp + D / 2 + 8 * sub, b);
        }
      }
    }
  }
}

int repack_grid(int64_t S_pad, int rows_per_warp) {
  int64_t blocks = (S_pad + 8 * rows_per_warp - 1) / (8 * rows_per_warp);  // 8 warps per block
  const int64_t cap = 152 * 64;      // grid-stride beyond this
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

template <int D, bool TO_HEAD, int R>
cudaError_t launch_rows(int mode, const bf16* src, bf16* dst, const int32_t* pos,
                        const float* cs, int64_t rope_len, int64_t S, int64_t S_pad, int H,
                        int hp, unsigned* status, int64_t zz, int P, cudaStream_t st) {
  const int grid = repack_grid(S_pad, R);
  if (mode == 0)
    repack_kernel<D, 0, TO_HEAD, R><<<grid, 256, 0, st>>>(src, dst, pos, cs, rope_len, S, S_pad,
                                                          H, hp, status, zz, P);
  else if (mode > 0)
    repack_kernel<D, 1, TO_HEAD, R><<<grid, 256, 0, st>>>(src, dst, pos, cs, rope_len, S, S_pad,
                                                          H, hp, status, zz, P);
  else
    repack_kernel<D, -1, TO_HEAD, R><<<grid, 256, 0, st>>>(src, dst, pos, cs, rope_len, S,
                                                           S_pad, H, hp, status, zz, P);
  usp_count_launches(1);
  return cudaGetLastError();
}

// Two rows per warp when one row's heads fill at most half of a warp's
// load steps (H <= 2 * 32/(D/16)), one otherwise.
template <int D, bool TO_HEAD>
cudaError_t launch_mode(int mode, const bf16* src, bf16* dst, const int32_t* pos,
                        const float* cs, int64_t rope_len, int64_t S, int64_t S_pad, int H,
                        int hp, unsigned* status, int64_t zz, int P, cudaStream_t st) {
  constexpr int HPI = 32 / (D / 16);
  if (H <= 2 * HPI)
    return launch_rows<D, TO_HEAD, 2>(mode, src, dst, pos, cs, rope_len, S, S_pad, H, hp, status,
                                      zz, P, st);
  return launch_rows<D, TO_HEAD, 1>(mode, src, dst, pos, cs, rope_len, S, S_pad, H, hp, status,
                                    zz, P, st);
}

}  // namespace

cudaError_t usp_launch_pad_shard(const usp::Geometry& g, const void* x, int H, void* x_seq,
                                 int32_t* pos, int32_t* doc, const int32_t* cu, int n_docs,
                                 cudaStream_t st) {
  const int64_t row_vec = (int64_t)H * g.D * 2 / 16;
  const int64_t n_valid = (x_seq != nullptr) ? g.S * row_vec : 0;
  const int64_t n_total = (x_seq != nullptr) ? g.S_pad * row_vec : 0;
  int64_t work = n_total > g.S_pad ? n_total : g.S_pad;
  int64_t blocks = (work + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (blocks < 1) blocks = 1;
  pad_shard_kernel<<<(int)blocks, 256, 0, st>>>(
      reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(x_seq), n_valid, n_total,
      x == x_seq ? 1 : 0, pos, doc, cu, n_docs, g.S, g.S_pad, row_vec, g.zz_chunk, g.P,
      g.status);
  usp_count_launches(1);
  return cudaGetLastError();
}

cudaError_t usp_launch_repack(const usp::Geometry& g, const void* src, int H, const int32_t* pos,
                              const float* rope_cs, int64_t rope_len, int rope_mode,
                              bool to_head, void* dst, cudaStream_t st) {
  const int hp = H / g.P;
  const bf16* s = reinterpret_cast<const bf16*>(src);
  bf16* d = reinterpret_cast<bf16*>(dst);
  const int64_t zz = g.zz_chunk;
  if (g.D == 128)
    return to_head ? launch_mode<128, true>(rope_mode, s, d, pos, rope_cs, rope_len, g.S, g.S_pad,
                                            H, hp, g.status, zz, g.P, st)
                   : launch_mode<128, false>(rope_mode, s, d, pos, rope_cs, rope_len, g.S,
                                             g.S_pad, H, hp, g.status, zz, g.P, st);
  return to_head ? launch_mode<64, true>(rope_mode, s, d, pos, rope_cs, rope_len, g.S, g.S_pad, H,
                                         hp, g.status, zz, g.P, st)
                 : launch_mode<64, false>(rope_mode, s, d, pos, rope_cs, rope_len, g.S, g.S_pad,
                                          H, hp, g.status, zz, g.P, st);
}
