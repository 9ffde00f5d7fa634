// Causal per-document GQA attention, forward and backward, on CUDA cores.
//
// One thread per query row (forward, dQ) or per key row (dK, dV), fp32
// arithmetic, K/V or Q/dO tiles staged in shared memory.  This is the
// straightforward form of the computation (SpecForge PR #728, Modifications:
// local attention per head group after the all-to-all; Accuracy Test: loss
// and gradient parity with full-sequence attention).
#include "usp_common.cuh"

namespace {

using bf16 = __nv_bfloat16;
constexpr int kRows = 128;   // rows per block (one thread each)
constexpr int kTile = 32;    // staged rows of the other operand
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Args {
  const bf16 *q, *k, *v, *o, *dout;
  const float* lse;
  const int32_t *doc, *cu;
  bf16 *o_out, *dq, *dk, *dv;
  float *lse_out, *delta;
  int64_t S, S_pad;
  int hq, hkv, G;
  float scale;
};

__device__ __forceinline__ int64_t doc_start(const Args& a, int64_t t) {
  const int d = a.doc[t];
  if (d < 0) return -1;
  return a.cu ? (int64_t)a.cu[d] : 0;
}
__device__ __forceinline__ int64_t doc_end(const Args& a, int64_t t) {
  const int d = a.doc[t];
  if (d < 0) return -1;
  return a.cu ? (int64_t)a.cu[d + 1] : a.S;
}
template <int D>
__device__ __forceinline__ void load_rows_T(float* dstT, const bf16* base, int64_t row0,
                                            int64_t S_pad, int64_t row_stride) {
  // dstT[d * kRows + r] = base[(row0 + r) * row_stride + d]
  for (int idx = threadIdx.x; idx < kRows * D; idx += blockDim.x) {
    const int r = idx / D, d = idx - r * D;
    const int64_t t = row0 + r;
    dstT[d * kRows + r] = t < S_pad ? __bfloat162float(base[t * row_stride + d]) : 0.f;
  }
}

template <int D>
__device__ __forceinline__ void load_tile(float* dst, const bf16* base, int64_t row0,
                                          int64_t S_pad, int64_t row_stride) {
  for (int idx = threadIdx.x; idx < kTile * D; idx += blockDim.x) {
    const int r = idx / D, d = idx - r * D;
    const int64_t t = row0 + r;
    dst[r * D + d] = t < S_pad ? __bfloat162float(base[t * row_stride + d]) : 0.f;
  }
}

// ------------------------------------------------------------------ forward
template <int D>
__global__ void __launch_bounds__(kRows) fwd_kernel(Args a) {
  extern __shared__ float sm[];
  float* qT = sm;                    // [D][kRows]
  float* ks = qT + D * kRows;        // [kTile][D]
  float* vs = ks + kTile * D;        // [kTile][D]
  const int bh = blockIdx.y;
  const int g = bh / a.hq, j = bh - g * a.hq, jk = j / a.G;
  const int64_t t0 = (int64_t)blockIdx.x * kRows;
  const int64_t t = t0 + threadIdx.x;
  const int64_t qs = (int64_t)a.hq * D, ks_ = (int64_t)a.hkv * D;
  const bf16* qb = a.q + ((int64_t)g * a.S_pad * a.hq + j) * D;
  const bf16* kb = a.k + ((int64_t)g * a.S_pad * a.hkv + jk) * D;
  const bf16* vb = a.v + ((int64_t)g * a.S_pad * a.hkv + jk) * D;
  load_rows_T<D>(qT, qb, t0, a.S_pad, qs);
  const bool row_ok = t < a.S_pad;
  const int64_t ds = row_ok ? doc_start(a, t) : -1;
  // first key any row of this block can see
  int64_t lo = -1;
  {
    __shared__ int64_t s_lo;
    if (threadIdx.x == 0) {
      int64_t v = -1;
      for (int64_t r = t0; r < t0 + kRows && r < a.S_pad; ++r) {
        const int64_t d0 = doc_start(a, r);
        if (d0 >= 0) { v = d0; break; }
      }
      s_lo = v;
    }
    __syncthreads();
    lo = s_lo;
  }
  const float sl2 = a.scale * kLog2e;
  float m = -INFINITY, l = 0.f, acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;
  const int64_t hi = min(t0 + kRows, a.S_pad);
  if (lo >= 0) {
    for (int64_t u0 = (lo / kTile) * kTile; u0 < hi; u0 += kTile) {
      __syncthreads();
      load_tile<D>(ks, kb, u0, a.S_pad, ks_);
      load_tile<D>(vs, vb, u0, a.S_pad, ks_);
      __syncthreads();
      float sc[kTile];
      float mt = -INFINITY;
#pragma unroll 4
      for (int uu = 0; uu < kTile; ++uu) {
        const int64_t u = u0 + uu;
        float s = -INFINITY;
        if (ds >= 0 && u >= ds && u <= t) {
          float dot = 0.f;
#pragma unroll 16
          for (int d = 0; d < D; ++d) dot = fmaf(qT[d * kRows + threadIdx.x], ks[uu * D + d], dot);
          s = dot * sl2;
        }
        sc[uu] = s;
        mt = fmaxf(mt, s);
      }
      const float mn = fmaxf(m, mt);
      if (mn == -INFINITY) continue;
      const float corr = exp2f(m - mn);
      l *= corr;
#pragma unroll
      for (int d = 0; d < D; ++d) acc[d] *= corr;
      for (int uu = 0; uu < kTile; ++uu) {
        const float p = exp2f(sc[uu] - mn);
        if (p == 0.f) continue;
        l += p;
#pragma unroll
        for (int d = 0; d < D; ++d) acc[d] = fmaf(p, vs[uu * D + d], acc[d]);
      }
      m = mn;
    }
  }
  if (!row_ok) return;
  bf16* op = a.o_out + (((int64_t)g * a.S_pad + t) * a.hq + j) * D;
  const bool valid = l > 0.f;
  const float inv = valid ? 1.f / l : 0.f;
#pragma unroll
  for (int d = 0; d < D; ++d) op[d] = __float2bfloat16_rn(acc[d] * inv);
  a.lse_out[((int64_t)g * a.hq + j) * a.S_pad + t] = valid ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// --------------------------------------------------------- delta = dO . O
template <int D>
__global__ void delta_kernel(Args a) {
  const int64_t n = (int64_t)gridDim.y * a.S_pad;  // gridDim.y = P * hq
  const int bh = blockIdx.y;
  const int g = bh / a.hq, j = bh - g * a.hq;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < a.S_pad;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t off = (((int64_t)g * a.S_pad + t) * a.hq + j) * D;
    float s = 0.f;
    for (int d = 0; d < D; ++d)
      s = fmaf(__bfloat162float(a.dout[off + d]), __bfloat162float(a.o[off + d]), s);
    a.delta[((int64_t)g * a.hq + j) * a.S_pad + t] = s;
  }
  (void)n;
}

// ---------------------------------------------------------------------- dQ
template <int D>
__global__ void __launch_bounds__(kRows) dq_kernel(Args a) {
  extern __shared__ float sm[];
  float* qT = sm;                     // [D][kRows]
  float* dT = qT + D * kRows;         // [D][kRows] dO rows
  float* ks = dT + D * kRows;         // [kTile][D]
  float* vs = ks + kTile * D;         // [kTile][D]
  const int bh = blockIdx.y;
  const int g = bh / a.hq, j = bh - g * a.hq, jk = j / a.G;
  const int64_t t0 = (int64_t)blockIdx.x * kRows;
  const int64_t t = t0 + threadIdx.x;
  const int64_t qs = (int64_t)a.hq * D, ks_ = (int64_t)a.hkv * D;
  const int64_t qoff = ((int64_t)g * a.S_pad * a.hq + j) * D;
  load_rows_T<D>(qT, a.q + qoff, t0, a.S_pad, qs);
  load_rows_T<D>(dT, a.dout + qoff, t0, a.S_pad, qs);
  const bf16* kb = a.k + ((int64_t)g * a.S_pad * a.hkv + jk) * D;
  const bf16* vb = a.v + ((int64_t)g * a.S_pad * a.hkv + jk) * D;
  const bool row_ok = t < a.S_pad;
  const int64_t ds = row_ok ? doc_start(a, t) : -1;
  const int64_t li = ((int64_t)g * a.hq + j) * a.S_pad + t;
  const float lse2 = (row_ok && ds >= 0) ? a.lse[li] * kLog2e : 0.f;
  const float dl = (row_ok && ds >= 0) ? a.delta[li] : 0.f;
  __shared__ int64_t s_lo;
  if (threadIdx.x == 0) {
    int64_t v = -1;
    for (int64_t r = t0; r < t0 + kRows && r < a.S_pad; ++r) {
      const int64_t d0 = doc_start(a, r);
      if (d0 >= 0) { v = d0; break; }
    }
    s_lo = v;
  }
  __syncthreads();
  const int64_t lo = s_lo;
  const float sl2 = a.scale * kLog2e;
  float acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;
  const int64_t hi = min(t0 + kRows, a.S_pad);
  if (lo >= 0) {
    for (int64_t u0 = (lo / kTile) * kTile; u0 < hi; u0 += kTile) {
      __syncthreads();
      load_tile<D>(ks, kb, u0, a.S_pad, ks_);
      load_tile<D>(vs, vb, u0, a.S_pad, ks_);
      __syncthreads();
      for (int uu = 0; uu < kTile; ++uu) {
        const int64_t u = u0 + uu;
        if (!(ds >= 0 && u >= ds && u <= t)) continue;
        float s = 0.f, dp = 0.f;
#pragma unroll 16
        for (int d = 0; d < D; ++d) {
          s = fmaf(qT[d * kRows + threadIdx.x], ks[uu * D + d], s);
          dp = fmaf(dT[d * kRows + threadIdx.x], vs[uu * D + d], dp);
        }
        const float p = exp2f(s * sl2 - lse2);
        const float dsv = p * (dp - dl);
#pragma unroll
        for (int d = 0; d < D; ++d) acc[d] = fmaf(dsv, ks[uu * D + d], acc[d]);
      }
    }
  }
  if (!row_ok) return;
  bf16* out = a.dq + (((int64_t)g * a.S_pad + t) * a.hq + j) * D;
#pragma unroll
  for (int d = 0; d < D; ++d) out[d] = __float2bfloat16_rn(ds >= 0 ? acc[d] * a.scale : 0.f);
}

// --------------------------------------------------------------- dK or dV
template <int D, bool DK>
__global__ void __launch_bounds__(kRows) dkv_kernel(Args a) {
  extern __shared__ float sm[];
  float* kT = sm;                    // [D][kRows] own K rows
  float* vT = kT + D * kRows;        // [D][kRows] own V rows (dK only)
  float* qsm = vT + D * kRows;       // [kTile][D]
  float* dsm = qsm + kTile * D;      // [kTile][D]
  float* lsm = dsm + kTile * D;      // [kTile] lse*log2e
  float* dlm = lsm + kTile;          // [kTile] delta
  const int bh = blockIdx.y;         // (g, jk)
  const int g = bh / a.hkv, jk = bh - g * a.hkv;
  const int64_t u0 = (int64_t)blockIdx.x * kRows;
  const int64_t u = u0 + threadIdx.x;
  const int64_t ks_ = (int64_t)a.hkv * D, qs = (int64_t)a.hq * D;
  const int64_t koff = ((int64_t)g * a.S_pad * a.hkv + jk) * D;
  load_rows_T<D>(kT, a.k + koff, u0, a.S_pad, ks_);
  if (DK) load_rows_T<D>(vT, a.v + koff, u0, a.S_pad, ks_);
  const bool row_ok = u < a.S_pad;
  const int64_t ue = row_ok ? doc_end(a, u) : -1;   // queries t in [u, ue)
  __shared__ int64_t s_hi;
  if (threadIdx.x == 0) {
    int64_t v = -1;
    for (int64_t r = min(u0 + kRows, a.S_pad) - 1; r >= u0; --r) {
      const int64_t e = doc_end(a, r);
      if (e >= 0) { v = e; break; }
    }
    s_hi = v;
  }
  __syncthreads();
  const int64_t hi = s_hi;
  const float sl2 = a.scale * kLog2e;
  float acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;
  if (hi >= 0) {
    for (int i = 0; i < a.G; ++i) {
      const int j = jk * a.G + i;
      const int64_t qoff = ((int64_t)g * a.S_pad * a.hq + j) * D;
      const int64_t lbase = ((int64_t)g * a.hq + j) * a.S_pad;
      for (int64_t tq0 = u0; tq0 < hi; tq0 += kTile) {
        __syncthreads();
        load_tile<D>(qsm, a.q + qoff, tq0, a.S_pad, qs);
        load_tile<D>(dsm, a.dout + qoff, tq0, a.S_pad, qs);
        if (threadIdx.x < kTile) {
          const int64_t tt = tq0 + threadIdx.x;
          const bool ok = tt < a.S_pad && a.doc[tt] >= 0;
          lsm[threadIdx.x] = ok ? a.lse[lbase + tt] * kLog2e : 0.f;
          dlm[threadIdx.x] = ok ? a.delta[lbase + tt] : 0.f;
        }
        __syncthreads();
        for (int tt = 0; tt < kTile; ++tt) {
          const int64_t t = tq0 + tt;
          if (!(row_ok && ue >= 0 && t >= u && t < ue)) continue;
          float s = 0.f, dp = 0.f;
#pragma unroll 16
          for (int d = 0; d < D; ++d) {
            s = fmaf(kT[d * kRows + threadIdx.x], qsm[tt * D + d], s);
            if (DK) dp = fmaf(vT[d * kRows + threadIdx.x], dsm[tt * D + d], dp);
          }
          const float p = exp2f(s * sl2 - lsm[tt]);
          if (DK) {
            const float dsv = p * (dp - dlm[tt]);
#pragma unroll
            for (int d = 0; d < D; ++d) acc[d] = fmaf(dsv, qsm[tt * D + d], acc[d]);
          } else {
#pragma unroll
            for (int d = 0; d < D; ++d) acc[d] = fmaf(p, dsm[tt * D + d], acc[d]);
          }
        }
      }
    }
  }
  if (!row_ok) return;
  bf16* out = (DK ? a.dk : a.dv) + (((int64_t)g * a.S_pad + u) * a.hkv + jk) * D;
  const float f = DK ? a.scale : 1.f;
#pragma unroll
  for (int d = 0; d < D; ++d) out[d] = __float2bfloat16_rn(ue >= 0 ? acc[d] * f : 0.f);
}

template <int D>
cudaError_t fwd_launch(const Args& a, int P, cudaStream_t st) {
  const size_t smem = (size_t)(D * kRows + 2 * kTile * D) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.S_pad + kRows - 1) / kRows), (unsigned)(P * a.hq));
  fwd_kernel<D><<<grid, kRows, smem, st>>>(a);
  usp_count_launches(1);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_launch(const Args& a, int P, cudaStream_t st) {
  dim3 gd((unsigned)((a.S_pad + 255) / 256 < 1024 ? (a.S_pad + 255) / 256 : 1024), (unsigned)(P * a.hq));
  delta_kernel<D><<<gd, 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smq = (size_t)(2 * D * kRows + 2 * kTile * D) * sizeof(float);
  e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smq);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.S_pad + kRows - 1) / kRows), (unsigned)(P * a.hq));
  dq_kernel<D><<<grid, kRows, smq, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t smk = (size_t)(2 * D * kRows + 2 * kTile * D + 2 * kTile) * sizeof(float);
  e = cudaFuncSetAttribute(dkv_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dkv_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
  if (e != cudaSuccess) return e;
  dim3 gk((unsigned)((a.S_pad + kRows - 1) / kRows), (unsigned)(P * a.hkv));
  dkv_kernel<D, true><<<gk, kRows, smk, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dkv_kernel<D, false><<<gk, kRows, smk, st>>>(a);
  usp_count_launches(4);
  return cudaGetLastError();
}

Args make_args(const usp::Geometry& g) {
  Args a{};
  a.S = g.S; a.S_pad = g.S_pad; a.hq = g.hq; a.hkv = g.hkv; a.G = g.G; a.scale = g.scale;
  return a;
}

}  // namespace

cudaError_t usp_launch_attn_fwd_simt(const usp::Geometry& g, const void* q, const void* k,
                                const void* v, const int32_t* doc, const int32_t* cu,
                                void* o, float* lse, cudaStream_t st) {
  Args a = make_args(g);
  a.q = (const bf16*)q; a.k = (const bf16*)k; a.v = (const bf16*)v;
  a.doc = doc; a.cu = cu; a.o_out = (bf16*)o; a.lse_out = lse;
  return g.D == 128 ? fwd_launch<128>(a, g.P, st) : fwd_launch<64>(a, g.P, st);
}

size_t usp_attn_bwd_ws_bytes(const usp::Geometry& g) {
  const size_t delta = (size_t)g.P * g.hq * g.S_pad * sizeof(float);
  const size_t dqacc = (size_t)g.P * g.S_pad * g.hq * g.D * sizeof(float);
  return ((delta + 255) / 256) * 256 + dqacc;
}

cudaError_t usp_launch_attn_bwd(const usp::Geometry& g, const void* q, const void* k,
                                const void* v, const void* o, const float* lse,
                                const void* dout, const int32_t* doc, const int32_t* cu,
                                void* dq, void* dk, void* dv, void* ws, cudaStream_t st) {
  Args a = make_args(g);
  a.q = (const bf16*)q; a.k = (const bf16*)k; a.v = (const bf16*)v; a.o = (const bf16*)o;
  a.dout = (const bf16*)dout; a.lse = lse; a.doc = doc; a.cu = cu;
  a.dq = (bf16*)dq; a.dk = (bf16*)dk; a.dv = (bf16*)dv; a.delta = (float*)ws;
  return g.D == 128 ? bwd_launch<128>(a, g.P, st) : bwd_launch<64>(a, g.P, st);
}
