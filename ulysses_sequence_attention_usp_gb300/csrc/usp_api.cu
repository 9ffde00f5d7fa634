// C ABI of the USP hot path: argument validation, geometry, launches.
//
// Every entry point checks its arguments on the host and launches nothing
// when they are wrong (SpecForge PR #728 "feat(dspark): add Ulysses sequence
// parallel training", Modifications: Q and KV head counts must be divisible
// by the Ulysses degree; basetenlabs/Megatron-LM PR #7 "GLM-5.2 131k context
// parallelism", Purpose: the RoPE table must cover the padded length, since
// an out-of-range gather was a device-side assert there).
#include <math.h>
#include <string.h>

#include "usp_common.cuh"

#include <atomic>

namespace usp {
__device__ unsigned g_status = 0;
}

static std::atomic<uint64_t> g_launches{0};
void usp_count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {

// Device address of g_status on the current device.  Looked up on every
// call (a table lookup once the module is loaded), so nothing is cached
// across host threads and an address never outlives its context.
unsigned* status_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, usp::g_status) != cudaSuccess) return nullptr;
  return static_cast<unsigned*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

usp_status geometry(const usp_dims* d, usp::Geometry* g) {
  if (d == nullptr) return USP_ERR_INVALID_ARG;
  if (d->S < 0 || d->P < 1) return d->P < 1 ? USP_ERR_HEADS_NOT_DIVISIBLE : USP_ERR_INVALID_ARG;
  if (d->Hq < 1 || d->Hkv < 1) return USP_ERR_INVALID_ARG;
  if (d->Hq % d->P || d->Hkv % d->P || d->Hq % d->Hkv) return USP_ERR_HEADS_NOT_DIVISIBLE;
  if (d->D != 64 && d->D != 128) return USP_ERR_UNSUPPORTED;
  if (d->causal != 0 && d->causal != 1) return USP_ERR_INVALID_ARG;
  if (d->zigzag != 0 && d->zigzag != 1) return USP_ERR_INVALID_ARG;
  if (d->cu_seqlens != nullptr && d->n_docs < 1) return USP_ERR_INVALID_ARG;
  if (!(d->scale >= 0.f) || isinf(d->scale)) return USP_ERR_INVALID_ARG;
  const int64_t unit = d->zigzag ? 2 * (int64_t)d->P : (int64_t)d->P;
  const int64_t S_pad = (d->S + unit - 1) / unit * unit;
  if (S_pad > (int64_t)INT32_MAX) return USP_ERR_UNSUPPORTED;   // positions are int32
  if (d->cu_seqlens_host != nullptr) {
    const int32_t* cu = d->cu_seqlens_host;
    if (d->cu_seqlens == nullptr || cu[0] != 0 || (int64_t)cu[d->n_docs] != d->S)
      return USP_ERR_INVALID_ARG;
    for (int i = 0; i < d->n_docs; ++i)
      if (cu[i + 1] < cu[i]) return USP_ERR_INVALID_ARG;
  }
  g->S = d->S;
  g->P = d->P;
  g->causal = d->causal;
  g->S_pad = S_pad;
  g->S_loc = S_pad / d->P;
  g->zz_chunk = d->zigzag ? S_pad / (2 * (int64_t)d->P) : 0;
  g->Hq = d->Hq;
  g->Hkv = d->Hkv;
  g->D = d->D;
  g->hq = d->Hq / d->P;
  g->hkv = d->Hkv / d->P;
  g->G = d->Hq / d->Hkv;
  g->scale = d->scale > 0.f ? d->scale : (float)(1.0 / sqrt((double)d->D));
  g->n_docs = d->cu_seqlens != nullptr ? d->n_docs : 0;
  g->status = nullptr;
  return USP_OK;
}

// Positions never exceed S_pad - 1; with a host copy of cu_seqlens the bound
// is exact: the longest document, or the pad rows that keep counting in the
// last document.
int64_t max_position(const usp_dims* d, const usp::Geometry& g) {
  if (g.S_pad == 0) return -1;
  if (d->cu_seqlens == nullptr) return g.S_pad - 1;
  if (d->cu_seqlens_host == nullptr) return g.S_pad - 1;
  const int32_t* cu = d->cu_seqlens_host;
  int64_t m = 0;
  for (int i = 0; i < d->n_docs; ++i) m = m > cu[i + 1] - cu[i] ? m : cu[i + 1] - cu[i];
  const int64_t tail = g.S_pad - cu[d->n_docs - 1];   // pad rows continue the last doc
  return (m > tail ? m : tail) - 1;
}

usp_status rope_args(const usp_dims* d, const usp::Geometry& g, const int32_t* pos,
                     const float* cs, int64_t rope_len, int mode) {
  if (mode < -1 || mode > 1) return USP_ERR_INVALID_ARG;
  if (mode == 0) return USP_OK;
  if (pos == nullptr || cs == nullptr || !aligned16(cs) || ((uintptr_t)pos & 3u))
    return USP_ERR_INVALID_ARG;
  if (rope_len <= max_position(d, g)) return USP_ERR_INVALID_ARG;
  return USP_OK;
}

usp_status cuda_status(cudaError_t e) { return e == cudaSuccess ? USP_OK : USP_ERR_CUDA; }

}  // namespace

extern "C" {

int usp_abi_version(void) { return USP_ABI_VERSION; }

int usp_debug_build(void) {
#ifdef USP_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

uint64_t usp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* usp_status_string(usp_status s) {
  switch (s) {
    case USP_OK: return "ok";
    case USP_ERR_INVALID_ARG: return "invalid argument";
    case USP_ERR_HEADS_NOT_DIVISIBLE: return "head counts not divisible by the Ulysses degree";
    case USP_ERR_UNSUPPORTED: return "unsupported configuration";
    case USP_ERR_CUDA: return "CUDA error";
    case USP_ERR_TIMEOUT: return "device-side wait timed out";
    case USP_ERR_OUT_OF_BOUNDS: return "index outside a buffer's extent (debug build)";
  }
  return "unknown status";
}

usp_status usp_pad_shard(const usp_dims* dims, const void* x, int32_t H, void* x_seq,
                         int32_t* pos, int32_t* doc, void* stream) {
  usp::Geometry g;
  usp_status s = geometry(dims, &g);
  if (s != USP_OK) return s;
  if (H < 0 || (H > 0 && (x == nullptr || x_seq == nullptr))) return USP_ERR_INVALID_ARG;
  if (H == 0 && (x != nullptr || x_seq != nullptr)) return USP_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (x_seq && !aligned16(x_seq))) return USP_ERR_INVALID_ARG;
  if (((uintptr_t)pos & 3u) || ((uintptr_t)doc & 3u)) return USP_ERR_INVALID_ARG;
  if (g.zz_chunk > 0 && x != nullptr && x == x_seq) return USP_ERR_INVALID_ARG;
  if (g.S_pad == 0) return USP_OK;
  if ((g.status = status_word()) == nullptr) return USP_ERR_CUDA;
  return cuda_status(usp_launch_pad_shard(g, x, H, H > 0 ? x_seq : nullptr, pos, doc,
                                          dims->cu_seqlens, dims->n_docs,
                                          (cudaStream_t)stream));
}

static usp_status repack(const usp_dims* dims, const void* src, int32_t H, const int32_t* pos,
                         const float* cs, int64_t rope_len, int32_t mode, void* dst,
                         bool to_head, void* stream) {
  usp::Geometry g;
  usp_status s = geometry(dims, &g);
  if (s != USP_OK) return s;
  if (H < 1 || H % g.P) return USP_ERR_HEADS_NOT_DIVISIBLE;
  if (src == nullptr || dst == nullptr || !aligned16(src) || !aligned16(dst) || src == dst)
    return USP_ERR_INVALID_ARG;
  if ((s = rope_args(dims, g, pos, cs, rope_len, mode)) != USP_OK) return s;
  if (g.S_pad == 0) return USP_OK;
  if ((g.status = status_word()) == nullptr) return USP_ERR_CUDA;
  return cuda_status(usp_launch_repack(g, src, H, pos, cs, rope_len, mode, to_head, dst,
                                       (cudaStream_t)stream));
}

usp_status usp_seq_to_head_rope(const usp_dims* dims, const void* x_seq, int32_t H,
                                const int32_t* pos, const float* rope_cs, int64_t rope_len,
                                int32_t rope_mode, void* x_head, void* stream) {
  return repack(dims, x_seq, H, pos, rope_cs, rope_len, rope_mode, x_head, true, stream);
}

usp_status usp_head_to_seq(const usp_dims* dims, const void* x_head, int32_t H,
                           const int32_t* pos, const float* rope_cs, int64_t rope_len,
                           int32_t rope_mode, void* x_seq, void* stream) {
  return repack(dims, x_head, H, pos, rope_cs, rope_len, rope_mode, x_seq, false, stream);
}

static usp_status attn_fwd(const usp_dims* dims, const void* q_h, const void* k_h,
                           const void* v_h, const int32_t* doc, int64_t k_lo, int64_t k_hi,
                           bool window, void* o_h, float* lse, void* stream) {
  usp::Geometry g;
  usp_status s = geometry(dims, &g);
  if (s != USP_OK) return s;
  const void* ptrs[] = {q_h, k_h, v_h, o_h, lse};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return USP_ERR_INVALID_ARG;
  if (doc == nullptr || ((uintptr_t)doc & 3u)) return USP_ERR_INVALID_ARG;
  if (!window) {
    k_lo = 0;
    k_hi = g.S_pad;
  } else if (k_lo < 0 || k_lo > k_hi || k_hi > g.S_pad) {
    return USP_ERR_INVALID_ARG;
  }
  if (g.S_pad == 0) return USP_OK;
  if ((g.status = status_word()) == nullptr) return USP_ERR_CUDA;
  return cuda_status(usp_launch_attn_fwd(g, q_h, k_h, v_h, doc, dims->cu_seqlens, o_h, lse,
                                         (cudaStream_t)stream, k_lo, k_hi));
}

usp_status usp_attn_fwd(const usp_dims* dims, const void* q_h, const void* k_h,
                        const void* v_h, const int32_t* doc, void* o_h, float* lse,
                        void* stream) {
  return attn_fwd(dims, q_h, k_h, v_h, doc, 0, 0, false, o_h, lse, stream);
}

usp_status usp_attn_fwd_window(const usp_dims* dims, const void* q_h, const void* k_h,
                               const void* v_h, const int32_t* doc, int64_t k_lo, int64_t k_hi,
                               void* o_h, float* lse, void* stream) {
  return attn_fwd(dims, q_h, k_h, v_h, doc, k_lo, k_hi, true, o_h, lse, stream);
}

usp_status usp_lse_merge(const usp_dims* dims, float* o_acc, float* lse_acc, const void* o_part,
                         const float* lse_part, int32_t first, void* o_out, void* stream) {
  usp::Geometry g;
  usp_status s = geometry(dims, &g);
  if (s != USP_OK) return s;
  const void* ptrs[] = {o_acc, lse_acc, o_part, lse_part};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return USP_ERR_INVALID_ARG;
  if (o_out != nullptr && !aligned16(o_out)) return USP_ERR_INVALID_ARG;
  if (first != 0 && first != 1) return USP_ERR_INVALID_ARG;
  if (g.S_pad == 0) return USP_OK;
  if ((g.status = status_word()) == nullptr) return USP_ERR_CUDA;
  return cuda_status(usp_launch_lse_merge(g, o_acc, lse_acc, o_part, lse_part, first, o_out,
                                          (cudaStream_t)stream));
}

size_t usp_attn_bwd_workspace(const usp_dims* dims) {
  usp::Geometry g;
  if (geometry(dims, &g) != USP_OK) return 0;
  return usp_attn_bwd_ws_bytes(g);
}

usp_status usp_attn_bwd(const usp_dims* dims, const void* q_h, const void* k_h,
                        const void* v_h, const void* o_h, const float* lse, const void* do_h,
                        const int32_t* doc, void* dq_h, void* dk_h, void* dv_h,
                        void* workspace, size_t ws_bytes, void* stream) {
  usp::Geometry g;
  usp_status s = geometry(dims, &g);
  if (s != USP_OK) return s;
  const void* ptrs[] = {q_h, k_h, v_h, o_h, lse, do_h, dq_h, dk_h, dv_h};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return USP_ERR_INVALID_ARG;
  if (doc == nullptr || ((uintptr_t)doc & 3u)) return USP_ERR_INVALID_ARG;
  if (g.S_pad == 0) return USP_OK;
  if (workspace == nullptr || ((uintptr_t)workspace & 255u) || ws_bytes < usp_attn_bwd_ws_bytes(g))
    return USP_ERR_INVALID_ARG;
  if ((g.status = status_word()) == nullptr) return USP_ERR_CUDA;
  return cuda_status(usp_launch_attn_bwd(g, q_h, k_h, v_h, o_h, lse, do_h, doc,
                                         dims->cu_seqlens, dq_h, dk_h, dv_h, workspace,
                                         (cudaStream_t)stream));
}

usp_status usp_attn_bwd_noalloc(const usp_dims* dims, const void* q_h, const void* k_h,
                                const void* v_h, const void* o_h, const float* lse,
                                const void* do_h, const int32_t* doc, void* dq_h, void* dk_h,
                                void* dv_h, void* stream) {
  usp::Geometry g;
  usp_status s = geometry(dims, &g);
  if (s != USP_OK) return s;
  const void* ptrs[] = {q_h, k_h, v_h, o_h, lse, do_h, dq_h, dk_h, dv_h};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return USP_ERR_INVALID_ARG;
  if (doc == nullptr || ((uintptr_t)doc & 3u)) return USP_ERR_INVALID_ARG;
  if (g.S_pad == 0) return USP_OK;
  // size limit first: nothing touches the device for a problem that does not fit
  if (usp_attn_bwd_ws_bytes(g) > usp_noalloc_scratch_capacity()) return USP_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (usp_noalloc_scratch(&scratch) != cudaSuccess || scratch == nullptr) return USP_ERR_CUDA;
  if ((g.status = status_word()) == nullptr) return USP_ERR_CUDA;
  return cuda_status(usp_launch_attn_bwd(g, q_h, k_h, v_h, o_h, lse, do_h, doc,
                                         dims->cu_seqlens, dq_h, dk_h, dv_h, scratch,
                                         (cudaStream_t)stream));
}

usp_status usp_rope_table(int64_t n_pos, int32_t D, double base, double yarn_factor,
                          int32_t yarn_orig_ctx, float* out_host) {
  if (n_pos < 0 || D < 2 || (D & 1) || out_host == nullptr || !(base > 1.0))
    return USP_ERR_INVALID_ARG;
  if (!(yarn_factor >= 1.0) || (yarn_factor > 1.0 && yarn_orig_ctx < 1))
    return USP_ERR_INVALID_ARG;
  const int half = D / 2;
  double inv[512];
  if (half > 512) return USP_ERR_UNSUPPORTED;
  // YaRN "NTK-by-parts" blend over the pair index (Peng et al. 2023):
  // correction dimension of n turns over the original context.
  double lo = 0, hi = 1;
  if (yarn_factor > 1.0) {
    const double two_pi = 6.283185307179586;
    const double lb = log(base);
    lo = floor(D * log(yarn_orig_ctx / (32.0 * two_pi)) / (2 * lb));
    hi = ceil(D * log(yarn_orig_ctx / (1.0 * two_pi)) / (2 * lb));
    if (lo < 0) lo = 0;
    if (hi > D - 1) hi = D - 1;
    if (hi == lo) hi = lo + 0.001;
  }
  for (int i = 0; i < half; ++i) {
    const double f = pow(base, -2.0 * i / D);
    if (yarn_factor > 1.0) {
      double r = (i - lo) / (hi - lo);
      r = r < 0 ? 0 : (r > 1 ? 1 : r);
      inv[i] = f - r * (f - f / yarn_factor);
    } else {
      inv[i] = f;
    }
  }
  const double m = yarn_factor > 1.0 ? 0.1 * log(yarn_factor) + 1.0 : 1.0;
  for (int64_t p = 0; p < n_pos; ++p) {
    float* row = out_host + p * (int64_t)D;
    for (int i = 0; i < half; ++i) {
      const double th = (double)p * inv[i];
      row[2 * i] = (float)(cos(th) * m);
      row[2 * i + 1] = (float)(sin(th) * m);
    }
  }
  return USP_OK;
}

usp_status usp_selftest_bounded_wait(int32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return USP_ERR_INVALID_ARG;
  unsigned* word = status_word();
  if (word == nullptr) return USP_ERR_CUDA;
  return cuda_status(usp_launch_bounded_wait((int64_t)limit_us * 1000, word, (cudaStream_t)stream));
}

usp_status usp_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return USP_ERR_CUDA;
  unsigned word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, usp::g_status, sizeof(word)) != cudaSuccess) return USP_ERR_CUDA;
  if (word != 0 && cudaMemcpyToSymbol(usp::g_status, &zero, sizeof(zero)) != cudaSuccess)
    return USP_ERR_CUDA;
  if (word & usp::kErrTimeout) return USP_ERR_TIMEOUT;
  if (word & usp::kErrIndex) return USP_ERR_OUT_OF_BOUNDS;
  if (word & usp::kErrRopeRange) return USP_ERR_INVALID_ARG;
  return USP_OK;
}

}  // extern "C"
