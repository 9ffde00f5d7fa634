// Shared device helpers of the USP library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "usp.h"

namespace usp {

// Device status word: bit 0 = a bounded wait gave up, bit 1 = a position
// fell outside the RoPE table, bit 2 = a debug build's index guard stopped
// an out-of-range access.  Kernels receive its address as an argument;
// usp_device_status reports and clears it.
enum : unsigned { kErrTimeout = 1u, kErrRopeRange = 2u, kErrIndex = 4u };

__device__ __forceinline__ void set_status(unsigned* word, unsigned bits) {
  if (word) atomicOr(word, bits);
}

// Index guard of every global-memory access the kernels compute themselves
// (TMA tiles are clipped by their tensor maps).  Builds with
// USP_DEBUG_BOUNDS check that the `count` elements starting at element
// `idx` lie inside a buffer of `n` elements -- the extent usp_dims implies
// for that buffer -- and otherwise record kErrIndex and tell the caller to
// skip the access.  Release builds compile the guard to `true`.
__device__ __forceinline__ bool in_bounds(int64_t idx, int64_t count, int64_t n,
                                          unsigned* status) {
#ifdef USP_DEBUG_BOUNDS
  if (idx < 0 || count < 0 || idx > n - count) {
    set_status(status, kErrIndex);
    return false;
  }
#endif
  return true;
}

// Order of the CTAs of an attention launch over n_tiles row tiles x n_y head
// slots (a 1-D grid of n_tiles * n_y): bands of `band` consecutive head
// slots run one after the other; inside a band the tile rank varies slowest.
// Rank 0 is a kernel's heaviest causal tile, so the heaviest tiles of all the
// band's heads start first, while the heads running at the same time stay
// few enough to share their K/V (or Q/dO) tiles in L2.  Returns the tile
// rank and the head slot of this CTA.
__device__ __forceinline__ void cta_coords(int n_tiles, int band, int& rank, int& y) {
  const unsigned n_y = gridDim.x / (unsigned)n_tiles;
  const unsigned per_band = (unsigned)band * (unsigned)n_tiles;
  const unsigned b = blockIdx.x / per_band;
  const unsigned l = blockIdx.x - b * per_band;
  const unsigned w = min((unsigned)band, n_y - b * (unsigned)band);
  rank = (int)(l / w);
  y = (int)(b * (unsigned)band + l % w);
}

// Band width for cta_coords: the smallest power of two (at most n_y) whose
// band holds at least one CTA per SM, so that a band's heaviest tiles never
// wait behind a whole band of other heads (the tail of a small problem),
// while a large problem keeps one head per band.
// SMs of the current device (the attribute query is cached per device in
// atomics, so concurrent first calls from several host threads are benign).
inline int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev >= 64) {
    int n = 0;
    return cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                   n > 0 ? n : 1;
  }
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

inline int cta_band(int n_tiles, int n_y) {
  const int n_sm = sm_count();
  int band = 1;
  while (band < n_y && (int64_t)band * n_tiles < n_sm) band *= 2;
  return band < n_y ? band : (n_y > 0 ? n_y : 1);
}

// Host side helpers (usp_api.cu).
struct Geometry {
  int64_t S, S_pad, S_loc;
  int P, Hq, Hkv, D, hq, hkv, G;
  int causal;            // 1: keys u <= t of the document; 0: the whole document
  int64_t zz_chunk;      // zigzag chunk C = S_pad/(2P); 0 for contiguous shards
  int n_docs;            // documents in cu_seqlens (0: one document, no cu_seqlens)
  float scale;
  unsigned* status;   // device address of the status word of the current device
};

}  // namespace usp

// Host-side count of kernel launches (usp_launch_count); every launcher
// adds the kernels it enqueued.
void usp_count_launches(unsigned n);

// Kernel launchers implemented per translation unit; all return cudaError_t
// of the launch (cudaGetLastError after the launch).
cudaError_t usp_launch_pad_shard(const usp::Geometry& g, const void* x, int H, void* x_seq,
                                 int32_t* pos, int32_t* doc, const int32_t* cu, int n_docs,
                                 cudaStream_t st);
cudaError_t usp_launch_repack(const usp::Geometry& g, const void* src, int H, const int32_t* pos,
                              const float* rope_cs, int64_t rope_len, int rope_mode,
                              bool to_head, void* dst, cudaStream_t st);
cudaError_t usp_launch_attn_fwd(const usp::Geometry& g, const void* q, const void* k,
                                const void* v, const int32_t* doc, const int32_t* cu,
                                void* o, float* lse, cudaStream_t st, int64_t k_lo,
                                int64_t k_hi);
cudaError_t usp_launch_lse_merge(const usp::Geometry& g, float* o_acc, float* lse_acc,
                                 const void* o_part, const float* lse_part, int first,
                                 void* o_out, cudaStream_t st);
cudaError_t usp_launch_attn_bwd(const usp::Geometry& g, const void* q, const void* k,
                                const void* v, const void* o, const float* lse,
                                const void* dout, const int32_t* doc, const int32_t* cu,
                                void* dq, void* dk, void* dv, void* ws, cudaStream_t st);
size_t usp_attn_bwd_ws_bytes(const usp::Geometry& g);

cudaError_t usp_launch_bounded_wait(int64_t limit_ns, unsigned* status, cudaStream_t st);

// Fixed backward scratch for usp_attn_bwd_noalloc (attn_bwd_tc.cu).
size_t usp_noalloc_scratch_capacity();
cudaError_t usp_noalloc_scratch(void** ptr);

// Tensor map (TMA descriptor) over a head-layout bf16 tensor [P][S_pad][heads][D],
// boxes of 64 columns x box_rows rows with 128-byte swizzle (attn_fwd_tc.cu).
struct CUtensorMap_st;
bool usp_make_head_map(CUtensorMap_st* map, const void* base, int heads, int D, int64_t S_pad,
                       int P, int box_rows);
